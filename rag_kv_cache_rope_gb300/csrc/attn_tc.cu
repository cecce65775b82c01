// Tensor-core causal GQA attention of the recomputed rows over the full blended KV
// (CacheBlend blog, "Selective KV recompute": only the selected rows' attention rows
// are computed, each over every earlier token, reused or fresh).  Head dim 128 runs on
// CTA pairs (k_attn_pair, further below); k_attn_tc, described here, serves head dim 64
// and any device where a pair does not fit.
//
// q is stored per kv head as [pair][d] with pair = row * group + j, so 128 consecutive
// (row, head-of-group) pairs of one kv head form one TMA box and every K/V block is
// shared by the whole head group.  A work item is two consecutive 128-pair tiles (A
// and B) of one kv head and one request; items run longest first on persistent CTAs,
// dealt in snake order, and the two tiles share every K/V block.  Per 128-key block,
// for each tile:
//   S = Q . K^T   tcgen05.mma M128 N128 K16 x8, shared-memory operands -> TMEM
//   P             one softmax warpgroup per tile, one pair row per thread: the row's 128
//                 scores come to registers in one TMEM round trip; row maximum (causal mask
//                 on boundary blocks; three-input max), then bf16 P (base 2, scale folded
//                 into paired FMAs, sums in paired adds, 2^x on the MUFU unit) written back
//                 over S's first 64 TMEM columns in one more round trip.
//   O += P . V    tcgen05.mma M128 N128 K16 x8 with A = P read from TMEM and V an
//                 MN-major shared-memory operand; O stays in TMEM for the whole item.
// Per tile the products run S(j), PV(j), S(j+1): the tensor core executes one CTA's
// MMAs in order, so S(j+1) cannot overwrite P(j) before PV(j) has read it, and the
// completion of S(j) implies that of PV(j-1), which lets the softmax rescale O right
// after S(j) arrives.  The running maximum used for P is raised only when a row's
// maximum grows by more than 2^8 (then that warp rescales its rows of O in TMEM); the
// sum l uses the same maximum, so O / l is exact.  While one tile's softmax runs, the
// tensor core works on the other tile.
// Warps: 0 TMA producer, 1 TMEM owner + MMA issuer, 2..5 softmax of tile A, 6..9 of
// tile B.  All mbarrier waits are bounded (error word BLEND_ETIMEOUT, loads drained,
// TMEM freed).
#include <cmath>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "gemm_tc.cuh"

namespace blend {
namespace {

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int KV_STAGES = 2;
constexpr int QH_BYTES = BQ * 64 * 2;    // 16 KB: one 64-wide column half of a Q tile
constexpr int KH_BYTES = BKV * 64 * 2;   // 16 KB: one 64-wide column half of a K or V block
// Per head dim D (64 or 128): a Q tile and a K or V block hold D/64 column halves.
template <int D> struct AttnCfg {
    static constexpr int NH = D / 64;
    static constexpr int QT_BYTES = NH * QH_BYTES;          // one 128-pair Q tile
    static constexpr int KV_BYTES = 2 * NH * KH_BYTES;      // K halves, then V halves
    static constexpr int SMEM_BYTES = 2 * QT_BYTES + KV_STAGES * KV_BYTES + 1024;
    // kind::f16, bf16 inputs, fp32 accumulate, M128 N=D, B (V) MN-major
    static constexpr uint32_t IDESC_PV =
        (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((D >> 3) << 17) | ((BQ >> 4) << 24);
};
constexpr int TMEM_COLS = 512;  // tile t: S (and P over its first 64 columns) t*256+[0,128), O t*256+[128,256)
constexpr int THREADS = 320;
constexpr float RESCALE_LOG2 = 8.f;
constexpr long long SPIN_LIMIT = 1ll << 24;

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* b, int c) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(c) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t par) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(su32(b)), "r"(par)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t par, volatile int* abort_flag) {
    for (long long i = 0; i < SPIN_LIMIT; ++i) {
        if (mbar_try(b, par)) return true;
        if ((i & 255) == 255 && *abort_flag) return false;
    }
    return false;
}
// Warp-level bounded wait: every lane polls (a convergent loop, no lane-0 divergence)
// until all lanes have seen the phase complete.
__device__ __forceinline__ bool warp_wait(uint64_t* b, uint32_t par, volatile int* abort_flag) {
    for (long long i = 0; i < SPIN_LIMIT; ++i) {
        if (__all_sync(0xffffffffu, mbar_try(b, par))) return true;
        if ((i & 255) == 255 && __any_sync(0xffffffffu, *abort_flag != 0)) return false;
    }
    return false;
}
// Warp-level arrive (barriers count warps): __syncwarp orders every lane's prior work
// before lane 0's release-arrive.
__device__ __forceinline__ void warp_arrive(uint64_t* b) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(b);
}
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            su32(dst)),
        "l"((uint64_t)m), "r"(su32(bar)), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
            su32(dst)),
        "l"((uint64_t)m), "r"(su32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// K-major operand, 128-byte swizzle: rows of 128 B, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_k(uint32_t a) {
    return (uint64_t)((a & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// MN-major operand (V as B of P.V), 128-byte swizzle: each key row holds 64 d values
// (128 B); 8-key groups 1024 B apart (stride byte offset); the second 64-wide d half
// 16 KB further (leading byte offset).
__device__ __forceinline__ uint64_t desc_mn(uint32_t a) {
    return (uint64_t)((a & 0x3FFFF) >> 4) | ((uint64_t)(KH_BYTES >> 4) << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// kind::f16, bf16 inputs, fp32 accumulate, M128 N128 (S = Q K^T over 128 keys).
constexpr uint32_t IDESC_S = (1u << 4) | (1u << 7) | (1u << 10) | ((BKV >> 3) << 17) | ((BQ >> 4) << 24);

// D (TMEM) op= A (shared-memory descriptor) . B (shared-memory descriptor)
__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// D (TMEM) op= A (TMEM: lane = row, two bf16 per column) . B (shared-memory descriptor)
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void commit(uint64_t* b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(b))
                 : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Two fp32 values to one register of two bf16 (round to nearest even), lo in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
#define TMEM_LD32(taddr, r)                                                                          \
    asm volatile(                                                                                    \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"   \
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"             \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),   \
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),             \
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),             \
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])              \
        : "r"(taddr))
#define TMEM_ST32(taddr, r)                                                                          \
    asm volatile(                                                                                    \
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),   \
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),      \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), \
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),           \
        "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),           \
        "r"(r[30]), "r"(r[31])                                                                       \
        : "memory")
#define TMEM_ST16(taddr, r)                                                                          \
    asm volatile(                                                                                    \
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
        "%15,%16};" ::"r"(taddr),                                                                    \
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),      \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]) \
        : "memory")

struct Item {
    int g, row0, npairs, pair0_a, pair0_b, max_pos, tok_base, nblk;
};

// Work item w -> two tiles.  Request r has tiles_r = ceil(rows_r * group / 128) tiles per
// kv head, paired from the top (largest positions, longest KV range) down; items of the
// first pair of every kv head come first.
__device__ __forceinline__ bool get_item(int w, int n_req, const int32_t* req_row_end, const int32_t* row_pos,
                                         const int32_t* row_tok, int group, int hkv, Item& it) {
    int row0 = 0;
    for (int r = 0; r < n_req; ++r) {
        const int row1 = req_row_end[r];
        const int np = (row1 - row0) * group;
        const int tiles = (np + BQ - 1) / BQ;
        const int items = (tiles + 1) / 2;
        if (w < items * hkv) {
            const int ta = tiles - 1 - 2 * (w / hkv);
            const int tb = ta - 1;
            it.g = w % hkv;
            it.row0 = row0;
            it.npairs = np;
            it.pair0_a = ta * BQ;
            it.pair0_b = tb >= 0 ? tb * BQ : -1;
            const int last = min(ta * BQ + BQ, np) - 1;
            const int lrow = row0 + last / group;
            it.max_pos = row_pos[lrow];
            it.tok_base = row_tok[lrow] - it.max_pos;
            it.nblk = it.max_pos / BKV + 1;
            return true;
        }
        w -= items * hkv;
        row0 = row1;
    }
    return false;
}

// S of tile t (into its TMEM region) for the K block whose descriptor base is kd; the
// start-address field of a descriptor holds address / 16, so operand steps are added to
// the descriptor itself (shared addresses stay below 2^18, so the field never carries).
template <int D>
__device__ __forceinline__ void issue_s(uint32_t tb, int t, uint64_t qd, uint64_t kd) {
    const uint32_t sd = tb + t * 256;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk & 3) * 32, half = kk >> 2;
        umma_ss(sd, qd + ((half * QH_BYTES + off) >> 4), kd + ((half * KH_BYTES + off) >> 4), IDESC_S,
                kk > 0 ? 1u : 0u);
    }
}
// O of tile t += P (TMEM, first 64 columns of its S region) . V (block descriptor base vd).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tb, int t, uint64_t vd, bool first) {
    const uint32_t od = tb + t * 256 + 128;
    const uint32_t pa = tb + t * 256;
#pragma unroll
    for (int kk = 0; kk < BKV / 16; ++kk)
        umma_ts(od, pa + kk * 8, vd + ((kk * 2048) >> 4), AttnCfg<D>::IDESC_PV, (!first || kk > 0) ? 1u : 0u);
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
              const __grid_constant__ CUtensorMap mapV, int n_req, const int32_t* __restrict__ req_row_end,
              const int32_t* __restrict__ row_pos, const int32_t* __restrict__ row_tok, int group, int hkv,
              int m_cap, float scale_log2, bf16* __restrict__ out, int32_t* __restrict__ err) {
    constexpr int NH = AttnCfg<D>::NH;
    constexpr int QT_BYTES = AttnCfg<D>::QT_BYTES;
    constexpr int KV_BYTES = AttnCfg<D>::KV_BYTES;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_full, q_empty, kv_full[KV_STAGES], kv_empty[KV_STAGES], s_full[2], p_full[2],
        o_full[2], o_free[2];
    __shared__ uint32_t tmem_sh;
    __shared__ volatile int abort_flag;
    __shared__ int pend_kv[KV_STAGES];
    __shared__ int pend_q;

    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = smem;                  // tile t at t * QT_BYTES
    uint8_t* sKV = smem + 2 * QT_BYTES;  // stage s at s * KV_BYTES
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    int total = 0;
    {
        int row0 = 0;
        for (int r = 0; r < n_req; ++r) {
            const int row1 = req_row_end[r];
            const int tiles = ((row1 - row0) * group + BQ - 1) / BQ;
            total += hkv * ((tiles + 1) / 2);
            row0 = row1;
        }
    }
    if (threadIdx.x == 0) {
        mbar_init(&q_full, 1);
        mbar_init(&q_empty, 1);
        for (int s = 0; s < KV_STAGES; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
            pend_kv[s] = -1;
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 4);
            mbar_init(&o_full[t], 1);
            mbar_init(&o_free[t], 4);
        }
        pend_q = -1;
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_sh)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tb = tmem_sh;
    const int qslab = m_cap * group;  // pair rows per kv head in q
    // items are sorted longest first; round k gives CTA b item k*G + b (k even) or
    // k*G + G-1-b (k odd), which evens out the total length per CTA
    auto item_of = [&](int k) -> int {
        return k * (int)gridDim.x + ((k & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x);
    };

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t it = 0, tl = 0;
        for (int k = 0; !abort_flag; ++k, ++tl) {
            const int w = item_of(k);
            if (w >= total) break;
            Item m;
            get_item(w, n_req, req_row_end, row_pos, row_tok, group, hkv, m);
            if (!mbar_wait(&q_empty, (tl & 1) ^ 1, &abort_flag)) {
                abort_flag = 1;
                set_error(err, BLEND_ETIMEOUT);
                break;
            }
            mbar_expect_tx(&q_full, 2 * QT_BYTES);
            pend_q = (int)(tl & 1);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                // an absent second tile reloads the first (finite data, never stored)
                const int p0 = (t == 0 || m.pair0_b < 0) ? m.pair0_a : m.pair0_b;
                const int qrow = m.g * qslab + m.row0 * group + p0;
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) tma_2d(sQ + t * QT_BYTES + hh * QH_BYTES, &mapQ, &q_full, hh * 64, qrow);
            }
            for (int kb = 0; kb < m.nblk; ++kb, ++it) {
                const int st = it % KV_STAGES;
                if (!mbar_wait(&kv_empty[st], ((it / KV_STAGES) & 1) ^ 1, &abort_flag)) {
                    abort_flag = 1;
                    set_error(err, BLEND_ETIMEOUT);
                    break;
                }
                uint8_t* b = sKV + st * KV_BYTES;
                mbar_expect_tx(&kv_full[st], KV_BYTES);
                pend_kv[st] = (int)((it / KV_STAGES) & 1);
                const int tok = m.tok_base + kb * BKV;
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) {
                    tma_3d(b + hh * KH_BYTES, &mapK, &kv_full[st], hh * 64, m.g, tok);
                    tma_3d(b + (NH + hh) * KH_BYTES, &mapV, &kv_full[st], hh * 64, m.g, tok);
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        uint32_t it = 0, tl = 0;
        bool ok = true;
        const uint64_t qd0 = desc_k(su32(sQ)), qd1 = desc_k(su32(sQ + QT_BYTES));
        for (int k = 0; ok && !abort_flag; ++k, ++tl) {
            const int w = item_of(k);
            if (w >= total) break;
            Item m;
            get_item(w, n_req, req_row_end, row_pos, row_tok, group, hkv, m);
            if (!mbar_wait(&q_full, tl & 1, &abort_flag) ||
                !mbar_wait(&kv_full[it % KV_STAGES], (it / KV_STAGES) & 1, &abort_flag)) {
                ok = false;
                break;
            }
            pend_q = -1;
            pend_kv[it % KV_STAGES] = -1;
            fence_after();
            {
                const uint64_t kd = desc_k(su32(sKV + (it % KV_STAGES) * KV_BYTES));
                issue_s<D>(tb, 0, qd0, kd);
                commit(&s_full[0]);
                issue_s<D>(tb, 1, qd1, kd);
                commit(&s_full[1]);
            }
            for (int kb = 0; kb < m.nblk && ok; ++kb, ++it) {
                const int st = it % KV_STAGES;
                const uint64_t vd = desc_mn(su32(sKV + st * KV_BYTES + NH * KH_BYTES));
                const bool more = kb + 1 < m.nblk;
                for (int t = 0; t < 2; ++t) {
                    if (!mbar_wait(&p_full[t], it & 1, &abort_flag) ||
                        (kb == 0 && !mbar_wait(&o_free[t], (tl & 1) ^ 1, &abort_flag))) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    issue_pv<D>(tb, t, vd, kb == 0);
                    if (more) {
                        const int nst = (it + 1) % KV_STAGES;
                        if (t == 0) {
                            if (!mbar_wait(&kv_full[nst], ((it + 1) / KV_STAGES) & 1, &abort_flag)) {
                                ok = false;
                                break;
                            }
                            pend_kv[nst] = -1;
                            fence_after();
                        }
                        issue_s<D>(tb, t, t == 0 ? qd0 : qd1, desc_k(su32(sKV + nst * KV_BYTES)));
                        commit(&s_full[t]);
                    } else {
                        commit(&o_full[t]);
                    }
                }
                if (!ok) break;
                commit(&kv_empty[st]);  // both tiles' S and PV of this block are issued
            }
            if (!ok) break;
            commit(&q_empty);
        }
        if (!ok) {
            abort_flag = 1;
            set_error(err, BLEND_ETIMEOUT);
        }
    } else if (warp >= 2) {
        // ------------------------------------------------ softmax (tile t) + output
        const int t = (warp - 2) / 4;
        const int sp = warp & 3;  // TMEM lane quarter of this warp
        const int r_in = sp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
        const uint32_t s_col = tb + lane_off + t * 256;
        const uint32_t o_col = s_col + 128;
        uint32_t it = 0, tl = 0;
        bool ok = true;
        for (int k = 0; ok; ++k, ++tl) {
            const int w = item_of(k);
            if (w >= total) break;
            Item m;
            get_item(w, n_req, req_row_end, row_pos, row_tok, group, hkv, m);
            const int my_pair0 = t == 0 ? m.pair0_a : m.pair0_b;
            const bool have = my_pair0 >= 0;
            const int p = (have ? my_pair0 : 0) + r_in;
            const bool valid = have && p < m.npairs;
            const int row = m.row0 + (valid ? p / group : 0);
            const int my_pos = valid ? row_pos[row] : m.max_pos;
            float m_used = -INFINITY, l = 0.f;
            for (int kb = 0; kb < m.nblk; ++kb, ++it) {
                if (!warp_wait(&s_full[t], it & 1, &abort_flag)) {
                    ok = false;
                    break;
                }
                fence_after();
                const int k0 = kb * BKV;
                // all 128 scores of the row in registers with a single TMEM round trip
                uint32_t s[128];
                TMEM_LD32(s_col, s);
                TMEM_LD32(s_col + 32, (s + 32));
                TMEM_LD32(s_col + 64, (s + 64));
                TMEM_LD32(s_col + 96, (s + 96));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (k0 + BKV - 1 > my_pos) {
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (k0 + i > my_pos) s[i] = __float_as_uint(-INFINITY);
                }
                float mx;
                {
                    // row maximum: 8 independent chains, then a short tree
                    float a[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) a[i] = fmaxf(__uint_as_float(s[i]), __uint_as_float(s[i + 8]));
#pragma unroll
                    for (int i = 16; i < 128; i += 16)
#pragma unroll
                        for (int c = 0; c < 8; ++c) a[c] = max3f(a[c], __uint_as_float(s[i + c]), __uint_as_float(s[i + 8 + c]));
                    mx = max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
                }
                const float mxs = mx * scale_log2;
                const bool need = mxs > m_used + RESCALE_LOG2;
                const bool rescale = __any_sync(0xffffffffu, need);
                float corr = 1.f;
                if (rescale) {
                    const float m_new = need ? mxs : m_used;
                    corr = ex2(m_used - m_new);
                    l *= corr;
                    m_used = m_new;
                }
                // P = 2^(s * scale - m_used) as bf16 pairs, packed in place: word e (keys 2e,
                // 2e+1) lands in s[e], whose own score was consumed at step e/2
                float2 acc2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(-m_used, -m_used);
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])), sc2, nm2);
                    const float p0 = ex2(x.x), p1 = ex2(x.y);
                    acc2[e & 1] = __fadd2_rn(acc2[e & 1], make_float2(p0, p1));
                    s[e] = pack_bf16x2(p0, p1);
                }
                const float2 accs = __fadd2_rn(acc2[0], acc2[1]);
                TMEM_ST32(s_col, s);
                TMEM_ST32(s_col + 32, (s + 32));
                if (rescale && kb > 0) {
                    // S of this block completed after P.V of the previous one, so O is settled;
                    // bring it to the new maximum before this block's P.V adds to it
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t o[32];
                        TMEM_LD32(o_col + c, o);
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
                        TMEM_ST32(o_col + c, o);
                    }
                }
                l += accs.x + accs.y;
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                fence_before();
                warp_arrive(&p_full[t]);
            }
            if (!ok) break;
            // O of this tile is final once the last P.V has completed
            if (!warp_wait(&o_full[t], tl & 1, &abort_flag)) {
                ok = false;
                break;
            }
            fence_after();
            const float inv = 1.f / l;
            bf16* dst = out + (long long)row * (hkv * group * D) + (long long)(m.g * group + (valid ? p % group : 0)) * D;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                TMEM_LD32(o_col + c, o);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (valid) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint32_t w4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w4[e] = pack_bf16x2(__uint_as_float(o[v * 8 + 2 * e]) * inv,
                                                __uint_as_float(o[v * 8 + 2 * e + 1]) * inv);
                        *reinterpret_cast<uint4*>(dst + c + v * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            }
            fence_before();
            warp_arrive(&o_free[t]);
        }
        if (!ok) {
            abort_flag = 1;
            if (lane == 0) set_error(err, BLEND_ETIMEOUT);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) {
        // let every load still in flight land before the shared memory is released
        for (int s = 0; s < KV_STAGES; ++s)
            if (pend_kv[s] >= 0)
                for (long long i = 0; i < SPIN_LIMIT && !mbar_try(&kv_full[s], (uint32_t)pend_kv[s]); ++i) {
                }
        if (pend_q >= 0)
            for (long long i = 0; i < SPIN_LIMIT && !mbar_try(&q_full, (uint32_t)pend_q); ++i) {
            }
    }
    __syncthreads();
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tb), "r"(TMEM_COLS) : "memory");
    }
}

// ---------------------------------------------------------------- CTA-pair kernel (D = 128)
// The two CTAs of a cluster take the two tiles of one work item.  Each holds its own Q
// tile, and per 128-key block each stages half of the block's keys (for S) and half of
// V's d columns (for P.V), so every block is loaded once for both tiles and each SM
// reads a third less operand data per FLOP.  The leading CTA issues, for both:
//   S = Q . K^T   tcgen05.mma.cta_group::2 M256 N128 K16 x8 (A: each CTA's Q tile; B:
//                 each CTA's 64 keys) into S buffer j % 3
//   O += P . V    tcgen05.mma.cta_group::2 M256 N128 K16 x8 (A: each CTA's P in TMEM;
//                 B: each CTA's 64 d columns of V, MN-major)
// S has three TMEM buffers of 128 fp32 columns, and each block's P (64 columns of bf16
// pairs) is written over the first half of its own S buffer, so S, P and O take all 512
// columns.  Two threads of the leading CTA issue the products: one issues S(j) once
// P.V(j-3) has read the P over that buffer and commits it to s_full; the other issues
// P.V(j) once P(j) is ready and commits it to kv_empty, which frees block j's K/V stage
// and S buffer.  A single issuer spent about 650 of every 1 650 cycles per block on
// barrier checks and commits between its bursts while the tensor core, with an issue
// queue about one product deep, sat idle; two issuers overlap those gaps.  The softmax
// skips the block maximum while its running reference keeps every exponential of the
// block below 2^50 (the block's sum says so); a row's first block and any block past that
// bound take the exact path (maximum, conditional rescale by more than 2^8).  With three
// S buffers, S(j) runs up to two blocks ahead of the softmax and the softmax never waits
// for a P buffer (two buffers for S plus two for P measured about 6 % slower); one that
// must rescale O first waits for P.V(j-1).  The softmax is the single-tile one of
// k_attn_tc, one pair row per thread.
namespace pairk {
constexpr int THREADS2 = 224;  // warp 0 TMA, 1 TMEM + P.V issue, 2..5 softmax, 6 S issue (leaders)
constexpr int S_WARP = 6;
constexpr int STAGES2 = 5;
constexpr int KQ_BYTES = 64 * 64 * 2;                  // 64 keys x one 64-wide d half
constexpr int VH_BYTES = BKV * 64 * 2;                 // 128 keys x this CTA's 64 d columns
constexpr int STAGE_BYTES = 2 * KQ_BYTES + VH_BYTES;   // 32 KB
constexpr int QT_BYTES = 2 * QH_BYTES;                 // one 128-pair tile, two d halves
constexpr int SMEM_BYTES = 2 * QT_BYTES + STAGES2 * STAGE_BYTES + 1024;
constexpr int COLS2 = 512;  // S buffers at 0, 128 and 256 (each block's P goes over its S), O at 384
constexpr int NSBUF = 3;
constexpr uint32_t O_COL = 384;
// kind::f16, bf16 inputs, fp32 accumulate, M256 (the pair) N128; P.V with B MN-major
constexpr uint32_t IDESC_S2 = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((256u >> 4) << 24);
constexpr uint32_t IDESC_PV2 = IDESC_S2 | (1u << 16);

__device__ __forceinline__ uint32_t cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t leader_addr(const void* p) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(su32(p)));
    return r;
}
__device__ __forceinline__ void tma_2d_pair(void* dst, const CUtensorMap* m, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4}], [%2];" ::"r"(su32(dst)),
        "l"((uint64_t)m), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void tma_3d_pair(void* dst, const CUtensorMap* m, uint32_t bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4, %5}], [%2];" ::"r"(su32(dst)),
        "l"((uint64_t)m), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void umma_ss2(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void umma_ts2(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// arrive on this barrier in both CTAs once the MMAs issued so far complete
__device__ __forceinline__ void commit2(uint64_t* b) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            su32(b)),
        "h"((uint16_t)3)
        : "memory");
}
__device__ __forceinline__ bool try_cl(uint64_t* b, uint32_t par) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(su32(b)), "r"(par)
        : "memory");
    return ok != 0;
}
// Non-blocking test of the phase: a blocking try_wait on a barrier that the other CTA
// arrives on was measured to resume up to ~1.5 K cycles after the phase completed.
__device__ __forceinline__ bool test_cl(uint64_t* b, uint32_t par) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(su32(b)), "r"(par)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool wait_cl(uint64_t* b, uint32_t par, volatile int* abort_flag) {
    for (long long i = 0; i < 64 * SPIN_LIMIT; ++i) {
        if (test_cl(b, par)) return true;
        if ((i & 1023) == 1023 && *abort_flag) return false;
    }
    return false;
}
__device__ __forceinline__ bool warp_wait_cl(uint64_t* b, uint32_t par, volatile int* abort_flag) {
    for (long long i = 0; i < SPIN_LIMIT; ++i) {
        if (__all_sync(0xffffffffu, try_cl(b, par))) return true;
        if ((i & 255) == 255 && __any_sync(0xffffffffu, *abort_flag != 0)) return false;
    }
    return false;
}
// Warp-level arrive on the leader's barrier: local in the leader, remote from rank 1
// (default semantics: a cluster-scope release here was measured to cost ~1 K cycles per
// block; the TMEM stores it follows are complete by tcgen05.wait::st).
__device__ __forceinline__ void warp_arrive_leader(uint64_t* b, int rank) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        if (rank == 0)
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
        else
            asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(leader_addr(b)) : "memory");
    }
}
}  // namespace pairk

__global__ void __launch_bounds__(pairk::THREADS2, 1)
    k_attn_pair(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                const __grid_constant__ CUtensorMap mapV, int n_req, const int32_t* __restrict__ req_row_end,
                const int32_t* __restrict__ row_pos, const int32_t* __restrict__ row_tok, int group, int hkv,
                int m_cap, float scale_log2, bf16* __restrict__ out, int32_t* __restrict__ err) {
    using namespace pairk;
    constexpr int D = 128;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_full[2], q_empty[2], kv_full[STAGES2], kv_empty[STAGES2], s_full[NSBUF],
        p_full[NSBUF], o_full, o_free;
    __shared__ uint32_t tmem_sh;
    __shared__ volatile int abort_flag;
    __shared__ int pend_kv[STAGES2];
    __shared__ int pend_q[2];

    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = smem;                  // Q buffer qb at qb * QT_BYTES
    uint8_t* sKV = smem + 2 * QT_BYTES;  // stage s at s * STAGE_BYTES: K d-half 0, K d-half 1, V half
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int rank = (int)cta_rank();
    const int grp = (int)(blockIdx.x >> 1), n_grp = (int)(gridDim.x >> 1);

    int total = 0;
    {
        int row0 = 0;
        for (int r = 0; r < n_req; ++r) {
            const int row1 = req_row_end[r];
            const int tiles = ((row1 - row0) * group + BQ - 1) / BQ;
            total += hkv * ((tiles + 1) / 2);
            row0 = row1;
        }
    }
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&q_full[b], 1);
            mbar_init(&q_empty[b], 1);
            pend_q[b] = -1;
        }
        for (int b = 0; b < NSBUF; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 8);  // 4 softmax warps in each CTA
        }
        for (int s = 0; s < STAGES2; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
            pend_kv[s] = -1;
        }
        mbar_init(&o_full, 1);
        mbar_init(&o_free, 8);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        // allocated collectively: one warp of each CTA, the same columns in both
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_sh)),
                     "r"(COLS2)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before either signals the other's
    fence_after();
    const uint32_t tb = tmem_sh;
    const int qslab = m_cap * group;
    auto item_of = [&](int k) -> int { return k * n_grp + ((k & 1) ? n_grp - 1 - grp : grp); };

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        uint32_t it = 0;
        for (int k = 0, tl = 0; !abort_flag; ++k, ++tl) {
            const int w = item_of(k);
            if (w >= total) break;
            Item m;
            get_item(w, n_req, req_row_end, row_pos, row_tok, group, hkv, m);
            const int qb = tl & 1;
            if (!wait_cl(&q_empty[qb], ((tl >> 1) & 1) ^ 1, &abort_flag)) {
                abort_flag = 1;
                set_error(err, BLEND_ETIMEOUT);
                break;
            }
            if (rank == 0) {
                mbar_expect_tx(&q_full[qb], 2 * QT_BYTES);  // both CTAs' tiles count here
                pend_q[qb] = (tl >> 1) & 1;
            }
            {
                // an absent second tile reloads the first (finite data, never stored)
                const int p0 = (rank == 0 || m.pair0_b < 0) ? m.pair0_a : m.pair0_b;
                const int qrow = m.g * qslab + m.row0 * group + p0;
                const uint32_t qf = leader_addr(&q_full[qb]);
                tma_2d_pair(sQ + qb * QT_BYTES, &mapQ, qf, 0, qrow);
                tma_2d_pair(sQ + qb * QT_BYTES + QH_BYTES, &mapQ, qf, 64, qrow);
            }
            for (int kb = 0; kb < m.nblk; ++kb, ++it) {
                const int st = it % STAGES2;
                if (!wait_cl(&kv_empty[st], ((it / STAGES2) & 1) ^ 1, &abort_flag)) {
                    abort_flag = 1;
                    set_error(err, BLEND_ETIMEOUT);
                    break;
                }
                uint8_t* b = sKV + st * STAGE_BYTES;
                if (rank == 0) {
                    mbar_expect_tx(&kv_full[st], 2 * STAGE_BYTES);
                    pend_kv[st] = (int)((it / STAGES2) & 1);
                }
                const uint32_t kf = leader_addr(&kv_full[st]);
                const int tok = m.tok_base + kb * BKV;
                // this CTA's 64 keys (both d halves) and its 64 d columns of V (all keys)
                tma_3d_pair(b, &mapK, kf, 0, m.g, tok + 64 * rank);
                tma_3d_pair(b + KQ_BYTES, &mapK, kf, 64, m.g, tok + 64 * rank);
                tma_3d_pair(b + 2 * KQ_BYTES, &mapV, kf, 64 * rank, m.g, tok);
            }
        }
    } else if (warp == S_WARP && lane == 0 && rank == 0) {
        // ------------------------------------------------ S issuer (leader, for both CTAs)
        // S(it) goes into S buffer it % 3 once P.V(it - 3) has read the P that its softmax
        // wrote over that buffer, and is committed to s_full on its own
        uint32_t it = 0;
        bool ok = true;
        for (int k = 0, tl = 0; ok && !abort_flag; ++k, ++tl) {
            const int w = item_of(k);
            if (w >= total) break;
            Item m;
            get_item(w, n_req, req_row_end, row_pos, row_tok, group, hkv, m);
            const int qb = tl & 1;
            if (!wait_cl(&q_full[qb], (tl >> 1) & 1, &abort_flag)) {
                ok = false;
                break;
            }
            pend_q[qb] = -1;
            const uint64_t qd = desc_k(su32(sQ + qb * QT_BYTES));
            for (int kb = 0; kb < m.nblk; ++kb, ++it) {
                const int b = it % NSBUF, st = it % STAGES2;
                const uint32_t pv = it - NSBUF;  // the P.V that last read this buffer
                if ((it >= NSBUF && !wait_cl(&kv_empty[pv % STAGES2], (pv / STAGES2) & 1, &abort_flag)) ||
                    !wait_cl(&kv_full[st], (it / STAGES2) & 1, &abort_flag)) {
                    ok = false;
                    break;
                }
                pend_kv[st] = -1;
                fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32, half = kk >> 2;
                    umma_ss2(tb + b * 128, qd + ((half * QH_BYTES + off) >> 4),
                             desc_k(su32(sKV + st * STAGE_BYTES)) + ((half * KQ_BYTES + off) >> 4), IDESC_S2,
                             kk > 0 ? 1u : 0u);
                }
                commit2(&s_full[b]);
            }
            if (!ok) break;
            commit2(&q_empty[qb]);  // every S product of the item has read this Q tile
        }
        if (!ok) {
            abort_flag = 1;
            set_error(err, BLEND_ETIMEOUT);
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ------------------------------------------------ P.V issuer (leader, for both CTAs)
        // P.V(it) once both CTAs' softmax warps have written P(it); its commit frees block
        // it's K/V stage (S(it) completed before that softmax began) and its S buffer
        uint32_t it = 0;
        bool ok = true;
        for (int k = 0, tl = 0; ok && !abort_flag; ++k, ++tl) {
            const int w = item_of(k);
            if (w >= total) break;
            Item m;
            get_item(w, n_req, req_row_end, row_pos, row_tok, group, hkv, m);
            for (int kb = 0; kb < m.nblk; ++kb, ++it) {
                const int b = it % NSBUF, st = it % STAGES2;
                if (!wait_cl(&p_full[b], (it / NSBUF) & 1, &abort_flag) ||
                    (kb == 0 && !wait_cl(&o_free, (tl & 1) ^ 1, &abort_flag))) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint64_t vd = desc_mn(su32(sKV + st * STAGE_BYTES + 2 * KQ_BYTES));
                const uint32_t pa = tb + b * 128;  // P over its block's S columns
#pragma unroll
                for (int kk = 0; kk < BKV / 16; ++kk)
                    umma_ts2(tb + O_COL, pa + kk * 8, vd + ((kk * 2048) >> 4), IDESC_PV2, (kb > 0 || kk > 0) ? 1u : 0u);
                commit2(&kv_empty[st]);
            }
            if (!ok) break;
            commit2(&o_full);
        }
        if (!ok) {
            abort_flag = 1;
            set_error(err, BLEND_ETIMEOUT);
        }
    } else if (warp >= 2 && warp < S_WARP) {
        // ------------------------------------------------ softmax of this CTA's tile + output
        const int sp = warp & 3;  // TMEM lane quarter of this warp
        const int r_in = sp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
        const uint32_t o_col = tb + lane_off + O_COL;
        uint32_t it = 0;
        bool ok = true;
        for (int k = 0, tl = 0; ok; ++k, ++tl) {
            const int w = item_of(k);
            if (w >= total) break;
            Item m;
            get_item(w, n_req, req_row_end, row_pos, row_tok, group, hkv, m);
            const int my_pair0 = rank == 0 ? m.pair0_a : m.pair0_b;
            const bool have = my_pair0 >= 0;
            const int p = (have ? my_pair0 : 0) + r_in;
            const bool valid = have && p < m.npairs;
            const int row = m.row0 + (valid ? p / group : 0);
            const int my_pos = valid ? row_pos[row] : m.max_pos;
            float m_used = -INFINITY, l = 0.f;
            for (int kb = 0; kb < m.nblk; ++kb, ++it) {
                const int b = it % NSBUF;
                const uint32_t s_col = tb + lane_off + b * 128;
                // S(it) is the (it / 3)-th product into S buffer b; S(it + 3) waits for
                // P.V(it), which waits for this block's P, so the barrier is never a phase ahead
                const bool got = warp_wait_cl(&s_full[b], (it / NSBUF) & 1, &abort_flag);
                if (!got) {
                    ok = false;
                    break;
                }
                fence_after();
                const int k0 = kb * BKV;
                uint32_t s[128];
                TMEM_LD32(s_col, s);
                TMEM_LD32(s_col + 32, (s + 32));
                TMEM_LD32(s_col + 64, (s + 64));
                TMEM_LD32(s_col + 96, (s + 96));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (k0 + BKV - 1 > my_pos) {
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (k0 + i > my_pos) s[i] = __float_as_uint(-INFINITY);
                }
                const float2 sc2 = make_float2(scale_log2, scale_log2);
                float2 accs = make_float2(0.f, 0.f);
                bool rescale = false;
                float corr = 1.f;
                // Fast path: exponentiate against the running reference without this block's
                // maximum.  Values up to 2^50 are exact enough in fp32 and bf16 and far from
                // overflow in P, the row sum and O, so only a block whose sum passes 2^50 (or
                // a row's first block) takes the exact path below with its maximum and rescale.
                bool exact = !__all_sync(0xffffffffu, m_used != -INFINITY);
                if (!exact) {
                    float2 acc2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    const float2 nm2 = make_float2(-m_used, -m_used);
#pragma unroll
                    for (int e = 0; e < 64; ++e) {
                        const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])), sc2, nm2);
                        const float p0 = ex2(x.x), p1 = ex2(x.y);
                        acc2[e & 1] = __fadd2_rn(acc2[e & 1], make_float2(p0, p1));
                        s[e] = pack_bf16x2(p0, p1);
                    }
                    accs = __fadd2_rn(acc2[0], acc2[1]);
                    exact = __any_sync(0xffffffffu, !(accs.x + accs.y <= 0x1p50f));
                    if (exact) {
                        // the scores were overwritten by P: load them again
                        TMEM_LD32(s_col, s);
                        TMEM_LD32(s_col + 32, (s + 32));
                        TMEM_LD32(s_col + 64, (s + 64));
                        TMEM_LD32(s_col + 96, (s + 96));
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                        if (k0 + BKV - 1 > my_pos) {
#pragma unroll
                            for (int i = 0; i < 128; ++i)
                                if (k0 + i > my_pos) s[i] = __float_as_uint(-INFINITY);
                        }
                    }
                }
                if (exact) {
                    float mx;
                    {
                        float a[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) a[i] = fmaxf(__uint_as_float(s[i]), __uint_as_float(s[i + 8]));
#pragma unroll
                        for (int i = 16; i < 128; i += 16)
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                a[c] = max3f(a[c], __uint_as_float(s[i + c]), __uint_as_float(s[i + 8 + c]));
                        mx = max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
                    }
                    const float mxs = mx * scale_log2;
                    const bool need = mxs > m_used + RESCALE_LOG2;
                    rescale = __any_sync(0xffffffffu, need);
                    if (rescale) {
                        const float m_new = need ? mxs : m_used;
                        corr = ex2(m_used - m_new);
                        l *= corr;
                        m_used = m_new;
                    }
                    float2 acc2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    const float2 nm2 = make_float2(-m_used, -m_used);
#pragma unroll
                    for (int e = 0; e < 64; ++e) {
                        const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])), sc2, nm2);
                        const float p0 = ex2(x.x), p1 = ex2(x.y);
                        acc2[e & 1] = __fadd2_rn(acc2[e & 1], make_float2(p0, p1));
                        s[e] = pack_bf16x2(p0, p1);
                    }
                    accs = __fadd2_rn(acc2[0], acc2[1]);
                }
                // P goes over the first 64 columns of its own S buffer (the scores are in
                // registers; the buffer's next product waits for this block's P.V)
                TMEM_ST32(s_col, s);
                TMEM_ST32(s_col + 32, (s + 32));
                if (rescale && kb > 0) {
                    // O must hold every block before this one: wait for the previous P.V
                    // (the previous block's stage is released when its P.V completes, at most
                    // one use of that stage behind)
                    const uint32_t pv = it - 1;
                    if (!warp_wait_cl(&kv_empty[pv % STAGES2], (pv / STAGES2) & 1, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    fence_after();
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t o[32];
                        TMEM_LD32(o_col + c, o);
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
                        TMEM_ST32(o_col + c, o);
                    }
                }
                l += accs.x + accs.y;
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                fence_before();
                warp_arrive_leader(&p_full[b], rank);
            }
            if (!ok) break;
            // O of this tile is final once the item's last P.V has completed
            if (!warp_wait_cl(&o_full, tl & 1, &abort_flag)) {
                ok = false;
                break;
            }
            fence_after();
            const float inv = 1.f / l;
            bf16* dst = out + (long long)row * (hkv * group * D) + (long long)(m.g * group + (valid ? p % group : 0)) * D;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                TMEM_LD32(o_col + c, o);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (valid) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint32_t w4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w4[e] = pack_bf16x2(__uint_as_float(o[v * 8 + 2 * e]) * inv,
                                                __uint_as_float(o[v * 8 + 2 * e + 1]) * inv);
                        *reinterpret_cast<uint4*>(dst + c + v * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            }
            fence_before();
            warp_arrive_leader(&o_free, rank);
        }
        if (!ok) {
            abort_flag = 1;
            if (lane == 0) set_error(err, BLEND_ETIMEOUT);
        }
    }
    fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag && rank == 0) {
        // let the copies still in flight land (both CTAs' bytes count on these barriers)
        for (int s = 0; s < STAGES2; ++s)
            if (pend_kv[s] >= 0)
                for (long long i = 0; i < SPIN_LIMIT && !mbar_try(&kv_full[s], (uint32_t)pend_kv[s]); ++i) {
                }
        for (int b = 0; b < 2; ++b)
            if (pend_q[b] >= 0)
                for (long long i = 0; i < SPIN_LIMIT && !mbar_try(&q_full[b], (uint32_t)pend_q[b]); ++i) {
                }
    }
    __syncthreads();
    cluster_sync();  // neither CTA leaves while the other may still signal its barriers
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tb), "r"(COLS2) : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;
int g_sms = 0;

bool encode(CUtensorMap* map, int rank, const void* base, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box) {
    cuuint32_t es[3] = {1, 1, 1};
    return g_enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_attn_supported(int head_dim) { return (head_dim == 64 || head_dim == 128) && tc_available(); }

template <int D>
int launch_attn_d(const void* q, int m_cap, int n_req, const int32_t* req_row_end, const int32_t* row_pos,
                  const int32_t* row_tok, int M_max, const void* k_cache, const void* v_cache, long long n_tokens,
                  void* o, int hq, int hkv, int32_t* err, cudaStream_t s) {
    const int group = hq / hkv;
    CUtensorMap mq, mk, mv;
    cuuint64_t qd[2] = {(cuuint64_t)D, (cuuint64_t)hkv * m_cap * group};
    cuuint64_t qs[1] = {(cuuint64_t)D * 2};
    cuuint32_t qb[2] = {64, BQ};
    cuuint64_t kd[3] = {(cuuint64_t)D, (cuuint64_t)hkv, (cuuint64_t)n_tokens};
    cuuint64_t ks[2] = {(cuuint64_t)D * 2, (cuuint64_t)hkv * D * 2};
    cuuint32_t kbx[3] = {64, 1, BKV};
    if (!encode(&mq, 2, q, qd, qs, qb) || !encode(&mk, 3, k_cache, kd, ks, kbx) || !encode(&mv, 3, v_cache, kd, ks, kbx))
        return BLEND_EUNSUPPORTED;
    const long long tiles = (((long long)M_max * group) + BQ - 1) / BQ + n_req;
    const long long items = (long long)hkv * ((tiles + 1) / 2 + n_req);
    const int grid = (int)(items < g_sms ? items : g_sms);
    const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));  // log2(e) / sqrt(d)
    k_attn_tc<D><<<grid, THREADS, AttnCfg<D>::SMEM_BYTES, s>>>(mq, mk, mv, n_req, req_row_end, row_pos, row_tok,
                                                               group, hkv, m_cap, scale_log2, (bf16*)o, err);
    note_launch(1);
    return BLEND_OK;
}

// D = 128 on CTA pairs: clusters of two CTAs, one tile each (k_attn_pair).  Returns
// BLEND_EUNSUPPORTED when no cluster of two such CTAs fits on the device.
int launch_attn_pair(const void* q, int m_cap, int n_req, const int32_t* req_row_end, const int32_t* row_pos,
                     const int32_t* row_tok, int M_max, const void* k_cache, const void* v_cache, long long n_tokens,
                     void* o, int hq, int hkv, int32_t* err, cudaStream_t s) {
    constexpr int D = 128;
    static int max_clusters = -1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(pairk::THREADS2);
    cfg.dynamicSmemBytes = pairk::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (max_clusters < 0) {
        cudaFuncSetAttribute(k_attn_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, pairk::SMEM_BYTES);
        cfg.gridDim = dim3(g_sms);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k_attn_pair, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        max_clusters = n < g_sms / 2 ? n : g_sms / 2;
    }
    if (max_clusters <= 0) return BLEND_EUNSUPPORTED;
    const int group = hq / hkv;
    CUtensorMap mq, mk, mv;
    cuuint64_t qd[2] = {(cuuint64_t)D, (cuuint64_t)hkv * m_cap * group};
    cuuint64_t qs[1] = {(cuuint64_t)D * 2};
    cuuint32_t qb[2] = {64, BQ};
    cuuint64_t kd[3] = {(cuuint64_t)D, (cuuint64_t)hkv, (cuuint64_t)n_tokens};
    cuuint64_t ks[2] = {(cuuint64_t)D * 2, (cuuint64_t)hkv * D * 2};
    cuuint32_t kbx[3] = {64, 1, 64};   // this CTA's 64 keys of a block, one d half
    cuuint32_t vbx[3] = {64, 1, BKV};  // all 128 keys of a block, this CTA's d half
    if (!encode(&mq, 2, q, qd, qs, qb) || !encode(&mk, 3, k_cache, kd, ks, kbx) || !encode(&mv, 3, v_cache, kd, ks, vbx))
        return BLEND_EUNSUPPORTED;
    const long long tiles = (((long long)M_max * group) + BQ - 1) / BQ + n_req;
    const long long items = (long long)hkv * ((tiles + 1) / 2 + n_req);
    const int clusters = (int)(items < max_clusters ? items : max_clusters);
    cfg.gridDim = dim3(2 * clusters);
    const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));  // log2(e) / sqrt(d)
    if (cudaLaunchKernelEx(&cfg, k_attn_pair, mq, mk, mv, n_req, req_row_end, row_pos, row_tok, group, hkv, m_cap,
                           scale_log2, (bf16*)o, err) != cudaSuccess) {
        cudaGetLastError();  // a configuration the device refuses: the single-CTA kernel takes over
        return BLEND_EUNSUPPORTED;
    }
    note_launch(1);
    return BLEND_OK;
}

int launch_attn_tc(const void* q, int m_cap, int n_req, const int32_t* req_row_end, const int32_t* row_pos,
                   const int32_t* row_tok, int M_max, const void* k_cache, const void* v_cache, long long n_tokens,
                   void* o, int hq, int hkv, int head_dim, int32_t* err, cudaStream_t s) {
    if (M_max <= 0) return BLEND_OK;
    if (!g_enc) {
        cudaDriverEntryPointQueryResult qr;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) !=
                cudaSuccess ||
            qr != cudaDriverEntryPointSuccess || !fn)
            return BLEND_EUNSUPPORTED;
        g_enc = (PFN_cuTensorMapEncodeTiled_v12000)fn;
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
        cudaFuncSetAttribute(k_attn_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnCfg<64>::SMEM_BYTES);
        cudaFuncSetAttribute(k_attn_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnCfg<128>::SMEM_BYTES);
    }
    if (head_dim == 64)
        return launch_attn_d<64>(q, m_cap, n_req, req_row_end, row_pos, row_tok, M_max, k_cache, v_cache, n_tokens,
                                 o, hq, hkv, err, s);
    if (head_dim == 128) {
        const int rc = launch_attn_pair(q, m_cap, n_req, req_row_end, row_pos, row_tok, M_max, k_cache, v_cache,
                                        n_tokens, o, hq, hkv, err, s);
        if (rc != BLEND_EUNSUPPORTED) return rc;
        return launch_attn_d<128>(q, m_cap, n_req, req_row_end, row_pos, row_tok, M_max, k_cache, v_cache, n_tokens,
                                  o, hq, hkv, err, s);
    }
    return BLEND_EUNSUPPORTED;
}

}  // namespace blend
