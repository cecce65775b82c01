// Tensor-core importance scores from the query rows' attention (CacheClip blog, "6.2
// Auxiliary-model-guided token selection": a chunk token's score is the mean, over the
// query rows and heads, of the attention weight on it; Cache-Craft notes, 3.2.2: a
// chunk's focus is the same weights summed over its tokens).  Two passes over
// tcgen05 products, bf16 operands, fp32 accumulation:
//
//   k_score_stats   per (query row, head) the softmax maximum and sum over every key
//                   the row sees (prefix, chunks, query rows up to itself).  A work item
//                   is 128 (row, head) pairs of one kv head against one span of at most
//                   SC_SPAN_BLOCKS 128-key blocks; S = Q . K^T (M128 N128, Q from TMEM
//                   where each thread wrote its pair's row, K by TMA) lands in TMEM, one
//                   pair row per thread, and each thread keeps a running base-2 maximum
//                   and sum.  Each span writes one partial (m, l) per pair.
//   k_score_colsum  per 128 chunk keys of a request: for every kv head and pair tile,
//                   S^T = K . Q^T (M128 keys, N128 pairs, both operands in shared
//                   memory), one key per thread; the thread merges the pairs' partials
//                   into (m, 1/l) once per tile (in shared memory) and adds
//                   2^(s - m) / l over the pairs in a fixed order.  No reduction crosses
//                   threads, so the sums are fp32 and run-to-run identical.
//
// Warps: 0 TMA producer, 1 TMEM owner + MMA issuer, 2..5 one TMEM lane quarter each.
// Every mbarrier wait is bounded; on expiry the kernel records BLEND_ETIMEOUT, stops,
// lets its copies land and frees TMEM.
#include <cmath>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "gemm_tc.cuh"

namespace blend {
namespace {

constexpr int SC_THREADS = 192;
constexpr int SC_BLK = 128;         // keys per block
constexpr int SC_STAGES = 3;
constexpr int SC_SPAN_BLOCKS = 8;   // key blocks per statistics span
constexpr long long SC_SPIN = 1ll << 24;
constexpr int SC_HALF_BYTES = SC_BLK * 64 * 2;  // 128 rows x one 64-wide d half: 16 KB

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* b, int c) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(c) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
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
    for (long long i = 0; i < SC_SPIN; ++i) {
        if (mbar_try(b, par)) return true;
        if ((i & 255) == 255 && *abort_flag) return false;
    }
    return false;
}
__device__ __forceinline__ bool warp_wait(uint64_t* b, uint32_t par, volatile int* abort_flag) {
    for (long long i = 0; i < SC_SPIN; ++i) {
        if (__all_sync(0xffffffffu, mbar_try(b, par))) return true;
        if ((i & 255) == 255 && __any_sync(0xffffffffu, *abort_flag != 0)) return false;
    }
    return false;
}
__device__ __forceinline__ void warp_arrive(uint64_t* b) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
            su32(dst)),
        "l"((uint64_t)m), "r"(su32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// K-major operand with the 128-byte swizzle: rows of 64 bf16 (128 B), 8-row groups 1 KB apart.
__device__ __forceinline__ uint64_t desc_k(uint32_t a) {
    return (uint64_t)((a & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// kind::f16, bf16 operands, fp32 accumulate, K-major A and B, M128 N128
constexpr uint32_t SC_IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %3, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, p;\n\t}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(acc), "r"(SC_IDESC)
        : "memory");
}
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %3, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n\t}\n" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(acc), "r"(SC_IDESC)
        : "memory");
}
__device__ __forceinline__ void commit(uint64_t* b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(b))
                 : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
#define SC_LD32(taddr, r)                                                                           \
    asm volatile(                                                                                   \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"  \
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"            \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),    \
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),  \
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),            \
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),            \
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])             \
        : "r"(taddr))
#define SC_ST32(taddr, r)                                                                           \
    asm volatile(                                                                                   \
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),  \
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),     \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), \
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),          \
        "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),          \
        "r"(r[30]), "r"(r[31])                                                                      \
        : "memory")

// Statistics work item w -> request, kv head, pair tile and key span.
struct StatItem {
    int r, g, t, span, nblk_total;
};
__device__ __forceinline__ int stat_tiles(const ReqDesc& rd, int group) { return (rd.Q * group + 127) / 128; }
__device__ __forceinline__ int stat_nblk(const ReqDesc& rd, int group, int t) {
    const int last_q = min(rd.Q - 1, (t * 128 + 127) / group);
    return (rd.P + rd.n_c + last_q) / SC_BLK + 1;
}
__device__ __forceinline__ bool stat_item(int w, const BatchDesc& bd, int group, int hkv, StatItem& it) {
    for (int r = 0; r < bd.n_req; ++r) {
        const ReqDesc& rd = bd.r[r];
        const int tiles = stat_tiles(rd, group);
        // spans per tile from the tile with the longest key range (the last one)
        const int spans = tiles > 0 ? (stat_nblk(rd, group, tiles - 1) + SC_SPAN_BLOCKS - 1) / SC_SPAN_BLOCKS : 0;
        const int n = hkv * tiles * spans;
        if (w < n) {
            it.r = r;
            it.span = w % spans;
            it.t = (w / spans) % tiles;
            it.g = w / (spans * tiles);
            it.nblk_total = stat_nblk(rd, group, it.t);
            return true;
        }
        w -= n;
    }
    return false;
}

// ---------------------------------------------------------------- pass 1: row statistics
template <int D>
__global__ void __launch_bounds__(SC_THREADS, 1)
    k_score_stats(const bf16* __restrict__ q_last, const __grid_constant__ CUtensorMap mapK,
                  const __grid_constant__ BatchDesc bd, int hq, int hkv, float scale_log2, int n_spans,
                  float2* __restrict__ part, int32_t* __restrict__ err) {
    constexpr int NH = D / 64;
    constexpr int STAGE = NH * SC_HALF_BYTES;
    constexpr uint32_t QC = D / 2;  // TMEM columns of one Q buffer (bf16 pairs)
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t kv_full[SC_STAGES], kv_empty[SC_STAGES], s_full[2], s_free[2], q_ready[2],
        q_free[2];
    __shared__ uint32_t tmem_sh;
    __shared__ volatile int abort_flag;
    __shared__ int pend[SC_STAGES];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int group = hq / hkv;
    int total = 0;
    for (int r = 0; r < bd.n_req; ++r) {
        const int tiles = stat_tiles(bd.r[r], group);
        total += tiles > 0 ? hkv * tiles * ((stat_nblk(bd.r[r], group, tiles - 1) + SC_SPAN_BLOCKS - 1) / SC_SPAN_BLOCKS)
                           : 0;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < SC_STAGES; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
            pend[s] = -1;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&s_free[b], 4);
            mbar_init(&q_ready[b], 4);
            mbar_init(&q_free[b], 1);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32(&tmem_sh)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tb = tmem_sh;  // S buffers at 0 and 128, Q buffers at 256 and 256 + QC

    auto blocks_of = [&](const StatItem& m, int& kb0, int& kb1) {
        kb0 = m.span * SC_SPAN_BLOCKS;
        kb1 = min(kb0 + SC_SPAN_BLOCKS, m.nblk_total);
    };
    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer: the item's key blocks of its kv head
        uint32_t it = 0;
        for (int w = blockIdx.x; w < total && !abort_flag; w += gridDim.x) {
            StatItem m;
            stat_item(w, bd, group, hkv, m);
            int kb0, kb1;
            blocks_of(m, kb0, kb1);
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int st = it % SC_STAGES;
                if (!mbar_wait(&kv_empty[st], ((it / SC_STAGES) & 1) ^ 1, &abort_flag)) {
                    abort_flag = 1;
                    set_error(err, BLEND_ETIMEOUT);
                    break;
                }
                mbar_expect_tx(&kv_full[st], STAGE);
                pend[st] = (int)((it / SC_STAGES) & 1);
                const int tok = bd.r[m.r].tok_off + kb * SC_BLK;
                for (int hh = 0; hh < NH; ++hh)
                    tma_3d(smem + st * STAGE + hh * SC_HALF_BYTES, &mapK, &kv_full[st], hh * 64, m.g, tok);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer: S = Q (TMEM) . K^T per block
        uint32_t it = 0;
        bool ok = true;
        for (int w = blockIdx.x, k = 0; w < total && ok && !abort_flag; w += gridDim.x, ++k) {
            StatItem m;
            stat_item(w, bd, group, hkv, m);
            int kb0, kb1;
            blocks_of(m, kb0, kb1);
            const int qb = k & 1;
            if (!mbar_wait(&q_ready[qb], (k >> 1) & 1, &abort_flag)) {
                ok = false;
                break;
            }
            fence_after();
            const uint32_t qa = tb + 256 + qb * QC;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int st = it % SC_STAGES, b = it & 1;
                if (!mbar_wait(&kv_full[st], (it / SC_STAGES) & 1, &abort_flag) ||
                    !mbar_wait(&s_free[b], ((it >> 1) & 1) ^ 1, &abort_flag)) {
                    ok = false;
                    break;
                }
                pend[st] = -1;
                fence_after();
                const uint64_t kd = desc_k(su32(smem + st * STAGE));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32, half = kk >> 2;
                    umma_ts(tb + b * 128, qa + kk * 8, kd + ((half * SC_HALF_BYTES + off) >> 4), kk > 0 ? 1u : 0u);
                }
                commit(&kv_empty[st]);
                commit(&s_full[b]);
            }
            if (!ok) break;
            commit(&q_free[qb]);
        }
        if (!ok) {
            abort_flag = 1;
            set_error(err, BLEND_ETIMEOUT);
        }
    } else if (warp >= 2) {
        // ---------------- one pair row per thread
        const int sp = warp & 3;
        const int row = sp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
        uint32_t it = 0;
        bool ok = true;
        for (int w = blockIdx.x, k = 0; w < total && ok; w += gridDim.x, ++k) {
            StatItem m;
            stat_item(w, bd, group, hkv, m);
            const ReqDesc& rd = bd.r[m.r];
            int kb0, kb1;
            blocks_of(m, kb0, kb1);
            const int pi = m.t * 128 + row;
            const int ql = pi / group, j = pi % group;
            const bool valid = ql < rd.Q;
            const int pos = rd.P + rd.n_c + (valid ? ql : 0);
            // this pair's q row into Q buffer k & 1 (zeros for a pair past the request)
            const int qb = k & 1;
            if (!warp_wait(&q_free[qb], ((k >> 1) & 1) ^ 1, &abort_flag)) {
                ok = false;
                break;
            }
            fence_after();
            {
                uint32_t v[D / 2];
                if (valid) {
                    const uint4* src = reinterpret_cast<const uint4*>(q_last + ((long long)(rd.q_off + ql) * hq + m.g * group + j) * D);
#pragma unroll
                    for (int i = 0; i < D / 8; ++i) {
                        const uint4 x = src[i];
                        v[4 * i] = x.x;
                        v[4 * i + 1] = x.y;
                        v[4 * i + 2] = x.z;
                        v[4 * i + 3] = x.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < D / 2; ++i) v[i] = 0u;
                }
                const uint32_t qc = tb + lane_off + 256 + qb * QC;
#pragma unroll
                for (int c = 0; c < D / 2; c += 32) SC_ST32(qc + c, (v + c));
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            fence_before();
            warp_arrive(&q_ready[qb]);
            float m2 = -INFINITY, l = 0.f;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int b = it & 1;
                if (!warp_wait(&s_full[b], (it >> 1) & 1, &abort_flag)) {
                    ok = false;
                    break;
                }
                fence_after();
                uint32_t s[128];
                const uint32_t sc = tb + lane_off + b * 128;
                SC_LD32(sc, s);
                SC_LD32(sc + 32, (s + 32));
                SC_LD32(sc + 64, (s + 64));
                SC_LD32(sc + 96, (s + 96));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                fence_before();
                warp_arrive(&s_free[b]);
                const int k0 = kb * SC_BLK;
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < 128; ++i) {
                    const float x = (k0 + i <= pos) ? __uint_as_float(s[i]) * scale_log2 : -INFINITY;
                    s[i] = __float_as_uint(x);
                    mx = fmaxf(mx, x);
                }
                if (mx > -INFINITY) {
                    const float mn = fmaxf(m2, mx);
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < 128; ++i) acc += ex2(__uint_as_float(s[i]) - mn);
                    l = (m2 == -INFINITY ? 0.f : l * ex2(m2 - mn)) + acc;
                    m2 = mn;
                }
            }
            if (!ok) break;
            if (valid) part[((long long)(rd.q_off + ql) * hq + m.g * group + j) * n_spans + m.span] = make_float2(m2, l);
        }
        if (!ok) {
            abort_flag = 1;
            if (lane == 0) set_error(err, BLEND_ETIMEOUT);
        }
    }
    fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) {
        for (int s = 0; s < SC_STAGES; ++s)
            if (pend[s] >= 0)
                for (long long i = 0; i < SC_SPIN && !mbar_try(&kv_full[s], (uint32_t)pend[s]); ++i) {
                }
    }
    __syncthreads();
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tb) : "memory");
    }
}

// ---------------------------------------------------------------- pass 2: column means
// Work item w -> request and its 128-key chunk block.
__device__ __forceinline__ bool col_item(int w, const BatchDesc& bd, int& r, int& kb) {
    for (r = 0; r < bd.n_req; ++r) {
        const int n = (bd.r[r].n_c + SC_BLK - 1) / SC_BLK;
        if (w < n) {
            kb = w;
            return true;
        }
        w -= n;
    }
    return false;
}

template <int D>
__global__ void __launch_bounds__(SC_THREADS, 1)
    k_score_colsum(const bf16* __restrict__ q_last, const __grid_constant__ CUtensorMap mapK,
                   const __grid_constant__ BatchDesc bd, int hq, int hkv, float scale_log2, int n_spans,
                   const float2* __restrict__ part, float* __restrict__ scores, int32_t* __restrict__ err) {
    constexpr int NH = D / 64;
    constexpr int KT = NH * SC_HALF_BYTES;  // one 128-row operand tile (keys or pairs)
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t k_full[2], k_empty[2], s_full[2], s_free[2], q_ready[2], q_free[2];
    __shared__ float2 st_sh[2][128];  // per pair of the tile: (max, 1 / sum), max = +inf for no pair
    __shared__ uint32_t tmem_sh;
    __shared__ volatile int abort_flag;
    __shared__ int pend[2];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sK = smem;           // key tile buffer b at b * KT
    uint8_t* sQ = smem + 2 * KT;  // pair tile buffer b at b * KT
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int group = hq / hkv;
    int total = 0;
    for (int r = 0; r < bd.n_req; ++r) total += (bd.r[r].n_c + SC_BLK - 1) / SC_BLK;
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&k_full[b], 1);
            mbar_init(&k_empty[b], 1);
            mbar_init(&s_full[b], 1);
            mbar_init(&s_free[b], 4);
            mbar_init(&q_ready[b], 4);
            mbar_init(&q_free[b], 1);
            pend[b] = -1;
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(su32(&tmem_sh)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tb = tmem_sh;  // S^T buffers at 0 and 128

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer: the item's 128 keys, once per kv head
        uint32_t kt = 0;
        for (int w = blockIdx.x; w < total && !abort_flag; w += gridDim.x) {
            int r, kb;
            col_item(w, bd, r, kb);
            const int tok = bd.r[r].tok_off + bd.r[r].P + kb * SC_BLK;
            for (int g = 0; g < hkv; ++g, ++kt) {
                const int b = kt & 1;
                if (!mbar_wait(&k_empty[b], ((kt >> 1) & 1) ^ 1, &abort_flag)) {
                    abort_flag = 1;
                    set_error(err, BLEND_ETIMEOUT);
                    break;
                }
                mbar_expect_tx(&k_full[b], KT);
                pend[b] = (int)((kt >> 1) & 1);
                for (int hh = 0; hh < NH; ++hh)
                    tma_3d(sK + b * KT + hh * SC_HALF_BYTES, &mapK, &k_full[b], hh * 64, g, tok);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer: S^T = K . Q^T per (kv head, pair tile)
        uint32_t kt = 0, qt = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < total && ok && !abort_flag; w += gridDim.x) {
            int r, kb;
            col_item(w, bd, r, kb);
            const int tiles = stat_tiles(bd.r[r], group);
            for (int g = 0; g < hkv && ok; ++g, ++kt) {
                const int b = kt & 1;
                if (!mbar_wait(&k_full[b], (kt >> 1) & 1, &abort_flag)) {
                    ok = false;
                    break;
                }
                pend[b] = -1;
                for (int t = 0; t < tiles; ++t, ++qt) {
                    const int qb = qt & 1;
                    if (!mbar_wait(&q_ready[qb], (qt >> 1) & 1, &abort_flag) ||
                        !mbar_wait(&s_free[qb], ((qt >> 1) & 1) ^ 1, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint64_t kd = desc_k(su32(sK + b * KT)), qd = desc_k(su32(sQ + qb * KT));
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk & 3) * 32, half = kk >> 2;
                        umma_ss(tb + qb * 128, kd + ((half * SC_HALF_BYTES + off) >> 4),
                                qd + ((half * SC_HALF_BYTES + off) >> 4), kk > 0 ? 1u : 0u);
                    }
                    commit(&q_free[qb]);
                    commit(&s_full[qb]);
                }
                commit(&k_empty[b]);
            }
        }
        if (!ok) {
            abort_flag = 1;
            set_error(err, BLEND_ETIMEOUT);
        }
    } else if (warp >= 2) {
        // ---------------- thread = one key of the block (TMEM lane), and one pair for
        // the tile's q rows and statistics
        const int sp = warp & 3;
        const int row = sp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
        uint32_t qt = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
            int r, kb;
            col_item(w, bd, r, kb);
            const ReqDesc& rd = bd.r[r];
            const int tiles = stat_tiles(rd, group);
            float acc = 0.f;
            for (int g = 0; g < hkv && ok; ++g) {
                for (int t = 0; t < tiles; ++t, ++qt) {
                    const int qb = qt & 1;
                    // this thread's pair: q row into the pair tile (swizzled K-major rows),
                    // merged statistics into shared memory
                    if (!warp_wait(&q_free[qb], ((qt >> 1) & 1) ^ 1, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    {
                        const int pi = t * 128 + row;
                        const int ql = pi / group, j = pi % group;
                        const bool valid = ql < rd.Q;
                        const long long pr = (long long)(rd.q_off + (valid ? ql : 0)) * hq + g * group + j;
                        uint8_t* dst = sQ + qb * KT;
#pragma unroll
                        for (int i = 0; i < D / 8; ++i) {
                            const uint4 x = valid ? reinterpret_cast<const uint4*>(q_last + pr * D)[i] : make_uint4(0, 0, 0, 0);
                            const int hh = i / 8, c16 = i % 8;  // d half, 16-byte piece within the 128-byte row
                            *reinterpret_cast<uint4*>(dst + hh * SC_HALF_BYTES + row * 128 + ((c16 ^ (row & 7)) << 4)) = x;
                        }
                        float2 st = make_float2(INFINITY, 0.f);
                        if (valid) {
                            // merge the spans' partials in span order
                            const int spans = (stat_nblk(rd, group, t) + SC_SPAN_BLOCKS - 1) / SC_SPAN_BLOCKS;
                            float mm = -INFINITY, ll = 0.f;
                            for (int c = 0; c < spans; ++c) {
                                const float2 pc = part[pr * n_spans + c];
                                if (pc.x == -INFINITY) continue;
                                const float mn = fmaxf(mm, pc.x);
                                ll = (mm == -INFINITY ? 0.f : ll * ex2(mm - mn)) + pc.y * ex2(pc.x - mn);
                                mm = mn;
                            }
                            st = make_float2(mm, 1.f / ll);
                        }
                        st_sh[qb][row] = st;
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    warp_arrive(&q_ready[qb]);
                    // every warp's pairs are in shared memory once all four have arrived (a
                    // warp reaches tile qt + 2, which rewrites this buffer, only after all
                    // four arrived for tile qt + 1, i.e. after they finished reading this one);
                    // then the tile's products: this key against the 128 pairs
                    if (!warp_wait(&q_ready[qb], (qt >> 1) & 1, &abort_flag) ||
                        !warp_wait(&s_full[qb], (qt >> 1) & 1, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    uint32_t s[128];
                    const uint32_t sc = tb + lane_off + qb * 128;
                    SC_LD32(sc, s);
                    SC_LD32(sc + 32, (s + 32));
                    SC_LD32(sc + 64, (s + 64));
                    SC_LD32(sc + 96, (s + 96));
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    fence_before();
                    warp_arrive(&s_free[qb]);
#pragma unroll
                    for (int i = 0; i < 128; ++i) {
                        const float2 st = st_sh[qb][i];  // same address in every lane
                        acc += ex2(fmaf(__uint_as_float(s[i]), scale_log2, -st.x)) * st.y;
                    }
                }
            }
            if (!ok) break;
            const int j = kb * SC_BLK + row;
            if (j < rd.n_c) scores[rd.nc_off + j] = acc / (float)(rd.Q * hq);
        }
        if (!ok) {
            abort_flag = 1;
            if (lane == 0) set_error(err, BLEND_ETIMEOUT);
        }
    }
    fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) {
        for (int b = 0; b < 2; ++b)
            if (pend[b] >= 0)
                for (long long i = 0; i < SC_SPIN && !mbar_try(&k_full[b], (uint32_t)pend[b]); ++i) {
                }
    }
    __syncthreads();
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tb) : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_sc_enc = nullptr;
int g_sc_sms = 0;

template <int D>
int launch_scores_d(const void* q_last, const void* K, long long n_tokens, const BatchDesc& bd, int hq, int hkv,
                    int n_spans, float2* part, float* scores, int32_t* err, cudaStream_t s) {
    constexpr int NH = D / 64;
    CUtensorMap mk;
    cuuint64_t kd[3] = {(cuuint64_t)D, (cuuint64_t)hkv, (cuuint64_t)n_tokens};
    cuuint64_t ks[2] = {(cuuint64_t)D * 2, (cuuint64_t)hkv * D * 2};
    cuuint32_t kbx[3] = {64, 1, SC_BLK};
    cuuint32_t es[3] = {1, 1, 1};
    if (g_sc_enc(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(K), kd, ks, kbx, es,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return BLEND_EUNSUPPORTED;
    const int group = hq / hkv;
    long long items1 = 0, items2 = 0;
    for (int r = 0; r < bd.n_req; ++r) {
        const ReqDesc& rd = bd.r[r];
        const int tiles = (rd.Q * group + 127) / 128;
        if (tiles > 0) {
            const int last_q = std::min(rd.Q - 1, ((tiles - 1) * 128 + 127) / group);
            const int nblk = (rd.P + rd.n_c + last_q) / SC_BLK + 1;
            items1 += (long long)hkv * tiles * ((nblk + SC_SPAN_BLOCKS - 1) / SC_SPAN_BLOCKS);
        }
        items2 += (rd.n_c + SC_BLK - 1) / SC_BLK;
    }
    const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    if (items1 > 0) {
        const int grid = (int)std::min<long long>(items1, g_sc_sms);
        k_score_stats<D><<<grid, SC_THREADS, SC_STAGES * NH * SC_HALF_BYTES + 1024, s>>>(
            (const bf16*)q_last, mk, bd, hq, hkv, scale_log2, n_spans, part, err);
        note_launch(1);
    }
    if (items2 > 0) {
        const int grid = (int)std::min<long long>(items2, g_sc_sms);
        k_score_colsum<D><<<grid, SC_THREADS, 4 * NH * SC_HALF_BYTES + 1024, s>>>(
            (const bf16*)q_last, mk, bd, hq, hkv, scale_log2, n_spans, part, scores, err);
        note_launch(1);
    }
    return BLEND_OK;
}

}  // namespace

int tc_score_spans(long long max_tokens) { return (int)((max_tokens + SC_BLK * SC_SPAN_BLOCKS - 1) / (SC_BLK * SC_SPAN_BLOCKS)); }

int launch_scores_tc(const void* q_last, const void* K, long long n_tokens, const BatchDesc& bd, int hq, int hkv,
                     int d, int n_spans, float2* part, float* scores, int32_t* err, cudaStream_t s) {
    if (d != 64 && d != 128) return BLEND_EUNSUPPORTED;
    if (((uintptr_t)q_last & 15) != 0 || !tc_available()) return BLEND_EUNSUPPORTED;
    if (!g_sc_enc) {
        cudaDriverEntryPointQueryResult qr;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) !=
                cudaSuccess ||
            qr != cudaDriverEntryPointSuccess || !fn)
            return BLEND_EUNSUPPORTED;
        g_sc_enc = (PFN_cuTensorMapEncodeTiled_v12000)fn;
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_sc_sms, cudaDevAttrMultiProcessorCount, dev);
        cudaFuncSetAttribute(k_score_stats<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, SC_STAGES * SC_HALF_BYTES + 1024);
        cudaFuncSetAttribute(k_score_stats<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SC_STAGES * 2 * SC_HALF_BYTES + 1024);
        cudaFuncSetAttribute(k_score_colsum<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, 4 * SC_HALF_BYTES + 1024);
        cudaFuncSetAttribute(k_score_colsum<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             8 * SC_HALF_BYTES + 1024);
    }
    if (d == 64) return launch_scores_d<64>(q_last, K, n_tokens, bd, hq, hkv, n_spans, part, scores, err, s);
    return launch_scores_d<128>(q_last, K, n_tokens, bd, hq, hkv, n_spans, part, scores, err, s);
}

}  // namespace blend
