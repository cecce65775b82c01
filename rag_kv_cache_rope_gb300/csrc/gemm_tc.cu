// Tensor-core GEMM for the gathered-row projections: C = A . B^T, A [M][K] bf16
// (recomputed rows), B [N][K] bf16 (weights, nn.Linear layout), fp32 accumulation in
// TMEM, fused epilogues (fp32 store, fp32 residual add, SwiGLU).
//
// Persistent kernel, one CTA per SM, 6 warps:
//   warp 0      TMA producer: 128x64 A tile + 256x64 B tile per stage (128-byte swizzle)
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma kind::f16, M=128 N=256 K=16,
//               4 per stage; tcgen05.commit frees the stage / publishes the accumulator
//   warps 2..5  epilogue: tcgen05.ld of their 32 TMEM lanes (one output row per thread);
//               fp32 store, fp32 residual add, SwiGLU, or the QKV epilogue (RoPE at each
//               row's position, q to its per-kv-head slab, k and v into the KV cache)
// Two 256-column fp32 accumulators (all 512 TMEM columns) let the epilogue of one tile
// overlap the main loop of the next.  M is read from the device; tiles past it are
// skipped.
// Tail split: tiles are dealt to the persistent CTAs (or CTA pairs) in waves.  When the
// last wave is at most half full, each of its tiles is cut into two K halves run by two
// units, so that wave takes half a tile's time.  Each half stores its raw fp32 partial
// tile to a workspace with tensor stores; k_split_combine then adds the two partials in
// a fixed order and runs the tile's epilogue (no CTA waits for another; column halves
// were measured to take as long as whole tiles).
// Residual-add epilogues of warps whose 32 rows are all live stage each 32-column chunk
// in shared memory and leave it as tensor stores.  Every mbarrier wait is bounded: on
// expiry the kernel records BLEND_ETIMEOUT in the error word, stops issuing work, drains
// its own copies and frees TMEM before returning.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gemm_tc.cuh"

namespace blend {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int THREADS = 192;
constexpr long long SPIN_LIMIT = 1ll << 24;
// Tile shape per N-tile width: 128x256 tiles with 4 stages of 48 KB, or 128x128 tiles
// with 6 stages of 32 KB (used where 256-wide tiles leave the last wave mostly empty).
// PAIR: a cluster of two CTAs computes a 256x256 tile with cta_group::2 MMAs; each CTA
// stages its own 128 rows of A and half of the tile's weight rows (6 stages of 32 KB),
// so per SM the operand bytes per FLOP are two thirds of the single-CTA tile's.
template <int BN, bool PAIR = false> struct TileCfg {
    static constexpr int TM = PAIR ? 2 * BM : BM;     // tile rows
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // weight rows one CTA stages for a whole tile
    static constexpr int B_BYTES = B_ROWS * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (PAIR || BN != 256) ? 6 : 4;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;  // + alignment slack
    // kind::f16 instruction descriptor: bf16 A and B (K-major), fp32 D, M = TM, N = BN
    static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((BN >> 3) << 17) | ((TM >> 4) << 24);
};
// Residual-add epilogue staging: per epilogue warp one 32-row x 32-column chunk of the
// fp32 sum (4 KB, 128-byte swizzle) and of bf16(x * g) (2 KB, 64-byte swizzle), which the
// TMA unit stores while the warp computes the next chunk.
constexpr int OUT_F32_BYTES = 32 * 32 * 4;
constexpr int OUT_WARP_BYTES = OUT_F32_BYTES + 32 * 32 * 2;
// staging for the residual-add epilogue and for the partials of split tiles
template <int EPI, int BN, bool PAIR = false> constexpr int smem_bytes() {
    return TileCfg<BN, PAIR>::SMEM_BYTES + (EPI != EPI_QKV_ROPE ? 4 * OUT_WARP_BYTES : 0);
}
// Split-tile workspace: up to GEMM_SPLIT_SMS / 2 split tiles, two K halves each, of
// 128 x 256 fp32 per 128-row block (a CTA pair's tile has two).
constexpr int GEMM_SPLIT_SMS = 160;

__device__ __forceinline__ uint32_t su32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(su32(dst)),
        "l"((uint64_t)map), "r"(su32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// Tensor store of a shared-memory box to global memory (bulk async-group of the
// issuing thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     (uint64_t)map),
                 "r"(su32(src)), "r"(c0), "r"(c1)
                 : "memory");
}

// Shared-memory matrix descriptor of a K-major tile stored with the 128-byte swizzle
// (rows of 64 bf16 = 128 bytes, 8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);  // start address
    d |= (uint64_t)1 << 16;                   // leading byte offset (unused with swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                   // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                   // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     su32(bar))
                 : "memory");
}
// ---- CTA-pair forms (cluster of two CTAs, rank 0 leads)
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of the same variable in the leading CTA
__device__ __forceinline__ uint32_t leader_addr(const void* p) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(su32(p)));
    return r;
}
// tensor load into this CTA's shared memory whose bytes count on the leader's barrier
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(su32(dst)),
        "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// arrive on the barrier at this address in both CTAs once the issued MMAs complete
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            su32(bar)),
        "h"((uint16_t)3)
        : "memory");
}
// arrive on a barrier of either CTA (default semantics; a cluster-scope release here was
// measured to cost ~1 K cycles)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Non-blocking test of the phase at cluster scope: a blocking try_wait on a barrier that
// the other CTA signals was measured to resume up to ~1.5 K cycles after the phase
// completed.
__device__ __forceinline__ bool mbar_test_cluster(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase of parity `parity`; false if it did not complete in time or
// another role gave up.  PAIR polls at cluster scope (the other CTA's arrivals and copies).
template <bool PAIR>
__device__ __forceinline__ bool mbar_wait_t(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
    const long long limit = PAIR ? 64 * SPIN_LIMIT : SPIN_LIMIT;
    for (long long i = 0; i < limit; ++i) {
        if (PAIR ? mbar_test_cluster(b, parity) : mbar_try(b, parity)) return true;
        if ((i & 1023) == 1023 && *abort_flag) return false;
    }
    return false;
}

// Work unit u -> tile, its K-block range and, for a unit of a split tile, which K part
// (-1: whole tile) and the split tile's index.
struct Unit {
    int t, half, sidx, k0, k1;
};
// Splitting (allowed for the non-QKV epilogues with 256-wide tiles and a workspace) is
// decided on the device from the device row count, identically in the GEMM and in
// k_split_combine:
//   n_total >= grid: the tiles of a last wave that is at most half full run as two K halves;
//   n_total <  grid: every tile may run as S = 2..4 K parts, in ceil(S n_total / grid) rounds
//                    of 1/S of a tile; S is the one with the fewest tile-times (ties: fewer
//                    parts), used only if that beats one whole round, and its partials fit
//                    the workspace (ws_blocks TM-row blocks).
// A split tile's parts are finished by k_split_combine.
struct Sched {
    int full;   // units dealt as whole tiles
    int split;  // split tiles
    int parts;  // K parts of a split tile
    int units;
};
__device__ __forceinline__ Sched make_sched(int n_total, int grid, bool can_split, int kblocks, int ws_blocks) {
    Sched sc;
    sc.parts = 2;
    sc.split = 0;
    if (can_split && kblocks >= 2 && n_total > 0) {
        if (n_total >= grid) {
            const int rem = n_total % grid;
            if (rem > 0 && 2 * rem <= grid) sc.split = rem;
        } else {
            int best_s = 1;
            long long best_num = 1, best_den = 1;  // tile-times of the best S: num / den
            for (int S = 2; S <= 4 && S <= kblocks && S * n_total <= ws_blocks; ++S) {
                const long long rounds = (S * n_total + grid - 1) / grid;
                if (rounds * best_den < best_num * S) {
                    best_num = rounds;
                    best_den = S;
                    best_s = S;
                }
            }
            if (best_s > 1) {
                sc.parts = best_s;
                sc.split = n_total;
            }
        }
    }
    sc.full = n_total - sc.split;
    sc.units = sc.full + sc.parts * sc.split;
    return sc;
}
__device__ __forceinline__ Unit unit_of(int u, const Sched& sc, int kblocks) {
    Unit r;
    if (u < sc.full) {
        r.t = u;
        r.half = -1;
        r.sidx = -1;
        r.k0 = 0;
        r.k1 = kblocks;
    } else {
        const int v = u - sc.full;
        r.sidx = v / sc.parts;
        r.t = sc.full + r.sidx;
        r.half = v % sc.parts;
        r.k0 = r.half * kblocks / sc.parts;
        r.k1 = (r.half + 1) * kblocks / sc.parts;
    }
    return r;
}

// Two fp32 values to one register of two bf16 (round to nearest even), lo in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

#define TMEM_LD32(taddr, r)                                                                        \
    asm volatile(                                                                                  \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"           \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),   \
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),           \
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),           \
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])            \
        : "r"(taddr))

// Row scale of the consumer side of NormEpi (1 when the GEMM reads normalised rows).
__device__ __forceinline__ float row_scale(const NormEpi& ne, int row) {
    if (ne.ssq_in == nullptr) return 1.f;
    float t = 0.f;
    for (int q = 0; q < ne.n_part; ++q) t += ne.ssq_in[(long long)row * ne.n_part + q];
    return 1.f / sqrtf(t * ne.inv_h + ne.eps);
}

// Epilogue of 32 accumulator columns of one row (fp32 store, fp32 residual add, or
// SwiGLU of 16 gate + 16 up columns to 16 bf16 outputs), after the row scale rs.  A
// residual add with ne.x_out also writes bf16(x * g) and adds the squares of the new row
// values to ssq (in column order).
template <int EPI>
__device__ __forceinline__ void epi_chunk(const uint32_t* r, int row, int col, void* Cv, int ldc, float rs,
                                          const NormEpi& ne, float& ssq) {
    if (EPI == EPI_STORE_F32 || EPI == EPI_ADD_F32) {
        float4* p = reinterpret_cast<float4*>((float*)Cv + (long long)row * ldc + col);
        float o[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            float4 w = make_float4(__uint_as_float(r[4 * v]) * rs, __uint_as_float(r[4 * v + 1]) * rs,
                                   __uint_as_float(r[4 * v + 2]) * rs, __uint_as_float(r[4 * v + 3]) * rs);
            if (EPI == EPI_ADD_F32) {
                const float4 x = p[v];
                w.x += x.x;
                w.y += x.y;
                w.z += x.z;
                w.w += x.w;
            }
            p[v] = w;
            o[4 * v] = w.x;
            o[4 * v + 1] = w.y;
            o[4 * v + 2] = w.z;
            o[4 * v + 3] = w.w;
        }
        if (EPI == EPI_ADD_F32 && ne.x_out != nullptr) {
            const uint4* gp = reinterpret_cast<const uint4*>(ne.g + col);
            uint4* xp = reinterpret_cast<uint4*>(ne.x_out + (long long)row * ne.ldx + col);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 gv = gp[v];
                const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
                uint32_t xw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = o[8 * v + 2 * e], b = o[8 * v + 2 * e + 1];
                    ssq = fmaf(a, a, ssq);
                    ssq = fmaf(b, b, ssq);
                    const float ga = __uint_as_float(gw[e] << 16), gb = __uint_as_float(gw[e] & 0xffff0000u);
                    xw[e] = pack_bf16x2(a * ga, b * gb);
                }
                xp[v] = make_uint4(xw[0], xw[1], xw[2], xw[3]);
            }
        }
    } else {
        // 32 columns = 16 gate + 16 up of the same hidden units
        uint32_t w8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float g0 = __uint_as_float(r[2 * i]) * rs, u0 = __uint_as_float(r[16 + 2 * i]) * rs;
            const float g1 = __uint_as_float(r[2 * i + 1]) * rs, u1 = __uint_as_float(r[17 + 2 * i]) * rs;
            w8[i] = pack_bf16x2(g0 / (1.f + expf(-g0)) * u0, g1 / (1.f + expf(-g1)) * u1);
        }
        uint4* p = reinterpret_cast<uint4*>((bf16*)Cv + (long long)row * ldc + col / 2);
        p[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
        p[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
    }
}

// Residual-add epilogue of 32 accumulator columns of the warp's 32 rows (row0 + lane)
// through the warp's staging chunk cb: the fp32 sum x + rs * acc and, with ne.x_out,
// bf16(sum * g) are written to shared memory in the TMA unit's swizzled layout and leave
// as tensor stores of whole 32 x 32 boxes (full lines, no per-thread global stores).  xr
// holds the thread's 32 residual values.  The chunk is reused once the previous stores
// have read it.
__device__ __forceinline__ void add_chunk_tma(const uint32_t* r, const float4* xr, int row0, int col, float rs,
                                              const NormEpi& ne, uint8_t* cb, const CUtensorMap* mapC,
                                              const CUtensorMap* mapX, float& ssq) {
    const int lane = threadIdx.x & 31;
    float o[32];
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        float4 w = make_float4(__uint_as_float(r[4 * v]) * rs, __uint_as_float(r[4 * v + 1]) * rs,
                               __uint_as_float(r[4 * v + 2]) * rs, __uint_as_float(r[4 * v + 3]) * rs);
        w.x += xr[v].x;
        w.y += xr[v].y;
        w.z += xr[v].z;
        w.w += xr[v].w;
        o[4 * v] = w.x;
        o[4 * v + 1] = w.y;
        o[4 * v + 2] = w.z;
        o[4 * v + 3] = w.w;
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    __syncwarp();
    // 128-byte swizzle: 16-byte piece j of row i sits at piece j ^ (i % 8)
    uint8_t* rowp = cb + lane * 128;
#pragma unroll
    for (int v = 0; v < 8; ++v)
        *reinterpret_cast<float4*>(rowp + ((v ^ (lane & 7)) << 4)) =
            make_float4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
    const bool has_x = ne.x_out != nullptr;
    if (has_x) {
        // 64-byte swizzle over 64-byte rows: piece j of row i sits at piece j ^ ((i / 2) % 4)
        const uint4* gp = reinterpret_cast<const uint4*>(ne.g + col);
        uint8_t* xrow = cb + OUT_F32_BYTES + lane * 64;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint4 gv = gp[v];
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
            uint32_t xw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a = o[8 * v + 2 * e], b = o[8 * v + 2 * e + 1];
                ssq = fmaf(a, a, ssq);
                ssq = fmaf(b, b, ssq);
                const float ga = __uint_as_float(gw[e] << 16), gb = __uint_as_float(gw[e] & 0xffff0000u);
                xw[e] = pack_bf16x2(a * ga, b * gb);
            }
            *reinterpret_cast<uint4*>(xrow + ((v ^ ((lane >> 1) & 3)) << 4)) = make_uint4(xw[0], xw[1], xw[2], xw[3]);
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(mapC, cb, col, row0);
        if (has_x) tma_store_2d(mapX, cb + OUT_F32_BYTES, col, row0);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
}

// Raw fp32 partial of 32 accumulator columns of the warp's 32 rows (a K half of a split
// tile) through the warp's staging chunk into the split workspace (tensor store).
__device__ __forceinline__ void part_chunk_tma(const uint32_t* r, int ws_row0, int col, uint8_t* cb,
                                               const CUtensorMap* mapW) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    __syncwarp();
    uint8_t* rowp = cb + lane * 128;
#pragma unroll
    for (int v = 0; v < 8; ++v)
        *reinterpret_cast<uint4*>(rowp + ((v ^ (lane & 7)) << 4)) = make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(mapW, cb, col, ws_row0);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
}

template <int EPI, int BN, bool PAIR>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB, int K, int N,
              const int32_t* __restrict__ M_dev,
              void* __restrict__ Cv, int ldc, int32_t* __restrict__ err, const __grid_constant__ QkvEpi qe,
              int can_split, const __grid_constant__ NormEpi ne, const __grid_constant__ CUtensorMap mapC,
              const __grid_constant__ CUtensorMap mapX, int tma_out, const __grid_constant__ CUtensorMap mapW) {
    using TC = TileCfg<BN, PAIR>;
    constexpr int STAGES = TC::STAGES;
    constexpr int STAGE_BYTES = TC::STAGE_BYTES;
    constexpr int TMEM_COLS = TC::TMEM_COLS;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;
    __shared__ int pending[STAGES];  // parity a stage's last issued load completes with, or -1

    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // a CTA pair works as one unit: units are dealt per cluster, rank 1 takes rows 128..255
    const int rank = PAIR ? (int)cluster_rank() : 0;
    const int grp = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int n_grp = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const int M = *M_dev;
    const int m_tiles = (M + TC::TM - 1) / TC::TM, n_tiles = (N + BN - 1) / BN;  // the last N-tile may be partial
    const int n_total = m_tiles * n_tiles;
    const int kblocks = K / BK;
    constexpr int HALF = BN / 2;
    const Sched sc = make_sched(n_total, n_grp, EPI != EPI_QKV_ROPE && BN == 256 && can_split != 0, kblocks,
                                (int)(GEMM_SPLIT_WS_FLOATS / 256 / TC::TM));

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            pending[s] = -1;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], PAIR ? 8 : 4);  // one arrival per epilogue warp (of both CTAs)
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        // a pair allocates collectively: one warp of each CTA, the same columns in both
        if (PAIR) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             su32(&tmem_base_sh)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             su32(&tmem_base_sh)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    // both CTAs' barriers are initialised before either signals the other's
    if (PAIR) cluster_sync();
    tc_fence_after();
    const uint32_t tbase = tmem_base_sh;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        int s = 0;
        uint32_t ph = 0;
        for (int u = grp; u < sc.units && !abort_flag; u += n_grp) {
            const Unit un = unit_of(u, sc, kblocks);
            const int mt = un.t % m_tiles, nt = un.t / m_tiles;
            // this CTA's A rows and its share of the weight rows, over the unit's K range
            const int brow = nt * BN + rank * TC::B_ROWS;
            const int arow = mt * TC::TM + rank * BM;
            const uint32_t bytes = (uint32_t)(A_BYTES + TC::B_ROWS * BK * 2);
            for (int kb = un.k0; kb < un.k1; ++kb) {
                if (!mbar_wait_t<PAIR>(&empty[s], ph ^ 1, &abort_flag)) {
                    abort_flag = 1;
                    set_error(err, BLEND_ETIMEOUT);
                    break;
                }
                uint8_t* st = smem + s * STAGE_BYTES;
                if (PAIR) {
                    // both CTAs' copies count on the leader's barrier, which expects them all
                    if (rank == 0) {
                        mbar_expect_tx(&full[s], 2 * bytes);
                        pending[s] = (int)ph;
                    }
                    const uint32_t fb = leader_addr(&full[s]);
                    tma_load_2d_pair(st, &mapA, fb, kb * BK, arow);
                    tma_load_2d_pair(st + A_BYTES, &mapB, fb, kb * BK, brow);
                } else {
                    mbar_expect_tx(&full[s], bytes);
                    pending[s] = (int)ph;
                    tma_load_2d(st, &mapA, &full[s], kb * BK, arow);
                    tma_load_2d(st + A_BYTES, &mapB, &full[s], kb * BK, brow);
                }
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ---------------- MMA issuer (the leading CTA of a pair issues for both)
        int s = 0, b = 0;
        uint32_t ph = 0, tph = 0;
        for (int u = grp; u < sc.units && !abort_flag; u += n_grp) {
            const Unit un = unit_of(u, sc, kblocks);
            const uint32_t idesc = TC::IDESC;
            if (!mbar_wait_t<PAIR>(&tempty[b], tph ^ 1, &abort_flag)) {
                abort_flag = 1;
                set_error(err, BLEND_ETIMEOUT);
                break;
            }
            tc_fence_after();
            const uint32_t d = tbase + (uint32_t)(b * BN);
            for (int kb = un.k0; kb < un.k1; ++kb) {
                if (!mbar_wait_t<PAIR>(&full[s], ph, &abort_flag)) {
                    abort_flag = 1;
                    set_error(err, BLEND_ETIMEOUT);
                    break;
                }
                tc_fence_after();
                pending[s] = -1;
                const uint32_t a_addr = su32(smem + s * STAGE_BYTES);
                const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    if (PAIR)
                        umma_bf16_pair(d, sdesc_sw128(a_addr + kk * 32), sdesc_sw128(b_addr + kk * 32), idesc,
                                       (kb != un.k0 || kk != 0) ? 1u : 0u);
                    else
                        umma_bf16(d, sdesc_sw128(a_addr + kk * 32), sdesc_sw128(b_addr + kk * 32), idesc,
                                  (kb != un.k0 || kk != 0) ? 1u : 0u);
                }
                if (PAIR)
                    umma_commit_pair(&empty[s]);
                else
                    umma_commit(&empty[s]);
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1;
                }
            }
            if (PAIR)
                umma_commit_pair(&tfull[b]);
            else
                umma_commit(&tfull[b]);
            b ^= 1;
            if (b == 0) tph ^= 1;
        }
    } else if (warp >= 2) {
        // ---------------- epilogue: thread = one row of the 128-row tile
        const int sp = warp & 3;  // TMEM lane quarter this warp may access
        const int r_in = sp * 32 + lane;
        int b = 0;
        uint32_t tph = 0;
        for (int u = grp; u < sc.units; u += n_grp) {
            const Unit un = unit_of(u, sc, kblocks);
            const int mt = un.t % m_tiles, nt = un.t / m_tiles;
            // lane 0 waits and broadcasts; the warp stays converged for the .sync.aligned
            // tcgen05.ld below
            bool ok = true;
            if (lane == 0) ok = mbar_wait_t<PAIR>(&tfull[b], tph, &abort_flag);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            __syncwarp();
            if (!ok) {
                abort_flag = 1;
                if (lane == 0) set_error(err, BLEND_ETIMEOUT);
                break;
            }
            tc_fence_after();
            const int row = mt * TC::TM + rank * BM + r_in;
            const uint32_t tl = tbase + ((uint32_t)(sp * 32) << 16) + (uint32_t)(b * BN);
            const float rs = row < M ? row_scale(ne, row) : 1.f;
            // residual add of a warp whose 32 rows are all live: through shared memory and
            // tensor stores (warp-uniform)
            const int row0 = mt * TC::TM + rank * BM + sp * 32;
            const bool tma_rows = EPI == EPI_ADD_F32 && tma_out != 0 && row0 + 32 <= M;
            uint8_t* cb = smem + STAGES * STAGE_BYTES + sp * OUT_WARP_BYTES;
            if (EPI == EPI_QKV_ROPE) {
                // the tile holds BN/128 whole heads of this row: q and k heads are rotated at
                // the row's position (pairs i, i+64), then q goes to its per-kv-head slab and
                // k, v to the cache row of the row's token
                const bool live = row < M;
                const int pos = live ? qe.row_pos[row] : 0;
                const long long tok = live ? qe.row_tok[row] : 0;
#pragma unroll 1
                for (int hh = 0; hh < BN / 128; ++hh) {
                    const int head = nt * (BN / 128) + hh;
                    bf16* dst;
                    bool rotate = true;
                    if (head < qe.hq) {
                        dst = qe.q + (((long long)(head / qe.group) * qe.m_cap + row) * qe.group + head % qe.group) * 128;
                    } else if (head < qe.hq + qe.hkv) {
                        dst = qe.k_cache + (tok * qe.hkv + (head - qe.hq)) * 128;
                    } else {
                        dst = qe.v_cache + (tok * qe.hkv + (head - qe.hq - qe.hkv)) * 128;
                        rotate = false;
                    }
#pragma unroll 1
                    for (int c = 0; c < 64; c += 32) {
                        uint32_t x1[32], x2[32];
                        TMEM_LD32(tl + hh * 128 + c, x1);
                        TMEM_LD32(tl + hh * 128 + 64 + c, x2);
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                        if (live) {
                            uint32_t w1[16], w2[16];
                            if (rotate) {
                                const float4* cs = reinterpret_cast<const float4*>(qe.rope + (long long)pos * 64 + c);
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    const float4 t = cs[i];  // (cos, sin) of pairs 2i and 2i+1
                                    const float a0 = __uint_as_float(x1[2 * i]) * rs, b0 = __uint_as_float(x2[2 * i]) * rs;
                                    const float a1 = __uint_as_float(x1[2 * i + 1]) * rs;
                                    const float b1 = __uint_as_float(x2[2 * i + 1]) * rs;
                                    w1[i] = pack_bf16x2(a0 * t.x - b0 * t.y, a1 * t.z - b1 * t.w);
                                    w2[i] = pack_bf16x2(b0 * t.x + a0 * t.y, b1 * t.z + a1 * t.w);
                                }
                            } else {
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    w1[i] = pack_bf16x2(__uint_as_float(x1[2 * i]) * rs, __uint_as_float(x1[2 * i + 1]) * rs);
                                    w2[i] = pack_bf16x2(__uint_as_float(x2[2 * i]) * rs, __uint_as_float(x2[2 * i + 1]) * rs);
                                }
                            }
                            uint4* d1 = reinterpret_cast<uint4*>(dst + c);
                            uint4* d2 = reinterpret_cast<uint4*>(dst + 64 + c);
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                d1[v] = make_uint4(w1[4 * v], w1[4 * v + 1], w1[4 * v + 2], w1[4 * v + 3]);
                                d2[v] = make_uint4(w2[4 * v], w2[4 * v + 1], w2[4 * v + 2], w2[4 * v + 3]);
                            }
                        }
                    }
                }
            } else if (un.half >= 0) {
                // a K part of a split tile: its raw partial goes to the workspace rows of
                // (split tile, part); k_split_combine finishes the tile
                // (a warp whose 32 rows all lie past the device row count has nothing to keep:
                // the combine reads live rows only)
                const int ws_row0 = (un.sidx * sc.parts + un.half) * TC::TM + rank * BM + sp * 32;
                if (row0 < M) {
#pragma unroll 1
                    for (int c = 0; c < BN; c += 32) {
                        uint32_t r[32];
                        TMEM_LD32(tl + c, r);
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                        part_chunk_tma(r, ws_row0, c, cb, &mapW);
                    }
                }
            } else {
                // a whole tile; the folded-norm sums of squares are kept per BN/2 columns
                const int cbase = nt * BN;
                if (EPI == EPI_ADD_F32 && tma_rows) {
                    // residual add of 32 live rows: the next chunk's residual loads are in
                    // flight while this chunk is added and stored
                    const float* xrow = (const float*)Cv + (long long)row * ldc + cbase;
                    float4 xn[8];
                    if (cbase < N) {
#pragma unroll
                        for (int v = 0; v < 8; ++v) xn[v] = reinterpret_cast<const float4*>(xrow)[v];
                    }
                    float ssq = 0.f;
#pragma unroll 1
                    for (int c = 0; c < BN; c += 32) {
                        const int col = cbase + c;
                        uint32_t r[32];
                        TMEM_LD32(tl + c, r);
                        float4 xr[8];
#pragma unroll
                        for (int v = 0; v < 8; ++v) xr[v] = xn[v];
                        if (c + 32 < BN && col + 32 < N) {
#pragma unroll
                            for (int v = 0; v < 8; ++v) xn[v] = reinterpret_cast<const float4*>(xrow + c + 32)[v];
                        }
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                        if (col < N) add_chunk_tma(r, xr, row0, col, rs, ne, cb, &mapC, &mapX, ssq);
                        if (c + 32 == HALF || c + 32 == BN) {
                            const int col0 = cbase + (c + 32 == HALF ? 0 : HALF);
                            if (ne.x_out != nullptr && col0 < N)
                                ne.ssq_out[(long long)row * ne.ssq_stride + col0 / HALF] = ssq;
                            ssq = 0.f;
                        }
                    }
                } else {
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    float ssq = 0.f;
#pragma unroll 1
                    for (int c = hh * HALF; c < (hh + 1) * HALF; c += 32) {
                        uint32_t r[32];
                        TMEM_LD32(tl + c, r);
                        const int col = cbase + c;
                        if (EPI == EPI_ADD_F32 && tma_rows && col < N) {
                            float4 xr[8];
                            const float4* xp =
                                reinterpret_cast<const float4*>((const float*)Cv + (long long)row * ldc + col);
#pragma unroll
                            for (int v = 0; v < 8; ++v) xr[v] = xp[v];
                            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                            add_chunk_tma(r, xr, row0, col, rs, ne, cb, &mapC, &mapX, ssq);
                        } else {
                            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                            if (row < M && col < N) epi_chunk<EPI>(r, row, col, Cv, ldc, rs, ne, ssq);
                        }
                    }
                    const int col0 = cbase + hh * HALF;
                    if (EPI == EPI_ADD_F32 && ne.x_out != nullptr && row < M && col0 < N)
                        ne.ssq_out[(long long)row * ne.ssq_stride + col0 / HALF] = ssq;
                }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR)
                    mbar_arrive_cluster(leader_addr(&tempty[b]));  // the leader reuses the columns
                else
                    mbar_arrive(&tempty[b]);
            }
            b ^= 1;
            if (b == 0) tph ^= 1;
        }
        // the staging chunk belongs to this CTA: its last stores must be done before exit
        if (EPI != EPI_QKV_ROPE && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) {
        // drain loads still in flight so no copy lands in shared memory after exit
        for (int s = 0; s < STAGES; ++s)
            if (pending[s] >= 0) {
                for (long long i = 0; i < SPIN_LIMIT && !mbar_try(&full[s], (uint32_t)pending[s]); ++i) {
                }
            }
    }
    tc_fence_before();
    __syncthreads();
    // neither CTA of a pair leaves while the other may still signal its barriers
    if (PAIR) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(TMEM_COLS)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(TMEM_COLS)
                         : "memory");
    }
}

// Finishes the split tiles of a k_gemm_tc launch (BN = 256): the K-part partials of
// every row of a split tile are added in a fixed order (part 0 + part 1 + ...), scaled by
// the row's folded-norm factor, and the tile's epilogue runs on the sum: fp32 store, residual
// add (with bf16(x * g) and the two per-128-column sums of squares of a norm producer) or
// SwiGLU.  One warp per row, eight consecutive columns per lane.  The split set is the
// kernel's own (same schedule from the device row count).
template <int EPI, int TM>
__device__ __forceinline__ void combine_tile(const float* __restrict__ ws, int N, int M, int m_tiles, const Sched& sc,
                                             int sidx, void* __restrict__ Cv, int ldc, const NormEpi& ne);

template <int EPI, int TM>
__global__ void __launch_bounds__(128)
    k_split_combine(const float* __restrict__ ws, int K, int N, const int32_t* __restrict__ M_dev, int n_grp,
                    void* __restrict__ Cv, int ldc, const __grid_constant__ NormEpi ne) {
    const int M = *M_dev;
    const int m_tiles = (M + TM - 1) / TM, n_tiles = (N + 255) / 256;
    const Sched sc = make_sched(m_tiles * n_tiles, n_grp, true, K / BK, (int)(GEMM_SPLIT_WS_FLOATS / 256 / TM));
    // split tiles blockIdx.x, blockIdx.x + gridDim.x, ...
    for (int sidx = blockIdx.x; sidx < sc.split; sidx += gridDim.x)
        combine_tile<EPI, TM>(ws, N, M, m_tiles, sc, sidx, Cv, ldc, ne);
}

template <int EPI, int TM>
__device__ __forceinline__ void combine_tile(const float* __restrict__ ws, int N, int M, int m_tiles, const Sched& sc,
                                             int sidx, void* __restrict__ Cv, int ldc, const NormEpi& ne) {
    const int t = sc.full + sidx, mt = t % m_tiles, nt = t / m_tiles;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int r_t = blockIdx.y * 4 + warp;  // row within the tile
    const int row = mt * TM + r_t;
    if (r_t >= TM || row >= M) return;
    const float rs = row_scale(ne, row);
    const int c0 = lane * 8, col = nt * 256 + c0;
    const bool live = col < N;  // N % 32 == 0: a lane's eight columns are all in or all out
    float v[8];
    if (live) {
        const float4* p0 = reinterpret_cast<const float4*>(ws + ((long long)(sidx * sc.parts) * TM + r_t) * 256 + c0);
        float4 a0 = __ldcg(p0), a1 = __ldcg(p0 + 1);
        for (int q = 1; q < sc.parts; ++q) {
            const float4* pq = p0 + (long long)q * TM * 64;  // next part: TM rows of 256 floats on
            const float4 b0 = __ldcg(pq), b1 = __ldcg(pq + 1);
            a0.x += b0.x;
            a0.y += b0.y;
            a0.z += b0.z;
            a0.w += b0.w;
            a1.x += b1.x;
            a1.y += b1.y;
            a1.z += b1.z;
            a1.w += b1.w;
        }
        v[0] = a0.x * rs;
        v[1] = a0.y * rs;
        v[2] = a0.z * rs;
        v[3] = a0.w * rs;
        v[4] = a1.x * rs;
        v[5] = a1.y * rs;
        v[6] = a1.z * rs;
        v[7] = a1.w * rs;
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.f;
    }
    if (EPI == EPI_STORE_F32) {
        if (live) {
            float4* p = reinterpret_cast<float4*>((float*)Cv + (long long)row * ldc + col);
            p[0] = make_float4(v[0], v[1], v[2], v[3]);
            p[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
    } else if (EPI == EPI_ADD_F32) {
        float ssq = 0.f;
        if (live) {
            float4* p = reinterpret_cast<float4*>((float*)Cv + (long long)row * ldc + col);
            const float4 x0 = p[0], x1 = p[1];
            v[0] += x0.x;
            v[1] += x0.y;
            v[2] += x0.z;
            v[3] += x0.w;
            v[4] += x1.x;
            v[5] += x1.y;
            v[6] += x1.z;
            v[7] += x1.w;
            p[0] = make_float4(v[0], v[1], v[2], v[3]);
            p[1] = make_float4(v[4], v[5], v[6], v[7]);
            if (ne.x_out != nullptr) {
                const uint4 gv = *reinterpret_cast<const uint4*>(ne.g + col);
                const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
                uint32_t xw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    ssq = fmaf(v[2 * e], v[2 * e], ssq);
                    ssq = fmaf(v[2 * e + 1], v[2 * e + 1], ssq);
                    xw[e] = pack_bf16x2(v[2 * e] * __uint_as_float(gw[e] << 16),
                                        v[2 * e + 1] * __uint_as_float(gw[e] & 0xffff0000u));
                }
                *reinterpret_cast<uint4*>(ne.x_out + (long long)row * ne.ldx + col) = make_uint4(xw[0], xw[1], xw[2], xw[3]);
            }
        }
        if (ne.x_out != nullptr) {
            // sums of squares of the two 128-column halves: 16 lanes each, fixed tree
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
            const int seg = lane >> 4;
            if ((lane & 15) == 0 && nt * 256 + seg * 128 < N)
                ne.ssq_out[(long long)row * ne.ssq_stride + 2 * nt + seg] = ssq;
        }
    } else if (EPI == EPI_SWIGLU) {
        // a 32-column group holds 16 gate then 16 up columns of the same hidden units:
        // lanes 4i, 4i+1 hold the gates, 4i+2, 4i+3 the matching ups
        float u[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) u[e] = __shfl_down_sync(0xffffffffu, v[e], 2);
        if (live && (lane & 3) < 2) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float g0 = v[2 * e], g1 = v[2 * e + 1];
                w[e] = pack_bf16x2(g0 / (1.f + expf(-g0)) * u[2 * e], g1 / (1.f + expf(-g1)) * u[2 * e + 1]);
            }
            const int ocol = (nt * 256 + (lane >> 2) * 32) / 2 + (lane & 3) * 8;
            *reinterpret_cast<uint4*>((bf16*)Cv + (long long)row * ldc + ocol) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
int g_tc_state = -1;  // -1 unknown, 0 unavailable, 1 available
int g_num_sms = 0;

bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
               uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Output map of the residual-add epilogue: [outer][inner] elements of `bytes` each with a
// row stride of ld elements, 32 x 32 boxes, the given swizzle.
bool encode_out(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int bytes, uint64_t inner,
                uint64_t outer, uint64_t ld, CUtensorMapSwizzle sw) {
    if (((uintptr_t)base & 15) != 0 || (ld * bytes) % 16 != 0) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * bytes};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          sw, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

int tc_available() {
    if (g_tc_state >= 0) return g_tc_state;
    g_tc_state = 0;
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (!(prop.major == 10 && prop.minor == 3)) return 0;  // built for sm_103a only
    g_num_sms = prop.multiProcessorCount;
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return 0;
    }
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
#define SET_SMEM(E, N, P) \
    cudaFuncSetAttribute(k_gemm_tc<E, N, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<E, N, P>())
    SET_SMEM(EPI_STORE_F32, 256, false);
    SET_SMEM(EPI_ADD_F32, 256, false);
    SET_SMEM(EPI_SWIGLU, 256, false);
    SET_SMEM(EPI_QKV_ROPE, 256, false);
    SET_SMEM(EPI_STORE_F32, 128, false);
    SET_SMEM(EPI_ADD_F32, 128, false);
    SET_SMEM(EPI_SWIGLU, 128, false);
    SET_SMEM(EPI_QKV_ROPE, 128, false);
    SET_SMEM(EPI_STORE_F32, 256, true);
    SET_SMEM(EPI_ADD_F32, 256, true);
    SET_SMEM(EPI_SWIGLU, 256, true);
    SET_SMEM(EPI_QKV_ROPE, 256, true);
#undef SET_SMEM
    g_tc_state = 1;
    return 1;
}

bool tc_gemm_supported(int K, int N, int epi, int ldc, int M_cap) {
    if (epi == EPI_QKV_ROPE && N % 256 != 0) return false;
    return K >= BK && K % BK == 0 && N >= 128 && N % 32 == 0 && ldc % 8 == 0 && M_cap >= BM;
}

// N-tile width: 256, or 128 when N is a multiple of 128 but not of 256 or smaller than
// 256 (the weight tensor must be at least one box high).  Otherwise the last 256-wide
// tile is partial: the TMA fills the rows past N with zeros and the epilogue skips
// those columns.  (128-wide tiles everywhere fill the waves better for N = 5120 at ~3.3K
// rows, but measured 30-40 % slower per FLOP; only a half-full last wave runs as halves.)
int pick_bn(int N) { return (N < 256 || (N % 256 != 0 && N % 128 == 0)) ? 128 : 256; }

int gemm_tc_norm_parts(int N) {
    const int half = pick_bn(N) / 2;
    return (N + half - 1) / half;
}

template <int BN, bool PAIR>
void launch_bn(const CUtensorMap& ma, const CUtensorMap& mb, int K, int N, const int32_t* M_dev, int M_max, int epi,
               void* C, int ldc, int32_t* err, cudaStream_t s, const QkvEpi& qe, const float* split_ws,
               const CUtensorMap& mw, const NormEpi& ne, const CUtensorMap& mc, const CUtensorMap& mx, int tma_out) {
    // one work unit per CTA, or per cluster of two CTAs: as many as can be resident at once
    int slots = g_num_sms;
    if (PAIR) {
        static int max_clusters[4] = {0, 0, 0, 0};
        int& mc = max_clusters[epi & 3];
        if (mc == 0) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(g_num_sms);
            q.blockDim = dim3(THREADS);
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = 2;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            int n = 0;
            cudaError_t e = cudaSuccess;
            switch (epi) {
                case EPI_STORE_F32:
                    q.dynamicSmemBytes = smem_bytes<EPI_STORE_F32, BN, PAIR>();
                    e = cudaOccupancyMaxActiveClusters(&n, k_gemm_tc<EPI_STORE_F32, BN, PAIR>, &q);
                    break;
                case EPI_ADD_F32:
                    q.dynamicSmemBytes = smem_bytes<EPI_ADD_F32, BN, PAIR>();
                    e = cudaOccupancyMaxActiveClusters(&n, k_gemm_tc<EPI_ADD_F32, BN, PAIR>, &q);
                    break;
                case EPI_SWIGLU:
                    q.dynamicSmemBytes = smem_bytes<EPI_SWIGLU, BN, PAIR>();
                    e = cudaOccupancyMaxActiveClusters(&n, k_gemm_tc<EPI_SWIGLU, BN, PAIR>, &q);
                    break;
                default:
                    q.dynamicSmemBytes = smem_bytes<EPI_QKV_ROPE, BN, PAIR>();
                    e = cudaOccupancyMaxActiveClusters(&n, k_gemm_tc<EPI_QKV_ROPE, BN, PAIR>, &q);
            }
            if (e != cudaSuccess || n <= 0) {
                cudaGetLastError();
                n = g_num_sms / 2;
            }
            mc = n < g_num_sms / 2 ? n : g_num_sms / 2;
        }
        slots = mc;
    }
    const int tiles = ((M_max + TileCfg<BN, PAIR>::TM - 1) / TileCfg<BN, PAIR>::TM) * ((N + BN - 1) / BN);
    int groups = tiles < slots ? tiles : slots;
    const bool split = split_ws != nullptr && epi != EPI_QKV_ROPE && BN == 256 && K / BK >= 2;
    // with splitting allowed the device may run each of few tiles as up to four K parts
    // (make_sched): give it up to four units per tile of the host's bound
    if (split) groups = 4 * tiles < slots ? 4 * tiles : slots;
    const int cs = split ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(PAIR ? 2 * groups : groups);
    cfg.blockDim = dim3(THREADS);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = PAIR ? 2 : 1;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
#define LAUNCH(E)                                                                                              \
    do {                                                                                                       \
        cfg.dynamicSmemBytes = smem_bytes<E, BN, PAIR>();                                                      \
        cudaLaunchKernelEx(&cfg, k_gemm_tc<E, BN, PAIR>, ma, mb, K, N, M_dev, C, ldc, err, qe, cs, ne, mc, mx,   \
                           tma_out, mw);                                                                       \
    } while (0)
    if (epi == EPI_STORE_F32)
        LAUNCH(EPI_STORE_F32);
    else if (epi == EPI_ADD_F32)
        LAUNCH(EPI_ADD_F32);
    else if (epi == EPI_SWIGLU)
        LAUNCH(EPI_SWIGLU);
    else
        LAUNCH(EPI_QKV_ROPE);
#undef LAUNCH
    if (split) {
        // the split tiles (if the device row count gives any) are finished here
        constexpr int TM = TileCfg<BN, PAIR>::TM;
        // the tail rule splits at most groups / 2 tiles; with fewer tiles than slots every
        // tile may be split: one column of CTAs per tile, so none takes two
        const int n_split = tiles < slots ? tiles : (groups / 2 > 0 ? groups / 2 : 1);
        const dim3 grid(n_split, TM / 4);
        if (epi == EPI_STORE_F32)
            k_split_combine<EPI_STORE_F32, TM><<<grid, 128, 0, s>>>(split_ws, K, N, M_dev, groups, C, ldc, ne);
        else if (epi == EPI_ADD_F32)
            k_split_combine<EPI_ADD_F32, TM><<<grid, 128, 0, s>>>(split_ws, K, N, M_dev, groups, C, ldc, ne);
        else
            k_split_combine<EPI_SWIGLU, TM><<<grid, 128, 0, s>>>(split_ws, K, N, M_dev, groups, C, ldc, ne);
        note_launch(1);
    }
}

// Tile-times of T tiles on `slots` units under make_sched's rules (workspace limit aside):
// whole waves, a last wave at most half full as K halves, or fewer tiles than slots as up
// to four K parts.
double est_tile_times(int T, int slots, bool can_split, int kblocks) {
    if (T <= 0 || slots <= 0) return 0.0;
    if (T >= slots) {
        const int full = T / slots, rem = T % slots;
        if (rem == 0) return full;
        return full + ((can_split && kblocks >= 2 && 2 * rem <= slots) ? 0.5 : 1.0);
    }
    double best = 1.0;
    if (can_split)
        for (int S = 2; S <= 4 && S <= kblocks; ++S) {
            const double t = (double)((S * T + slots - 1) / slots) / S;
            if (t < best) best = t;
        }
    return best;
}

int launch_gemm_tc(const void* A, int K, int M_cap, const void* B, int N, const int32_t* M_dev, int M_max,
                   int epi, void* C, int ldc, int32_t* err, cudaStream_t s, const QkvEpi* qkv, float* split_ws,
                   const NormEpi* norm) {
    if (M_max <= 0) return BLEND_OK;
    const int bn = pick_bn(N);
    if (epi == EPI_QKV_ROPE && (qkv == nullptr || bn != 256)) return BLEND_EUNSUPPORTED;
    QkvEpi qe{};
    if (qkv) qe = *qkv;
    NormEpi ne{};
    if (norm) ne = *norm;
    if (ne.x_out && (epi != EPI_ADD_F32 || ne.ssq_out == nullptr || ne.g == nullptr || ne.ldx % 8 != 0 ||
                     ne.ssq_stride != gemm_tc_norm_parts(N)))
        return BLEND_EUNSUPPORTED;
    // 256-wide tiles over more than one 128-row block run on CTA pairs (256x256 tiles; each
    // CTA of a pair stages half of a tile's weight rows, a third less operand traffic per
    // SM), unless single-CTA 128-row tiles take clearly fewer tile-times: few rows, where
    // 256-row tiles pad more and the waves fill worse (both sides with the device's split
    // rules).  A single tile-time measured ~15 % longer than a pair's at ~500 rows (8B
    // gate/up: 4.0 single waves took longer than 4.5 pair waves), hence the margin.
    bool pair = bn == 256 && M_max > BM && g_num_sms >= 2;
    if (pair) {
        const bool can_split = split_ws != nullptr && epi != EPI_QKV_ROPE;
        const int nt = (N + bn - 1) / bn, kb = K / BK;
        const double t_pair = est_tile_times((M_max + 2 * BM - 1) / (2 * BM) * nt, g_num_sms / 2, can_split, kb);
        const double t_one = est_tile_times((M_max + BM - 1) / BM * nt, g_num_sms, can_split, kb);
        if (t_one * 1.15 < t_pair) pair = false;
    }
    const uint32_t brows = pair ? (uint32_t)bn / 2 : (uint32_t)bn;
    CUtensorMap ma, mb;
    if (!encode_2d(&ma, A, (uint64_t)K, (uint64_t)M_cap, BK, BM) ||
        !encode_2d(&mb, B, (uint64_t)K, (uint64_t)N, BK, brows))
        return BLEND_EUNSUPPORTED;  // the operands cannot be described to the TMA unit
    // split workspace: rows (split tile, K half, tile row) of 256 fp32
    CUtensorMap mw{};
    if (split_ws != nullptr &&
        (g_num_sms > GEMM_SPLIT_SMS || !encode_out(&mw, split_ws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 256,
                                                    (uint64_t)GEMM_SPLIT_WS_FLOATS / 256, 256, CU_TENSOR_MAP_SWIZZLE_128B)))
        split_ws = nullptr;
    // residual add: the sum (and bf16(x * g)) of warps with 32 live rows leave as tensor
    // stores; the maps span the M_max rows the launch may write
    CUtensorMap mc{}, mx{};
    int tma_out = 0;
    if (epi == EPI_ADD_F32) {
        tma_out = encode_out(&mc, C, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)N, (uint64_t)M_max, (uint64_t)ldc,
                             CU_TENSOR_MAP_SWIZZLE_128B) &&
                  (ne.x_out == nullptr || encode_out(&mx, ne.x_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)N,
                                                     (uint64_t)M_max, (uint64_t)ne.ldx, CU_TENSOR_MAP_SWIZZLE_64B));
    }
    if (pair)
        launch_bn<256, true>(ma, mb, K, N, M_dev, M_max, epi, C, ldc, err, s, qe, split_ws, mw, ne, mc, mx, tma_out);
    else if (bn == 256)
        launch_bn<256, false>(ma, mb, K, N, M_dev, M_max, epi, C, ldc, err, s, qe, split_ws, mw, ne, mc, mx, tma_out);
    else
        launch_bn<128, false>(ma, mb, K, N, M_dev, M_max, epi, C, ldc, err, s, qe, split_ws, mw, ne, mc, mx, tma_out);
    note_launch(1);
    return BLEND_OK;
}

}  // namespace blend
