// Token selection on the device: top-k by score, then CacheClip sliding-window
// grouping under a row budget (CacheClip blog, "6.3 Sliding-window grouping" and its
// Figure 6; SpecCache 2.2 TopK with K = ceil(rho N)).
//
// The grouping rule is evaluated for every k at once through ranks:
//   rank(t)    = place of t when scores are sorted descending, ties by position
//                (-0 == +0, NaN after every number, disallowed positions never rank).
//   At a given k the candidates are {t : rank(t) < k}.  The window starting at t
//   (t <= n - w) passes iff t is a candidate and it holds >= tau candidates, i.e. iff
//   k > qual(t) = max(rank(t), tau-th smallest rank inside [t, t+w)).
//   Position p is in the set iff some window covering it passes:
//   cover(p) = min over t in (p-w, p] of qual(t);  p in R(k)  <=>  cover(p) < k.
// CANDIDATE mode uses k = min(budget, #allowed).  FINAL mode needs the largest
// k <= that bound with |R(k)| <= budget: |R(k)| = #{p : cover(p) < k} is monotone in
// k, so the answer is either the bound itself or the (budget+1)-th smallest cover
// value.  All arithmetic is integer, so the result is exact.
#include <climits>
#include <cstring>

#include "common.cuh"

namespace blend {

constexpr int SEL_THREADS = 1024;
constexpr int SEL_MAX_PER_THREAD = 32;  // n <= 32768 per job
constexpr int RANK_TILE = 2048;

__device__ __forceinline__ unsigned long long sel_key(float s, int t) {
    uint32_t u = __float_as_uint(s);
    uint32_t k;
    if ((u & 0x7fffffffu) > 0x7f800000u) {
        k = 0xffffffffu;  // NaN ranks after every number
    } else {
        if (u == 0x80000000u) u = 0u;  // -0 counts as +0
        uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // ascending with value
        k = ~ord;                                                   // descending with value
    }
    return ((unsigned long long)k << 32) | (uint32_t)t;
}

// rank[t] = #{u allowed : key(u) < key(t)} for allowed t, INT_MAX otherwise, in two
// steps over tiles of RANK_TILE positions:
//   k_rank_tiles  one CTA per tile bitonic-sorts the tile's 64-bit keys (disallowed and
//                 padding positions get ~0, which sorts after every real key) in shared
//                 memory and stores the sorted tile;
//   k_rank_merge  one CTA per tile takes its sorted keys and, for every sorted tile in
//                 turn, counts the keys below each of them by binary search in shared
//                 memory; the sum over tiles is the rank (keys are distinct: the position
//                 is part of the key).
// O(n log n) work instead of the n^2 comparisons of a direct count.
constexpr int RANK_THREADS = 1024;  // RANK_TILE = 2 keys per thread

__global__ void __launch_bounds__(RANK_THREADS)
    k_rank_tiles(const __grid_constant__ SelectBatch sb, unsigned long long* __restrict__ sorted,
                 int sorted_stride, int32_t* __restrict__ rank) {
    __shared__ unsigned long long key[RANK_TILE];
    const SelectJob& jb = sb.j[blockIdx.y];
    const int n = jb.n;
    const int base = blockIdx.x * RANK_TILE;
    if (base >= n) return;
    for (int i = threadIdx.x; i < RANK_TILE; i += RANK_THREADS) {
        const int t = base + i;
        unsigned long long k = ~0ull;
        if (t < n) {
            if (jb.allowed == nullptr || jb.allowed[t] != 0) k = sel_key(jb.scores[t], t);
            else rank[jb.rank_off + t] = INT_MAX;
        }
        key[i] = k;
    }
    __syncthreads();
    // bitonic network, ascending: one compare-exchange per thread and stage
    const int i = threadIdx.x;
    for (int k = 2; k <= RANK_TILE; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            const int l = 2 * i - (i & (j - 1));
            const int r = l + j;
            const unsigned long long a = key[l], b = key[r];
            if ((a > b) == ((l & k) == 0)) {
                key[l] = b;
                key[r] = a;
            }
            __syncthreads();
        }
    }
    unsigned long long* dst = sorted + (long long)blockIdx.y * sorted_stride + base;
    for (int e = threadIdx.x; e < RANK_TILE; e += RANK_THREADS) dst[e] = key[e];
}

__global__ void __launch_bounds__(RANK_THREADS)
    k_rank_merge(const __grid_constant__ SelectBatch sb, const unsigned long long* __restrict__ sorted,
                 int sorted_stride, int32_t* __restrict__ rank) {
    __shared__ unsigned long long tile[RANK_TILE];
    const SelectJob& jb = sb.j[blockIdx.y];
    const int n = jb.n;
    const int a0 = blockIdx.x * RANK_TILE;
    if (a0 >= n) return;
    const unsigned long long* srt = sorted + (long long)blockIdx.y * sorted_stride;
    const unsigned long long q0 = srt[a0 + threadIdx.x], q1 = srt[a0 + RANK_THREADS + threadIdx.x];
    int c0 = 0, c1 = 0;
    const int n_tiles = (n + RANK_TILE - 1) / RANK_TILE;
    for (int bt = 0; bt < n_tiles; ++bt) {
        __syncthreads();
        for (int e = threadIdx.x; e < RANK_TILE; e += RANK_THREADS) tile[e] = srt[bt * RANK_TILE + e];
        __syncthreads();
        // number of keys below q in the sorted tile (lower bound)
        int l0 = 0, l1 = 0;
#pragma unroll
        for (int step = RANK_TILE / 2; step > 0; step >>= 1) {
            if (tile[l0 + step - 1] < q0) l0 += step;
            if (tile[l1 + step - 1] < q1) l1 += step;
        }
        c0 += l0 + (tile[l0] < q0 ? 1 : 0);
        c1 += l1 + (tile[l1] < q1 ? 1 : 0);
    }
    if (q0 != ~0ull) rank[jb.rank_off + (int)(uint32_t)q0] = c0;
    if (q1 != ~0ull) rank[jb.rank_off + (int)(uint32_t)q1] = c1;
}

// One CTA per job.  Positions are walked in rounds of SEL_THREADS consecutive positions
// (round e, thread i: p = e * SEL_THREADS + i), so the accesses of a warp to shared and
// global memory are consecutive.
__global__ void __launch_bounds__(SEL_THREADS)
    k_select_finish(const __grid_constant__ SelectBatch sb, const int32_t* __restrict__ rank_all) {
    extern __shared__ int32_t cov[];  // n ints: qual, then cover
    __shared__ int warp_tot[SEL_THREADS / 32];
    __shared__ int bcast;
    const SelectJob& jb = sb.j[blockIdx.x];
    const int n = jb.n;
    const int w = sb.window, tau = sb.tau;
    const int* rank = rank_all + jb.rank_off;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    int loc = 0;
    for (int t = tid; t < n; t += SEL_THREADS) loc += rank[t] != INT_MAX;
    const int n_ok = block_sum_i32(loc, warp_tot, &bcast);
    const int kmax = min(jb.budget, n_ok);

    // qual(t); ranks >= kmax can never be candidates and count as infinite.
    for (int t = tid; t < n; t += SEL_THREADS) {
        int q = INT_MAX;
        const int rt = rank[t];
        if (t <= n - w && rt < kmax) {
            if (tau <= 1) {
                q = rt;
            } else {
                // tau-th smallest of the window's ranks (ranks are distinct):
                // repeated extraction of the next larger rank
                int last = -1, found = INT_MAX;
                for (int seen = 0; seen < tau; ++seen) {
                    int m = INT_MAX;
                    for (int j = t; j < t + w; ++j) {
                        const int r = rank[j];
                        if (r < kmax && r > last && r < m) m = r;
                    }
                    if (m == INT_MAX) break;
                    last = m;
                    if (seen == tau - 1) found = m;
                }
                q = found == INT_MAX ? INT_MAX : max(rt, found);
            }
        }
        cov[t] = q;
    }
    __syncthreads();
    // cover(p) = min of qual over the windows (p-w, p] covering p; kept in registers until
    // every thread has read the qual values it needs
    int cl[SEL_MAX_PER_THREAD];
#pragma unroll
    for (int e = 0; e < SEL_MAX_PER_THREAD; ++e) {
        const int p = e * SEL_THREADS + tid;
        int c = INT_MAX;
        if (p < n && (jb.allowed == nullptr || jb.allowed[p] != 0)) {
            const int lo = max(0, p - w + 1);
            for (int t = lo; t <= p; ++t) c = min(c, cov[t]);
        }
        cl[e] = c;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < SEL_MAX_PER_THREAD; ++e) {
        const int p = e * SEL_THREADS + tid;
        if (p < n) cov[p] = cl[e];
    }
    __syncthreads();

    int k = kmax;
    if (sb.budget_mode == BLEND_BUDGET_FINAL && kmax > 0) {
        loc = 0;
#pragma unroll
        for (int e = 0; e < SEL_MAX_PER_THREAD; ++e) loc += cl[e] < kmax;
        const int f = block_sum_i32(loc, warp_tot, &bcast);
        if (f > jb.budget) {
            // smallest v with #{cover <= v} >= budget + 1
            int lo = 0, hi = kmax - 1;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                loc = 0;
#pragma unroll
                for (int e = 0; e < SEL_MAX_PER_THREAD; ++e) loc += cl[e] <= mid;
                const int c = block_sum_i32(loc, warp_tot, &bcast);
                if (c >= jb.budget + 1) hi = mid;
                else lo = mid + 1;
            }
            k = lo;
        }
    }

    // ordered compaction of {p : cover(p) < k}
    const int written = compact_in_order(n, jb.base, jb.out, [&](int p) { return cov[p] < k; }, warp_tot, &bcast);
    if (tid == 0) *jb.out_n = written;
}

void launch_rank(const SelectBatch& sb, int32_t* rank_scratch, unsigned long long* sort_scratch, int max_n,
                 cudaStream_t s) {
    if (sb.n_job <= 0) return;
    if (max_n <= 0) max_n = 1;
    const int tiles = (max_n + RANK_TILE - 1) / RANK_TILE;
    const int stride = tiles * RANK_TILE;
    dim3 g(tiles, sb.n_job);
    k_rank_tiles<<<g, RANK_THREADS, 0, s>>>(sb, sort_scratch, stride, rank_scratch);
    k_rank_merge<<<g, RANK_THREADS, 0, s>>>(sb, sort_scratch, stride, rank_scratch);
    note_launch(2);
}

void launch_select(const SelectBatch& sb, int32_t* rank_scratch, unsigned long long* sort_scratch, int max_n,
                   cudaStream_t s) {
    if (sb.n_job <= 0) return;
    if (max_n <= 0) max_n = 1;
    launch_rank(sb, rank_scratch, sort_scratch, max_n, s);
    if (sb.rule == BLEND_GROUP_SPAN) {
        launch_span_finish(sb, rank_scratch, max_n, s);
        return;
    }
    const size_t smem = (size_t)max_n * sizeof(int32_t);
    cudaFuncSetAttribute(k_select_finish, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         SEL_THREADS * SEL_MAX_PER_THREAD * (int)sizeof(int32_t));
    k_select_finish<<<sb.n_job, SEL_THREADS, smem, s>>>(sb, rank_scratch);
    note_launch(1);
}

// ---------------------------------------------------------------- allocation-free variant
// Scratch of topk_select_dilate_noalloc: fixed arrays in device memory, so the call needs
// neither a handle nor any allocation.  Every GPU that loads the library holds these
// 384 KB (32768 ranks and 32768 sorted 64-bit keys) until the process exits.
constexpr int NOALLOC_MAX_N = 32768;
static __device__ __align__(256) int32_t g_noalloc_rank[NOALLOC_MAX_N];
static __device__ __align__(256) unsigned long long g_noalloc_sorted[NOALLOC_MAX_N];

namespace {
struct NoallocScratch {
    int32_t* rank = nullptr;
    unsigned long long* sorted = nullptr;
};

// Device addresses of the scratch arrays on the current device, looked up on every call
// with that device current (a host-side query that allocates nothing), so no address
// outlives the module instance it came from (after cudaDeviceReset the module may load
// at another address).  The host-side names of the arrays are only stand-ins and must
// not reach a kernel.
int noalloc_scratch(NoallocScratch* out) {
    void* pr = nullptr;
    void* ps = nullptr;
    if (cudaGetSymbolAddress(&pr, g_noalloc_rank) != cudaSuccess || pr == nullptr) return BLEND_ECUDA;
    if (cudaGetSymbolAddress(&ps, g_noalloc_sorted) != cudaSuccess || ps == nullptr) return BLEND_ECUDA;
    out->rank = static_cast<int32_t*>(pr);
    out->sorted = static_cast<unsigned long long*>(ps);
    return BLEND_OK;
}
}  // namespace

}  // namespace blend

extern "C" int topk_select_dilate_noalloc(const float* scores, int32_t n, int32_t base, int32_t budget,
                                          int32_t window, int32_t tau, int32_t budget_mode,
                                          const uint8_t* allowed, int32_t* idx_out, int32_t* n_out,
                                          void* stream) {
    using namespace blend;
    if (!scores || !idx_out || !n_out) return report_error(BLEND_EINVAL, "topk_select_dilate_noalloc: NULL pointer");
    if (n < 0 || n > NOALLOC_MAX_N)
        return report_error(BLEND_EINVAL, "topk_select_dilate_noalloc: n outside 0..32768 (size of its fixed scratch)");
    if (budget < 0 || window < 1 || window > BLEND_MAX_WINDOW || tau < 1 || tau > window)
        return report_error(BLEND_EINVAL, "topk_select_dilate_noalloc: bad budget/window/tau");
    if (budget_mode != BLEND_BUDGET_FINAL && budget_mode != BLEND_BUDGET_CANDIDATE)
        return report_error(BLEND_EINVAL, "topk_select_dilate_noalloc: bad budget_mode");
    NoallocScratch scr;
    int rc = noalloc_scratch(&scr);
    if (rc != BLEND_OK) {
        cudaGetLastError();
        return report_error(rc, "topk_select_dilate_noalloc: cannot get the device address of the fixed scratch");
    }
    SelectBatch sb;
    memset(&sb, 0, sizeof sb);
    sb.n_job = 1;
    sb.window = window;
    sb.tau = tau;
    sb.budget_mode = budget_mode;
    sb.j[0] = SelectJob{scores, allowed, idx_out, n_out, n, base, budget, 0, 0};
    // every rank entry the call reads is written by the call first: nothing to clear
    launch_select(sb, scr.rank, scr.sorted, n, (cudaStream_t)stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return report_error(BLEND_ECUDA, cudaGetErrorString(e));
    return BLEND_OK;
}
