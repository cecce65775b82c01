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
#include <mutex>

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

// rank[t] = #{u allowed : key(u) < key(t)} for allowed t, INT_MAX otherwise.
__global__ void __launch_bounds__(256)
    k_rank(const __grid_constant__ SelectBatch sb, int32_t* __restrict__ rank) {
    __shared__ unsigned long long tile[RANK_TILE];
    const SelectJob& jb = sb.j[blockIdx.y];
    const int n = jb.n;
    if (blockIdx.x * blockDim.x >= n) return;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const bool mine_ok = t < n && (jb.allowed == nullptr || jb.allowed[t] != 0);
    const unsigned long long mine = mine_ok ? sel_key(jb.scores[t], t) : ~0ull;
    int cnt = 0;
    for (int base = 0; base < n; base += RANK_TILE) {
        for (int i = threadIdx.x; i < RANK_TILE; i += blockDim.x) {
            int u = base + i;
            unsigned long long key = ~0ull;
            if (u < n && (jb.allowed == nullptr || jb.allowed[u] != 0)) key = sel_key(jb.scores[u], u);
            tile[i] = key;
        }
        __syncthreads();
        const int lim = min(RANK_TILE, n - base);
#pragma unroll 8
        for (int i = 0; i < lim; ++i) cnt += (tile[i] < mine) ? 1 : 0;
        __syncthreads();
    }
    if (t < n) rank[jb.rank_off + t] = mine_ok ? cnt : INT_MAX;
}

__device__ __forceinline__ int block_sum_int(int v, int* red) {
    const int t = threadIdx.x;
    red[t] = v;
    __syncthreads();
    for (int s = blockDim.x >> 1; s > 0; s >>= 1) {
        if (t < s) red[t] += red[t + s];
        __syncthreads();
    }
    int r = red[0];
    __syncthreads();
    return r;
}

// One CTA per job.  Thread i owns the contiguous positions [i*per, (i+1)*per).
__global__ void __launch_bounds__(SEL_THREADS)
    k_select_finish(const __grid_constant__ SelectBatch sb, const int32_t* __restrict__ rank_all) {
    extern __shared__ int32_t cov[];  // n ints: qual, then cover
    __shared__ int red[SEL_THREADS];
    const SelectJob& jb = sb.j[blockIdx.x];
    const int n = jb.n;
    const int w = sb.window, tau = sb.tau;
    const int* rank = rank_all + jb.rank_off;
    const int per = (n + SEL_THREADS - 1) / SEL_THREADS;
    const int p0 = min(n, threadIdx.x * per), p1 = min(n, p0 + per);

    int loc = 0;
    for (int t = p0; t < p1; ++t) loc += rank[t] != INT_MAX;
    const int n_ok = block_sum_int(loc, red);
    const int kmax = min(jb.budget, n_ok);

    // qual(t); ranks >= kmax can never be candidates and count as infinite.
    for (int t = p0; t < p1; ++t) {
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
    int cl[SEL_MAX_PER_THREAD];
#pragma unroll
    for (int e = 0; e < SEL_MAX_PER_THREAD; ++e) {
        const int p = p0 + e;
        int c = INT_MAX;
        if (p < p1) {
            if (jb.allowed == nullptr || jb.allowed[p] != 0) {
                const int lo = max(0, p - w + 1);
                for (int t = lo; t <= p; ++t) c = min(c, cov[t]);
            }
        }
        cl[e] = c;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < SEL_MAX_PER_THREAD; ++e)
        if (p0 + e < p1) cov[p0 + e] = cl[e];
    __syncthreads();

    int k = kmax;
    if (sb.budget_mode == BLEND_BUDGET_FINAL && kmax > 0) {
        loc = 0;
        for (int p = p0; p < p1; ++p) loc += cov[p] < kmax;
        const int f = block_sum_int(loc, red);
        if (f > jb.budget) {
            // smallest v with #{cover <= v} >= budget + 1
            int lo = 0, hi = kmax - 1;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                loc = 0;
                for (int p = p0; p < p1; ++p) loc += cov[p] <= mid;
                const int c = block_sum_int(loc, red);
                if (c >= jb.budget + 1) hi = mid;
                else lo = mid + 1;
            }
            k = lo;
        }
    }

    // ordered compaction of {p : cover(p) < k}
    loc = 0;
    for (int p = p0; p < p1; ++p) loc += cov[p] < k;
    red[threadIdx.x] = loc;
    __syncthreads();
    for (int s = 1; s < SEL_THREADS; s <<= 1) {  // inclusive Hillis-Steele scan
        int v = threadIdx.x >= s ? red[threadIdx.x - s] : 0;
        __syncthreads();
        red[threadIdx.x] += v;
        __syncthreads();
    }
    int o = red[threadIdx.x] - loc;
    for (int p = p0; p < p1; ++p)
        if (cov[p] < k) jb.out[o++] = jb.base + p;
    if (threadIdx.x == SEL_THREADS - 1) *jb.out_n = red[SEL_THREADS - 1];
}

void launch_rank(const SelectBatch& sb, int32_t* rank_scratch, int max_n, cudaStream_t s) {
    if (sb.n_job <= 0) return;
    if (max_n <= 0) max_n = 1;
    dim3 g1((max_n + 255) / 256, sb.n_job);
    k_rank<<<g1, 256, 0, s>>>(sb, rank_scratch);
    note_launch(1);
}

void launch_select(const SelectBatch& sb, int32_t* rank_scratch, int max_n, cudaStream_t s) {
    if (sb.n_job <= 0) return;
    if (max_n <= 0) max_n = 1;
    launch_rank(sb, rank_scratch, max_n, s);
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
// Rank scratch of topk_select_dilate_noalloc: a fixed array in device memory, so the
// call needs neither a handle nor any allocation.  Every GPU that loads the library
// holds these 128 KB until the process exits.
constexpr int NOALLOC_MAX_N = 32768;
static __device__ __align__(256) int32_t g_noalloc_rank[NOALLOC_MAX_N];

namespace {
constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mu;
int32_t* g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {};

// Device address of g_noalloc_rank on the current device (looked up once per device;
// the host-side name of the array is only a stand-in and must not reach a kernel).
int noalloc_scratch(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BLEND_ECUDA;
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return BLEND_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_rank) != cudaSuccess || p == nullptr) return BLEND_ECUDA;
        g_noalloc_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_noalloc_ptr[dev];
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
    int32_t* rank = nullptr;
    int rc = noalloc_scratch(&rank);
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
    launch_select(sb, rank, n, (cudaStream_t)stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return report_error(BLEND_ECUDA, cudaGetErrorString(e));
    return BLEND_OK;
}
