// SpecCache token selection on the device (SpecCache notes, "2.3 Semantic span
// completion" with its global budget control, and "2.4 Cross-tokenizer alignment").
//
// Span completion through ranks (from k_rank_tiles / k_rank_merge: score descending, ties by position):
//   * scores are min-max normalised, n~ = (s - min) / (max - min), and token i+1 joins
//     token i's span while |n~(i+1) - n~(i)| / n~(i) < tau_smooth, at most max_span tokens
//     per span.  Every step is one fp32 operation rounded to nearest (no contraction),
//     so each merge decision matches a plain fp32 evaluation of the same formula.
//   * span j is completed at TopK size k iff #{p in j : rank p < k} * 10000 >=
//     tau_cover_bp * |j|, i.e. iff k > r_c(j), the c-th smallest rank in j with
//     c = ceil(tau_cover_bp * |j| / 10000).  So p is in the set at k iff
//     cover(p) = min(rank p, r_c(span of p)) < k, for every k at once.
//   * CANDIDATE: k = budget, then at most `cap` tokens kept, those of highest score.
//     FINAL: the largest k <= budget whose set has at most `budget` tokens (the set
//     grows with k, so it is the budget itself or the (budget+1)-th smallest cover).
// One CTA per request; n <= 32768.  All selection arithmetic is integer.
#include <climits>

#include "common.cuh"

namespace blend {
namespace {

constexpr int SP_THREADS = 1024;
constexpr int SP_MAX_PER_THREAD = 32;  // n <= 32768
constexpr int SP_MAX_N = SP_THREADS * SP_MAX_PER_THREAD;

__device__ __forceinline__ float canon(float x) { return x == 0.f ? 0.f : x; }  // -0 -> +0

// Normalised score of position p.
__device__ __forceinline__ float norm_at(const float* sc, int p, float lo, float rng) {
    return __fdiv_rn(__fsub_rn(canon(sc[p]), lo), rng);
}
// True when token i+1 may join token i's span (relative change below tau_smooth).  A NaN
// or infinite change (normalised score 0, all scores equal, NaN scores) is not below.
__device__ __forceinline__ bool smooth(const float* sc, int i, float lo, float rng, float tau) {
    const float a = norm_at(sc, i, lo, rng), b = norm_at(sc, i + 1, lo, rng);
    const float delta = __fdiv_rn(fabsf(__fsub_rn(b, a)), a);
    return delta < tau;
}

__global__ void __launch_bounds__(SP_THREADS)
    k_span_finish(const __grid_constant__ SelectBatch sb, const int32_t* __restrict__ rank_all) {
    extern __shared__ int32_t cov[];  // n ints (cover values), then n bytes of span-start flags
    __shared__ int red[SP_THREADS];
    __shared__ float fred[2][SP_THREADS / 32];
    __shared__ int warp_tot[SP_THREADS / 32];
    __shared__ int bcast;
    const SelectJob& jb = sb.j[blockIdx.x];
    const int n = jb.n;
    uint8_t* start = reinterpret_cast<uint8_t*>(cov + n);
    const int* rank = rank_all + jb.rank_off;
    const float* sc = jb.scores;
    const int L = sb.max_span;
    const int per = (n + SP_THREADS - 1) / SP_THREADS;
    const int p0 = min(n, (int)threadIdx.x * per), p1 = min(n, p0 + per);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;

    // 1. min and max over the non-NaN scores (fminf / fmaxf skip NaN; exact, so any order)
    float lo = INFINITY, hi = -INFINITY;
    for (int p = p0; p < p1; ++p) {
        const float x = canon(sc[p]);
        lo = fminf(lo, x);
        hi = fmaxf(hi, x);
    }
    for (int o = 16; o > 0; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
        fred[0][wid] = lo;
        fred[1][wid] = hi;
    }
    __syncthreads();
    lo = INFINITY;
    hi = -INFINITY;
    for (int w = 0; w < SP_THREADS / 32; ++w) {
        lo = fminf(lo, fred[0][w]);
        hi = fmaxf(hi, fred[1][w]);
    }
    const float rng = __fsub_rn(hi, lo);
    const float tau = sb.tau_smooth;

    // 2. span starts: a natural segment starts at 0 and after every non-smooth step; inside
    //    one, spans start every L tokens.  The natural start before p0 comes from a block
    //    max-scan of each thread's last natural start.
    int last = -1;
    for (int p = p0; p < p1; ++p)
        if (p == 0 || !smooth(sc, p - 1, lo, rng, tau)) last = p;
    red[threadIdx.x] = last;
    __syncthreads();
    for (int s = 1; s < SP_THREADS; s <<= 1) {  // inclusive max-scan
        const int v = threadIdx.x >= s ? red[threadIdx.x - s] : -1;
        __syncthreads();
        red[threadIdx.x] = max(red[threadIdx.x], v);
        __syncthreads();
    }
    int seg = threadIdx.x > 0 ? red[threadIdx.x - 1] : -1;
    __syncthreads();
    for (int p = p0; p < p1; ++p) {
        if (p == 0 || !smooth(sc, p - 1, lo, rng, tau)) seg = p;
        start[p] = (uint8_t)(((p - seg) % L) == 0);
    }
    __syncthreads();

    // 3. per span (handled by the thread owning its first token): c-th smallest rank, then
    //    cover(p) = min(rank p, r_c) for its members
    for (int u = p0; u < p1; ++u) {
        if (!start[u]) continue;
        int v = u;
        while (v + 1 < n && !start[v + 1]) ++v;
        const int len = v - u + 1;
        const int c = (int)(((long long)sb.tau_cover_bp * len + 9999) / 10000);
        int rc = INT_MAX;
        for (int m = u; m <= v; ++m) {  // ranks are distinct: r_m is c-th iff c-1 are smaller
            const int rm = rank[m];
            int smaller = 0;
            for (int q = u; q <= v; ++q) smaller += rank[q] < rm;
            if (smaller == c - 1) rc = rm;
        }
        for (int m = u; m <= v; ++m) cov[m] = min(rank[m], rc);
    }
    __syncthreads();

    // 4. TopK size and the budget (counts walk rounds of SP_THREADS consecutive positions:
    //    conflict-free shared-memory reads)
    const int tid = threadIdx.x;
    const int kmax = min(jb.budget, n);
    int k = kmax, vcap = INT_MAX;
    int loc = 0;
    for (int p = tid; p < n; p += SP_THREADS) loc += cov[p] < kmax;
    const int f = block_sum_i32(loc, warp_tot, &bcast);
    if (sb.budget_mode == BLEND_BUDGET_FINAL) {
        if (f > jb.budget) {
            // smallest v with #{cover <= v} >= budget + 1
            int a = 0, b = kmax - 1;
            while (a < b) {
                const int mid = (a + b) >> 1;
                loc = 0;
                for (int p = tid; p < n; p += SP_THREADS) loc += cov[p] <= mid;
                if (block_sum_i32(loc, warp_tot, &bcast) >= jb.budget + 1) b = mid;
                else a = mid + 1;
            }
            k = a;
        }
    } else if (f > jb.cap) {
        // keep the cap members of highest score: smallest v with #{member, rank <= v} >= cap
        int a = 0, b = n - 1;
        while (a < b) {
            const int mid = (a + b) >> 1;
            loc = 0;
            for (int p = tid; p < n; p += SP_THREADS) loc += cov[p] < k && rank[p] <= mid;
            if (block_sum_i32(loc, warp_tot, &bcast) >= jb.cap) b = mid;
            else a = mid + 1;
        }
        vcap = jb.cap > 0 ? a : -1;
    }

    // 5. ordered compaction of the members
    const int written =
        compact_in_order(n, jb.base, jb.out, [&](int p) { return cov[p] < k && rank[p] <= vcap; }, warp_tot, &bcast);
    if (tid == 0) *jb.out_n = written;
}

// SpecCache 2.4: mark every target token of every selected speculative token, then write
// the marked ones in order.  One CTA; marks live in shared memory (n_target bytes).
constexpr int AL_THREADS = 1024;
__global__ void __launch_bounds__(AL_THREADS)
    k_align_expand(const int32_t* __restrict__ sel, const int32_t* __restrict__ n_sel_p, int32_t max_sel,
                   int32_t sel_base, const int32_t* __restrict__ a_start, const int32_t* __restrict__ a_end,
                   int32_t n_spec, int32_t n_target, int32_t out_base, int32_t* __restrict__ out,
                   int32_t* __restrict__ n_out, int32_t* __restrict__ err) {
    extern __shared__ uint8_t mark[];
    __shared__ int red[AL_THREADS];
    for (int t = threadIdx.x; t < n_target; t += AL_THREADS) mark[t] = 0;
    __syncthreads();
    const int n_sel = min(max(*n_sel_p, 0), max_sel);
    for (int k = threadIdx.x; k < n_sel; k += AL_THREADS) {
        const int i = sel[k] - sel_base;
        if (i < 0 || i >= n_spec) {
            set_error(err, BLEND_EDEVICE);
            continue;
        }
        const int a = a_start[i], b = a_end[i];
        if (a < 0 || b < a || b > n_target) {
            set_error(err, BLEND_EDEVICE);
            continue;
        }
        for (int t = a; t < b; ++t) mark[t] = 1;  // benign: every writer stores 1
    }
    __syncthreads();
    const int per = (n_target + AL_THREADS - 1) / AL_THREADS;
    const int t0 = min(n_target, (int)threadIdx.x * per), t1 = min(n_target, t0 + per);
    int loc = 0;
    for (int t = t0; t < t1; ++t) loc += mark[t];
    red[threadIdx.x] = loc;
    __syncthreads();
    for (int s = 1; s < AL_THREADS; s <<= 1) {
        const int v = threadIdx.x >= s ? red[threadIdx.x - s] : 0;
        __syncthreads();
        red[threadIdx.x] += v;
        __syncthreads();
    }
    int o = red[threadIdx.x] - loc;
    for (int t = t0; t < t1; ++t)
        if (mark[t]) out[o++] = out_base + t;
    if (threadIdx.x == AL_THREADS - 1) *n_out = red[AL_THREADS - 1];
}

}  // namespace

void launch_span_finish(const SelectBatch& sb, const int32_t* rank_scratch, int max_n, cudaStream_t s) {
    if (sb.n_job <= 0) return;
    if (max_n <= 0) max_n = 1;
    const size_t smem = (size_t)max_n * (sizeof(int32_t) + 1);
    cudaFuncSetAttribute(k_span_finish, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         SP_MAX_N * (int)(sizeof(int32_t) + 1));
    k_span_finish<<<sb.n_job, SP_THREADS, smem, s>>>(sb, rank_scratch);
    note_launch(1);
}

void launch_align_expand(const int32_t* sel, const int32_t* n_sel, int32_t max_sel, int32_t sel_base,
                         const int32_t* a_start, const int32_t* a_end, int32_t n_spec, int32_t n_target,
                         int32_t out_base, int32_t* out, int32_t* n_out, int32_t* err, cudaStream_t s) {
    const size_t smem = (size_t)(n_target > 0 ? n_target : 1);
    cudaFuncSetAttribute(k_align_expand, cudaFuncAttributeMaxDynamicSharedMemorySize, BLEND_MAX_ALIGN_TARGETS);
    k_align_expand<<<1, AL_THREADS, smem, s>>>(sel, n_sel, max_sel, sel_base, a_start, a_end, n_spec, n_target,
                                               out_base, out, n_out, err);
    note_launch(1);
}

}  // namespace blend
