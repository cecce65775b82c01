// Auxiliary-model importance scores (CacheClip blog, "6.2 Auxiliary-model-guided token
// selection": the score of a chunk token is the mean, over the query rows, of the
// last-layer attention weight on it; CacheClip paper 4.2).  The auxiliary model's
// forward over the query rows is blend_prefill itself (FORCED mode with an empty stage:
// only the query rows are computed, over the chunk's cached rows); it leaves the last
// layer's keys in the blended cache and, on request, the query rows' last-layer q.
//
// bf16 models with head_dim 64 or 128 take the tensor-core form of these two passes
// (score_tc.cu); the CUDA-core passes below serve the rest:
//   k_aux_row_stats : per (query row, head) the softmax maximum m and sum l over every key
//                     the row sees (prefix, chunk and the query rows up to itself); one
//                     warp per (row, head), lane j takes keys j, j+32, ..., then a fixed
//                     butterfly merges the lanes' (m, l).
//   k_aux_colmean   : per chunk column j, sum over (row, head) of exp(s - m) / l in a fixed
//                     order, then divided by Q x hq.  Chunk columns precede every query
//                     position, so no causal mask applies to them.
// Both passes form s = (q . k) / sqrt(d) with the same sequential dot product.
#include <math.h>

#include "common.cuh"

namespace blend {
namespace {

template <typename T, int D>
__device__ __forceinline__ float dot_row(const float* q, const T* k) {
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < D; c += Vec<T>::N) {
        const Vec<T> v = ld16(k + c);
#pragma unroll
        for (int e = 0; e < Vec<T>::N; ++e) s = fmaf(q[c + e], v.get(e), s);
    }
    return s;
}

// Which request a query row (0..sum Q-1) belongs to.
__device__ __forceinline__ int req_of_qrow(const BatchDesc& bd, int qrow) {
    int r = 0;
    while (r + 1 < bd.n_req && bd.r[r + 1].q_off <= qrow) ++r;
    return r;
}

template <typename T>
__global__ void k_gather_qlast(const T* __restrict__ qslab, int m_cap, int group, int hkv, int d,
                               const __grid_constant__ BatchDesc bd, const int32_t* __restrict__ req_row_end,
                               T* __restrict__ q_last, int n_qrows) {
    const int qrow = blockIdx.x;
    if (qrow >= n_qrows) return;
    const int r = req_of_qrow(bd, qrow);
    const int row = req_row_end[r] - bd.r[r].Q + (qrow - bd.r[r].q_off);
    const int per = group * d;  // elements of one kv head's q heads
    for (int e = threadIdx.x * Vec<T>::N; e < hkv * per; e += blockDim.x * Vec<T>::N) {
        const int g = e / per, o = e % per;
        st16(q_last + (long long)qrow * hkv * per + e, ld16(qslab + ((long long)g * m_cap + row) * per + o));
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(128)
    k_aux_row_stats(const T* __restrict__ q_last, const T* __restrict__ K, const __grid_constant__ BatchDesc bd,
                    int hq, int hkv, float scale, int n_qrows, float2* __restrict__ stats) {
    const int item = blockIdx.x * 4 + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (item >= n_qrows * hq) return;
    const int qrow = item / hq, h = item % hq;
    const int r = req_of_qrow(bd, qrow);
    const ReqDesc& rd = bd.r[r];
    const int pos = rd.P + rd.n_c + (qrow - rd.q_off);  // keys 0..pos of the request
    const int g = h / (hq / hkv);
    float q[D];
#pragma unroll
    for (int c = 0; c < D; ++c) q[c] = to_f<T>(q_last[((long long)qrow * hq + h) * D + c]);
    float m = -INFINITY, l = 0.f;
    for (int j = lane; j <= pos; j += 32) {
        const float s = dot_row<T, D>(q, K + ((long long)(rd.tok_off + j) * hkv + g) * D) * scale;
        const float mn = fmaxf(m, s);
        l = l * expf(m - mn) + expf(s - mn);
        m = mn;
    }
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
        const float mn = fmaxf(m, m2);
        // a lane that saw no key has m = -inf, l = 0: it contributes nothing
        const float a = (m == -INFINITY) ? 0.f : l * expf(m - mn);
        const float b = (m2 == -INFINITY) ? 0.f : l2 * expf(m2 - mn);
        l = a + b;
        m = mn;
    }
    if (lane == 0) stats[item] = make_float2(m, l);
}

constexpr int CM_COLS = 32;
constexpr int CM_GROUPS = 8;

template <typename T, int D>
__global__ void __launch_bounds__(CM_COLS * CM_GROUPS)
    k_aux_colmean(const T* __restrict__ q_last, const T* __restrict__ K, const float2* __restrict__ stats,
                  const __grid_constant__ BatchDesc bd, int hq, int hkv, float scale, float* __restrict__ scores) {
    __shared__ float part[CM_GROUPS][CM_COLS];
    const int r = blockIdx.y;
    const ReqDesc& rd = bd.r[r];
    const int col = threadIdx.x % CM_COLS, grp = threadIdx.x / CM_COLS;
    const int j = blockIdx.x * CM_COLS + col;  // chunk column (0..n_c-1)
    const bool live = j < rd.n_c;
    const int group = hq / hkv;
    float acc = 0.f;
    if (blockIdx.x * CM_COLS < rd.n_c) {
        const long long key = rd.tok_off + rd.P + (live ? j : 0);
        for (int g = 0; g < hkv; ++g) {
            float k[D];
#pragma unroll
            for (int c = 0; c < D; ++c) k[c] = to_f<T>(K[(key * hkv + g) * D + c]);
            // (row, head) pairs of this kv head, dealt to the groups in a fixed order
            for (int t = grp; t < rd.Q * group; t += CM_GROUPS) {
                const int qrow = rd.q_off + t / group, h = g * group + t % group;
                const float s = dot_row<T, D>(k, q_last + ((long long)qrow * hq + h) * D);
                const float2 st = stats[(long long)qrow * hq + h];
                acc += expf(s * scale - st.x) / st.y;
            }
        }
    }
    part[grp][col] = acc;
    __syncthreads();
    if (grp == 0 && live) {
        float tot = 0.f;
        for (int q = 0; q < CM_GROUPS; ++q) tot += part[q][col];
        scores[rd.nc_off + j] = tot / (float)(rd.Q * hq);
    }
}

// One CTA per request: each chunk's attention mass (its tokens' scores summed in order by
// one thread), the total (fixed tree), the focused flags, then the ordered compaction of
// the request's set to the rows of focused chunks.
constexpr int FF_THREADS = 1024;
__global__ void __launch_bounds__(FF_THREADS)
    k_focus_filter(const __grid_constant__ BatchDesc bd, const __grid_constant__ FocusTable ft,
                   const float* __restrict__ scores, int32_t focus_bp, const int32_t* __restrict__ set_in,
                   const int32_t* __restrict__ n_in, int32_t* __restrict__ set_out, int32_t* __restrict__ n_out) {
    __shared__ float mass[BLEND_MAX_CHUNKS];
    __shared__ uint8_t focused[BLEND_MAX_CHUNKS];
    __shared__ float red[FF_THREADS];
    __shared__ int cnt[FF_THREADS];
    const int r = blockIdx.x;
    const ReqDesc& rd = bd.r[r];
    const int c0 = ft.chunk0[r], nch = ft.n_chunks[r];
    const float* sc = scores + rd.nc_off;
    for (int j = threadIdx.x; j < nch; j += FF_THREADS) {
        const int a = ft.start[c0 + j] - rd.P;  // chunk-row index of its first token
        float m = 0.f;
        for (int t = 0; t < ft.len[c0 + j]; ++t) m += sc[a + t];
        mass[j] = m;
    }
    __syncthreads();
    float part = 0.f;
    for (int j = threadIdx.x; j < nch; j += FF_THREADS) part += mass[j];
    red[threadIdx.x] = part;
    __syncthreads();
    for (int w = FF_THREADS / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    const float total = red[0];
    for (int j = threadIdx.x; j < nch; j += FF_THREADS)
        focused[j] = (uint8_t)(mass[j] * 10000.f >= (float)focus_bp * total);
    __syncthreads();
    const int n = min(max(n_in[r], 0), rd.n_c);
    const int32_t* in = set_in + rd.nc_off;
    const int per = (n + FF_THREADS - 1) / FF_THREADS;
    const int i0 = min(n, (int)threadIdx.x * per), i1 = min(n, i0 + per);
    auto keep = [&](int p) -> bool {  // chunk of position p by binary search over the starts
        int lo = 0, hi = nch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ft.start[c0 + mid] <= p) lo = mid;
            else hi = mid - 1;
        }
        return nch > 0 && focused[lo];
    };
    int loc = 0;
    for (int i = i0; i < i1; ++i) loc += keep(in[i]);
    cnt[threadIdx.x] = loc;
    __syncthreads();
    for (int w = 1; w < FF_THREADS; w <<= 1) {
        const int v = threadIdx.x >= w ? cnt[threadIdx.x - w] : 0;
        __syncthreads();
        cnt[threadIdx.x] += v;
        __syncthreads();
    }
    int o = cnt[threadIdx.x] - loc;
    for (int i = i0; i < i1; ++i)
        if (keep(in[i])) set_out[rd.nc_off + o++] = in[i];
    if (threadIdx.x == FF_THREADS - 1) n_out[r] = cnt[FF_THREADS - 1];
}

}  // namespace

void launch_focus_filter(const BatchDesc& bd, const FocusTable& ft, const float* scores, int32_t focus_bp,
                         const int32_t* set_in, const int32_t* n_in, int32_t* set_out, int32_t* n_out,
                         cudaStream_t s) {
    k_focus_filter<<<bd.n_req, FF_THREADS, 0, s>>>(bd, ft, scores, focus_bp, set_in, n_in, set_out, n_out);
    note_launch(1);
}

void launch_gather_qlast(int dtype, const void* qslab, int m_cap, int group, int hkv, int d, const BatchDesc& bd,
                         const int32_t* req_row_end, void* q_last, int n_qrows, cudaStream_t s) {
    if (n_qrows <= 0) return;
    if (dtype == BLEND_BF16)
        k_gather_qlast<bf16><<<n_qrows, 128, 0, s>>>((const bf16*)qslab, m_cap, group, hkv, d, bd, req_row_end,
                                                     (bf16*)q_last, n_qrows);
    else
        k_gather_qlast<float><<<n_qrows, 128, 0, s>>>((const float*)qslab, m_cap, group, hkv, d, bd, req_row_end,
                                                      (float*)q_last, n_qrows);
    note_launch(1);
}

template <typename T, int D>
void aux_scores_t(const void* q_last, const void* K, const BatchDesc& bd, int hq, int hkv, int n_qrows, int max_nc,
                  float2* stats, float* scores, cudaStream_t s) {
    const float scale = 1.f / sqrtf((float)D);
    const int items = n_qrows * hq;
    dim3 g2((max_nc + CM_COLS - 1) / CM_COLS, bd.n_req);
    k_aux_row_stats<T, D><<<(items + 3) / 4, 128, 0, s>>>((const T*)q_last, (const T*)K, bd, hq, hkv, scale, n_qrows,
                                                         stats);
    k_aux_colmean<T, D><<<g2, CM_COLS * CM_GROUPS, 0, s>>>((const T*)q_last, (const T*)K, stats, bd, hq, hkv, scale,
                                                          scores);
}

void launch_aux_scores(int dtype, const void* q_last, const void* K, const BatchDesc& bd, int hq, int hkv, int d,
                       int n_qrows, int max_nc, float2* stats, int n_spans, float* scores, int32_t* err,
                       bool tensor_cores, cudaStream_t s) {
    if (n_qrows <= 0 || max_nc <= 0) return;
    if (dtype == BLEND_BF16 && tensor_cores) {
        // tensor cores where they apply (score_tc.cu), else the CUDA-core passes below
        const ReqDesc& last = bd.r[bd.n_req - 1];
        const long long n_tokens = (long long)last.tok_off + last.P + last.n_c + last.Q;
        if (launch_scores_tc(q_last, K, n_tokens, bd, hq, hkv, d, n_spans, stats, scores, err, s) == BLEND_OK)
            return;
    }
    if (dtype == BLEND_BF16) {
        if (d == 64) aux_scores_t<bf16, 64>(q_last, K, bd, hq, hkv, n_qrows, max_nc, stats, scores, s);
        else aux_scores_t<bf16, 128>(q_last, K, bd, hq, hkv, n_qrows, max_nc, stats, scores, s);
    } else {
        if (d == 64) aux_scores_t<float, 64>(q_last, K, bd, hq, hkv, n_qrows, max_nc, stats, scores, s);
        else aux_scores_t<float, 128>(q_last, K, bd, hq, hkv, n_qrows, max_nc, stats, scores, s);
    }
    note_launch(2);
}

}  // namespace blend
