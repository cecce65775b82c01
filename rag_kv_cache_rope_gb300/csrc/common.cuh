// Shared device helpers and internal launch interfaces of libblend.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/blend.h"

namespace blend {

using bf16 = __nv_bfloat16;

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// 16-byte vector of T: 4 floats or 8 bf16.
template <typename T> struct Vec {
    static constexpr int N = 16 / sizeof(T);
    uint4 raw;
    __device__ __forceinline__ float get(int i) const {
        const T* p = reinterpret_cast<const T*>(&raw);
        return to_f<T>(p[i]);
    }
    __device__ __forceinline__ void set(int i, float v) {
        T* p = reinterpret_cast<T*>(&raw);
        p[i] = from_f<T>(v);
    }
};

template <typename T> __device__ __forceinline__ Vec<T> ld16(const T* p) {
    Vec<T> v;
    v.raw = *reinterpret_cast<const uint4*>(p);
    return v;
}
template <typename T> __device__ __forceinline__ void st16(T* p, const Vec<T>& v) {
    *reinterpret_cast<uint4*>(p) = v.raw;
}

// Counts kernel launches made by the library (process-wide; read by blend_launch_count).
void note_launch(int n = 1);
// Records `msg` as the text blend_last_error(NULL) returns and returns `code`.
int report_error(int code, const char* msg);

// Records the first device-side failure (code, where) in the handle's error word.
__device__ __forceinline__ void set_error(int32_t* err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

// Deterministic block-wide sum (fixed tree order) of one float per thread.
// `red` must hold blockDim.x floats; blockDim.x a power of two <= 1024.
__device__ __forceinline__ float block_sum(float v, float* red) {
    const int t = threadIdx.x;
    red[t] = v;
    __syncthreads();
    for (int s = blockDim.x >> 1; s > 0; s >>= 1) {
        if (t < s) red[t] += red[t + s];
        __syncthreads();
    }
    float r = red[0];
    __syncthreads();
    return r;
}

// Deterministic block-wide integer sum (warp reductions, then one warp over the warp
// totals); every thread gets the result.  Two barriers.
__device__ __forceinline__ int block_sum_i32(int v, int* warp_tot, int* bcast) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = __reduce_add_sync(0xffffffffu, v);
    if (lane == 0) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int x = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
        x = __reduce_add_sync(0xffffffffu, x);
        if (lane == 0) *bcast = x;
    }
    __syncthreads();
    return *bcast;
}

// Ordered compaction for one CTA: out[j] = base + p for the positions p < n with keep(p),
// in ascending order, walked in rounds of blockDim.x consecutive positions (ballots within a
// warp, a scan of the warp counts); returns the count to every thread.  warp_tot holds
// blockDim.x / 32 ints (blockDim.x a multiple of 32, at most 1024).
template <typename Keep>
__device__ __forceinline__ int compact_in_order(int n, int base, int32_t* out, Keep keep, int* warp_tot, int* bcast) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    int written = 0;
    for (int r0 = 0; r0 < n; r0 += blockDim.x) {
        const int p = r0 + tid;
        const bool take = p < n && keep(p);
        const unsigned m = __ballot_sync(0xffffffffu, take);
        if (lane == 0) warp_tot[warp] = __popc(m);
        __syncthreads();
        if (warp == 0) {
            const int v = lane < nw ? warp_tot[lane] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane < nw) warp_tot[lane] = incl - v;
            if (lane == 31) *bcast = incl;
        }
        __syncthreads();
        if (take) out[written + warp_tot[warp] + __popc(m & ((1u << lane) - 1u))] = base + p;
        written += *bcast;
        __syncthreads();
    }
    return written;
}

// Per-request description of a batch, passed to kernels by value.
struct ReqDesc {
    int32_t tok_off;  // first blended token of the request in the batch K/V
    int32_t P;        // prefix rows
    int32_t n_c;      // chunk rows
    int32_t Q;        // query rows
    int32_t nc_off;   // first chunk row of the request in per-chunk-row arrays
    int32_t q_off;    // first query row of the request in the hidden output
};
struct BatchDesc {
    int32_t n_req;
    ReqDesc r[BLEND_MAX_BATCH];
};

// Assembly segment: n_rows pool rows from src_row go to blended tokens dst_tok..,
// keys rotated by delta positions.
struct Seg {
    int32_t row0;     // first linear row of this segment (sum of earlier n_rows)
    int32_t src_row;
    int32_t dst_tok;
    int32_t n_rows;
    int32_t delta;
};
struct SegTable {
    int32_t n_seg;
    int32_t total_rows;
    Seg s[BLEND_MAX_CHUNKS + BLEND_MAX_BATCH];
};
struct QueryTable {
    int32_t n;
    const int32_t* ptr[BLEND_MAX_BATCH];
    int32_t dst_tok[BLEND_MAX_BATCH];
    int32_t len[BLEND_MAX_BATCH];
};

// Stage set of every request: positions at set + nc_off[r], count at count[r];
// iota 1: the set is every chunk row P..P+n_c-1; iota 2: every row 0..P+n_c-1.
// max_count > 0 caps every request's count (a caller-given count above it is reported).
struct StageDesc {
    const int32_t* set;
    const int32_t* count;
    int32_t iota;
    int32_t max_count;
};

// ------------------------------ launchers (kernels_mem.cu) -------------------------
// dev_out of launch_rope_qkv: per chunk row of each request (dev_by_row = 0, indexed
// nc_off + pos - P, other rows skipped) or per recomputed row (dev_by_row = 1).
void launch_rope_table(float2* tab, int max_pos, int head_dim, double theta, cudaStream_t s);
void launch_realign(int dtype, const void* src, void* dst, int n_rows, const int32_t* delta,
                    int n_layers, long long src_layer_rows, long long dst_layer_rows, int hkv, int d,
                    const float2* tab, int max_pos, int32_t* err, cudaStream_t s);
void launch_assemble(int dtype, const SegTable& segs, const void* pool_k, const void* pool_v,
                     long long pool_rows, void* out_k, void* out_v, long long out_tokens,
                     int n_layers, int hkv, int d, const float2* tab, int max_pos, int32_t* err,
                     cudaStream_t s, int layer0 = 0);
void launch_tokens(const SegTable& segs, const QueryTable& qt, const int32_t* pool_tokens,
                   int32_t* out_tokens, cudaStream_t s);
void launch_rmsnorm(int dtype, const float* x, const void* g, void* out, int H, float eps,
                    const int32_t* M_dev, int M_max, cudaStream_t s);
void launch_embed(int dtype, const void* embed, const int32_t* tokens, const int32_t* row_tok,
                  float* x, int H, int vocab, const int32_t* M_dev, int M_max, int32_t* err,
                  cudaStream_t s);
void launch_gather(const void* src, long long row_bytes, long long src_rows, const int32_t* idx,
                   const int32_t* n_dev, int max_n, void* dst, int32_t* err, cudaStream_t s);
void launch_rope_qkv(int dtype, const float* qkv, const int32_t* row_pos, const int32_t* row_tok,
                     const int32_t* row_req, const int32_t* M_dev, int M_max, const BatchDesc& bd,
                     int hq, int hkv, int d, int m_cap, const float2* tab, void* q_out, void* k_cache,
                     void* v_cache, float* dev_out, int dev_mode, int dev_by_row, cudaStream_t s);
void launch_deviation(int dtype, const void* k_new, const void* v_new, const void* k_cache,
                      const void* v_cache, const int32_t* pos, const int32_t* n_dev, int max_rows,
                      long long n_ctx, int kv_elems, int mode, float* dev_out, int32_t* err, cudaStream_t s);
void launch_scatter(int dtype, const void* k_new, const void* v_new, const int32_t* pos,
                    const int32_t* n_dev, int max_n, long long n_ctx, int kv_elems, void* k_cache,
                    void* v_cache, int32_t* err, cudaStream_t s);
void launch_final_norm(int dtype, const float* x, const void* g, void* hidden, int H, float eps,
                       const BatchDesc& bd, const int32_t* req_row_end, cudaStream_t s);
void launch_importance(int dtype, const void* hidden, int n, int n_layers, int dim, float* out,
                       cudaStream_t s);
// With old_row_tok/old_M (the previous plan) set, row_src receives each new row's row in
// the previous plan; positions missing from the previous plan are reported in err.
void launch_plan(const BatchDesc& bd, const StageDesc& st, int32_t* row_pos, int32_t* row_tok,
                 int32_t* row_req, int32_t* row_src, int32_t* pos2row, int32_t* M_dev,
                 int32_t* req_row_end, const int32_t* old_row_tok, const int32_t* old_M, int32_t* err,
                 cudaStream_t s);
void launch_set_mask(const BatchDesc& bd, const int32_t* set, const int32_t* count, uint8_t* mask,
                     cudaStream_t s);
void launch_fill_i32(int32_t* p, int32_t v, long long n, cudaStream_t s);
// EPIC sets: run q writes positions start[q] .. start[q]+count[q]-1 at set + out[q]; request
// r's set size is req_n[r].
struct EpicTable {
    int32_t n_run;
    int32_t n_req;
    int32_t start[BLEND_MAX_CHUNKS];
    int32_t count[BLEND_MAX_CHUNKS];
    int32_t out[BLEND_MAX_CHUNKS];
    int32_t req_n[BLEND_MAX_BATCH];
};
void launch_epic_set(const EpicTable& et, int32_t* set, int32_t* set_n, cudaStream_t s);
void launch_wait_flag(const int32_t* flag, long long max_polls, int32_t* err, cudaStream_t s);
// Cache-Craft focus filter: request r's chunks are chunk0[r] .. chunk0[r]+n_chunks[r]-1 of the
// tables (start = blended position of the chunk's first token, len = its tokens).
struct FocusTable {
    int32_t n_req;
    int32_t chunk0[BLEND_MAX_BATCH];
    int32_t n_chunks[BLEND_MAX_BATCH];
    int32_t start[BLEND_MAX_CHUNKS];
    int32_t len[BLEND_MAX_CHUNKS];
};
void launch_focus_filter(const BatchDesc& bd, const FocusTable& ft, const float* scores, int32_t focus_bp,
                         const int32_t* set_in, const int32_t* n_in, int32_t* set_out, int32_t* n_out,
                         cudaStream_t s);
void launch_copy_sets(const BatchDesc& bd, const int32_t* src, const int32_t* src_n, int32_t* dst,
                      int32_t* dst_n, cudaStream_t s);

// ------------------------------ selection (select.cu) ------------------------------
struct SelectJob {
    const float* scores;   // [n]
    const uint8_t* allowed;  // [n] or null (window rule only)
    int32_t* out;          // [n]
    int32_t* out_n;        // scalar
    int32_t n;
    int32_t base;
    int32_t budget;
    int32_t rank_off;      // offset of this job's rank scratch
    int32_t cap;           // span rule, CANDIDATE budget: most tokens kept after completion
};
struct SelectBatch {
    int32_t n_job;
    int32_t window, tau, budget_mode;
    int32_t rule;          // BLEND_GROUP_WINDOW or BLEND_GROUP_SPAN
    float tau_smooth;      // span rule: SpecCache 2.3 thresholds and span length
    int32_t tau_cover_bp, max_span;
    SelectJob j[BLEND_MAX_BATCH];
};
// Ranks (select.cu), then the window rule (select.cu) or the span rule (span.cu).
// sort_scratch: n_job * roundup(max_n, 2048) keys (select.cu, RANK_TILE).
void launch_select(const SelectBatch& sb, int32_t* rank_scratch, unsigned long long* sort_scratch, int max_n,
                   cudaStream_t s);
void launch_rank(const SelectBatch& sb, int32_t* rank_scratch, unsigned long long* sort_scratch, int max_n,
                 cudaStream_t s);
void launch_span_finish(const SelectBatch& sb, const int32_t* rank_scratch, int max_n, cudaStream_t s);
// CacheClip 6.2 auxiliary scores (aux.cu): the query rows' last-layer q out of the per-kv-head
// slab, then per chunk column the mean attention weight over query rows and heads.
void launch_gather_qlast(int dtype, const void* qslab, int m_cap, int group, int hkv, int d, const BatchDesc& bd,
                         const int32_t* req_row_end, void* q_last, int n_qrows, cudaStream_t s);
// stats: n_qrows * hq * n_spans pairs of floats (score_spans(max_tokens) spans per row
// and head for the tensor-core path, one for the CUDA-core path).
void launch_aux_scores(int dtype, const void* q_last, const void* K, const BatchDesc& bd, int hq, int hkv, int d,
                       int n_qrows, int max_nc, float2* stats, int n_spans, float* scores, int32_t* err,
                       bool tensor_cores, cudaStream_t s);
// Tensor-core form of the same two passes (score_tc.cu): bf16, head_dim 64 or 128.
// Returns BLEND_EUNSUPPORTED when it cannot run here.
int launch_scores_tc(const void* q_last, const void* K, long long n_tokens, const BatchDesc& bd, int hq, int hkv,
                     int d, int n_spans, float2* part, float* scores, int32_t* err, cudaStream_t s);
// Key spans per (query row, head) the tensor-core statistics pass writes for contexts of
// up to max_tokens tokens.
int tc_score_spans(long long max_tokens);
// SpecCache 2.4: sorted distinct union of [a_start[i], a_end[i]) over the selected i.
void launch_align_expand(const int32_t* sel, const int32_t* n_sel, int32_t max_sel, int32_t sel_base,
                         const int32_t* a_start, const int32_t* a_end, int32_t n_spec, int32_t n_target,
                         int32_t out_base, int32_t* out, int32_t* n_out, int32_t* err, cudaStream_t s);

// ------------------------------ GEMM (gemm_simt.cu) --------------------------------
enum Epi { EPI_STORE_F32 = 0, EPI_ADD_F32 = 1, EPI_SWIGLU = 2, EPI_QKV_ROPE = 3 };
// Extra arguments of the fused QKV epilogue (tensor-core GEMM, head_dim 128): rotate q and
// k at each row's blended position, store q per kv head ([m_cap][group][128] slabs) and
// k, v straight into this layer's cache rows [tok][hkv][128].
struct QkvEpi {
    const int32_t* row_pos;
    const int32_t* row_tok;
    const float2* rope;  // [max_pos][64] (cos, sin)
    bf16* q;
    bf16* k_cache;
    bf16* v_cache;
    int m_cap, group, hq, hkv;
};
// C = A[M,K] . B[N,K]^T with A, B of the model dtype; epilogue:
//   EPI_STORE_F32: C fp32 [M][ldc] = acc
//   EPI_ADD_F32:   C fp32 [M][ldc] += acc
//   EPI_SWIGLU:    C dtype [M][N/2]: gate/up interleaved in blocks of BLEND_GU_BLOCK
// RMSNorm folded into the tensor-core GEMMs: RMSNorm(x) . W = (1 / rms(x)) ((x * g) . W).
// Producer side (a residual-add GEMM, x_out set): besides the fp32 rows it writes
// bf16(x * g) to x_out [rows][ldx] (g: the next norm's gain, per column) and each row's sum
// of squares over the tile's columns to ssq_out[row * ssq_stride + n_tile].  Consumer side
// (ssq_in set): every accumulator of a row is scaled by 1 / sqrt(sum of its n_part partials
// * inv_h + eps) before the epilogue.
struct NormEpi {
    const float* ssq_in;
    int n_part;
    float inv_h, eps;
    bf16* x_out;
    const bf16* g;
    float* ssq_out;
    int ssq_stride;
    int ldx;
};

void launch_gemm_simt(int dtype, const void* A, int lda, const void* B, int ldb, int K, int N,
                      const int32_t* M_dev, int M_max, int epi, void* C, int ldc, cudaStream_t s);

// ------------------------------ attention (attn_simt.cu) ---------------------------
// q: per kv head g a slab [m_cap][group][d]; o: [M][hq*d].
void launch_attn_simt(int dtype, const void* q, int m_cap, const int32_t* row_pos, const int32_t* row_tok,
                      const int32_t* M_dev, int M_max, const void* k_cache, const void* v_cache,
                      void* o, int hq, int hkv, int d, cudaStream_t s);

}  // namespace blend
