// Tensor-core (tcgen05) GEMM interface: C = A[M,K] . B[N,K]^T in bf16 with fp32
// accumulation and the epilogues of Epi (common.cuh).
#pragma once
#include "common.cuh"

namespace blend {
// 1 when the current device is an sm_103 GPU and the TMA descriptor encoder is
// reachable; also sets the kernels' shared-memory limits.
int tc_available();
// Shapes the tensor-core kernel takes: K % 64 == 0, N >= 128 and N % 32 == 0 (N % 256 == 0
// for EPI_QKV_ROPE), ldc % 8 == 0, and an A buffer of at least 128 rows (M_cap).
bool tc_gemm_supported(int K, int N, int epi, int ldc, int M_cap);
// Split-tile workspace of launch_gemm_tc (fp32): the K-part partials of the split tiles,
// 640 blocks of 128 x 256 (a CTA-pair tile of 256 rows takes two per part), e.g. four
// parts of 76 CTA-pair tiles.
constexpr size_t GEMM_SPLIT_WS_FLOATS = (size_t)640 * 128 * 256;
// A: [M_cap][K] bf16 buffer whose first *M_dev rows are used; B: [N][K] bf16.  With
// split_ws (GEMM_SPLIT_WS_FLOATS, not for EPI_QKV_ROPE) a last wave that is at most half
// full runs as K halves, and a launch with fewer tiles than slots may run every tile as
// 2-4 K parts; a second small kernel finishes the split tiles.  A folded-norm producer (norm->x_out) writes gemm_tc_norm_parts(N) partial sums
// of squares per row (norm->ssq_stride must equal it).  Returns BLEND_OK or
// BLEND_EUNSUPPORTED (operands not describable by a tensor map).
int launch_gemm_tc(const void* A, int K, int M_cap, const void* B, int N, const int32_t* M_dev, int M_max,
                   int epi, void* C, int ldc, int32_t* err, cudaStream_t s, const QkvEpi* qkv = nullptr,
                   float* split_ws = nullptr, const NormEpi* norm = nullptr);
// Partial sums of squares per row that a folded-norm producer of width N writes (one per
// half N-tile).
int gemm_tc_norm_parts(int N);
// Tensor-core attention (attn_tc.cu): head_dim 64 or 128, bf16.
bool tc_attn_supported(int head_dim);
// q: per kv head a slab [m_cap][group][head_dim]; rows of request r are
// req_row_end[r-1]..req_row_end[r]-1 (device); caches: this layer's [n_tokens][hkv][head_dim].
int launch_attn_tc(const void* q, int m_cap, int n_req, const int32_t* req_row_end, const int32_t* row_pos,
                   const int32_t* row_tok, int M_max, const void* k_cache, const void* v_cache, long long n_tokens,
                   void* o, int hq, int hkv, int head_dim, int32_t* err, cudaStream_t s);
}  // namespace blend
