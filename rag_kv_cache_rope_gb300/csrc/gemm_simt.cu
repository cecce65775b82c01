// CUDA-core GEMM C = A . B^T for the fp32 model path (and as a GPU-side cross-check of
// the tensor-core path).  A [M][K] and B [N][K] are K-contiguous in the model dtype;
// accumulation is fp32.  64x64 output tile per CTA, 256 threads with 4x4 outputs each,
// K staged through shared memory 16 at a time.  M is read from the device so the grid
// can be sized for the largest possible row count.
#include "common.cuh"

namespace blend {

constexpr int GT = 64;  // tile M and N
constexpr int GK = 16;  // tile K

template <typename T, int EPI>
__global__ void __launch_bounds__(256)
    k_gemm_simt(const T* __restrict__ A, int lda, const T* __restrict__ B, int ldb, int K, int N,
                const int32_t* M_dev, void* __restrict__ Cv, int ldc) {
    __shared__ float As[GK][GT + 4];
    __shared__ float Bs[GK][GT + 4];
    __shared__ float Cs[GT][GT + 1];
    const int M = *M_dev;
    const int m0 = blockIdx.y * GT, n0 = blockIdx.x * GT;
    if (m0 >= M) return;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += GK) {
        // 64 rows x 16 k of A and of B: 1024 elements each, 4 per thread
        for (int e = threadIdx.x; e < GT * GK; e += 256) {
            int r = e / GK, c = e % GK;
            int gm = m0 + r, gn = n0 + r, gk = k0 + c;
            As[c][r] = (gm < M && gk < K) ? to_f<T>(A[(long long)gm * lda + gk]) : 0.f;
            Bs[c][r] = (gn < N && gk < K) ? to_f<T>(B[(long long)gn * ldb + gk]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < GK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = As[kk][ty * 4 + i];
                b[i] = Bs[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    if (EPI == EPI_STORE_F32 || EPI == EPI_ADD_F32) {
        float* C = (float*)Cv;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int gm = m0 + ty * 4 + i;
            if (gm >= M) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                int gn = n0 + tx * 4 + j;
                if (gn >= N) continue;
                float* p = C + (long long)gm * ldc + gn;
                if (EPI == EPI_ADD_F32) *p += acc[i][j];
                else *p = acc[i][j];
            }
        }
    } else {
        // gate/up interleaved in blocks of BLEND_GU_BLOCK: within each 32-column group
        // columns 0..15 are gate, 16..31 up of the same 16 hidden units
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) Cs[ty * 4 + i][tx * 4 + j] = acc[i][j];
        __syncthreads();
        T* C = (T*)Cv;
        constexpr int GB = BLEND_GU_BLOCK;
        for (int e = threadIdx.x; e < GT * (GT / 2); e += 256) {
            int r = e / (GT / 2), c = e % (GT / 2);   // output column within the tile
            int grp = c / GB, within = c % GB;
            int cg = grp * 2 * GB + within;           // gate column in the tile
            int gm = m0 + r, gcol = n0 + cg;
            if (gm >= M || gcol >= N) continue;
            float g = Cs[r][cg], u = Cs[r][cg + GB];
            float silu = g / (1.f + expf(-g));
            C[(long long)gm * ldc + n0 / 2 + c] = from_f<T>(silu * u);
        }
    }
}

void launch_gemm_simt(int dtype, const void* A, int lda, const void* B, int ldb, int K, int N,
                      const int32_t* M_dev, int M_max, int epi, void* C, int ldc, cudaStream_t s) {
    if (M_max <= 0 || N <= 0) return;
    dim3 grid((N + GT - 1) / GT, (M_max + GT - 1) / GT);
#define GEMM_CASE(T, E)                                                                         \
    k_gemm_simt<T, E><<<grid, 256, 0, s>>>((const T*)A, lda, (const T*)B, ldb, K, N, M_dev, C, ldc)
    if (dtype == BLEND_BF16) {
        if (epi == EPI_STORE_F32) GEMM_CASE(bf16, EPI_STORE_F32);
        else if (epi == EPI_ADD_F32) GEMM_CASE(bf16, EPI_ADD_F32);
        else GEMM_CASE(bf16, EPI_SWIGLU);
    } else {
        if (epi == EPI_STORE_F32) GEMM_CASE(float, EPI_STORE_F32);
        else if (epi == EPI_ADD_F32) GEMM_CASE(float, EPI_ADD_F32);
        else GEMM_CASE(float, EPI_SWIGLU);
    }
#undef GEMM_CASE
    note_launch(1);
}

}  // namespace blend
