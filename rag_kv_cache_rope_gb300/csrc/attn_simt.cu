// CUDA-core causal GQA attention of selected query rows over the full blended KV
// (the fp32 model path and a GPU-side cross-check of the tensor-core kernel).
//
// One CTA per (row, kv head); one warp per query head of the group, so each K/V
// tile is loaded once for the whole group.  Keys are processed 32 at a time: lane j
// scores key j, the tile's softmax update is done with warp shuffles (online softmax
// in base 2), and lane l accumulates output dims l, l+32, ...
#include <math.h>

#include "common.cuh"

namespace blend {

template <typename T>
__global__ void k_attn_simt(const T* __restrict__ q, int m_cap, const int32_t* __restrict__ row_pos,
                            const int32_t* __restrict__ row_tok, const int32_t* M_dev,
                            const T* __restrict__ Kc, const T* __restrict__ Vc, T* __restrict__ o,
                            int hq, int hkv, int d, float scale_log2) {
    extern __shared__ float sm[];
    const int row = blockIdx.x;
    if (row >= *M_dev) return;
    const int g = blockIdx.y;
    const int group = hq / hkv;
    const int pos = row_pos[row];
    const long long base = (long long)row_tok[row] - pos;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h = g * group + warp;
    float* Ks = sm;                 // [32][d+1]
    float* Vs = Ks + 32 * (d + 1);  // [32][d]
    float* qs = Vs + 32 * d;        // [group][d]
    const T* qr = q + ((long long)g * m_cap + row) * group * d;
    for (int e = threadIdx.x; e < group * d; e += blockDim.x) qs[e] = to_f<T>(qr[e]);
    const int nd = d / 32;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float m = -INFINITY, l = 0.f;
    const long long kstride = (long long)hkv * d;
    for (int k0 = 0; k0 <= pos; k0 += 32) {
        __syncthreads();
        for (int e = threadIdx.x; e < 32 * d; e += blockDim.x) {
            const int j = e / d, c = e % d;
            const int key = k0 + j;
            float kv = 0.f, vv = 0.f;
            if (key <= pos) {
                const long long a = (base + key) * kstride + (long long)g * d + c;
                kv = to_f<T>(Kc[a]);
                vv = to_f<T>(Vc[a]);
            }
            Ks[j * (d + 1) + c] = kv;
            Vs[j * d + c] = vv;
        }
        __syncthreads();
        const int key = k0 + lane;
        float s = -INFINITY;
        if (key <= pos) {
            float dot = 0.f;
            const float* kr = Ks + lane * (d + 1);
            const float* qh = qs + warp * d;
            for (int c = 0; c < d; ++c) dot = fmaf(qh[c], kr[c], dot);
            s = dot * scale_log2;
        }
        float mt = s;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
        const float m_new = fmaxf(m, mt);
        const float corr = exp2f(m - m_new);
        const float p = key <= pos ? exp2f(s - m_new) : 0.f;
        float ps = p;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        l = l * corr + ps;
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] *= corr;
        const int nk = min(32, pos - k0 + 1);
        for (int j = 0; j < nk; ++j) {
            const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (u < nd) acc[u] = fmaf(pj, Vs[j * d + lane + 32 * u], acc[u]);
        }
        m = m_new;
    }
    T* orow = o + (long long)row * hq * d + (long long)h * d;
    const float inv = 1.f / l;
#pragma unroll
    for (int u = 0; u < 4; ++u)
        if (u < nd) orow[lane + 32 * u] = from_f<T>(acc[u] * inv);
}

void launch_attn_simt(int dtype, const void* q, int m_cap, const int32_t* row_pos, const int32_t* row_tok,
                      const int32_t* M_dev, int M_max, const void* k_cache, const void* v_cache,
                      void* o, int hq, int hkv, int d, cudaStream_t s) {
    if (M_max <= 0) return;
    const int group = hq / hkv;
    dim3 grid(M_max, hkv);
    const size_t smem = (size_t)(32 * (d + 1) + 32 * d + group * d) * sizeof(float);
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)d));
    if (dtype == BLEND_BF16) {
        cudaFuncSetAttribute(k_attn_simt<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        k_attn_simt<bf16><<<grid, 32 * group, smem, s>>>((const bf16*)q, m_cap, row_pos, row_tok, M_dev,
                                                         (const bf16*)k_cache, (const bf16*)v_cache,
                                                         (bf16*)o, hq, hkv, d, scale_log2);
    } else {
        cudaFuncSetAttribute(k_attn_simt<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        k_attn_simt<float><<<grid, 32 * group, smem, s>>>((const float*)q, m_cap, row_pos, row_tok, M_dev,
                                                          (const float*)k_cache,
                                                          (const float*)v_cache, (float*)o, hq, hkv,
                                                          d, scale_log2);
    }
    note_launch(1);
}

}  // namespace blend
