// HBM-bound kernels of blended prefill: RoPE table, key realignment and cache
// assembly, fused RoPE + deviation + K/V scatter, RMSNorm, row gather, row plans.
//
// Rows are streamed with 16-byte vector accesses so a warp touches contiguous
// 512-byte spans; reductions run in a fixed order (no floating-point atomics) so
// results are bitwise reproducible run to run.
#include "common.cuh"

namespace blend {

// ---------------------------------------------------------------- RoPE table
// tab[p][i] = (cos a, sin a) with a = p * theta^(-2i/d), evaluated in fp64 and rounded
// to fp32 (an fp32 angle would be off by ~1e-3 rad at position 32K).
__global__ void k_rope_table(float2* tab, int max_pos, int half, double theta, int d) {
    long long total = (long long)max_pos * half;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        int p = (int)(idx / half);
        int i = (int)(idx % half);
        double inv = pow(theta, -2.0 * (double)i / (double)d);
        double a = (double)p * inv;
        double s, c;
        sincos(a, &s, &c);
        tab[idx] = make_float2((float)c, (float)s);
    }
}

void launch_rope_table(float2* tab, int max_pos, int head_dim, double theta, cudaStream_t s) {
    int half = head_dim / 2;
    long long total = (long long)max_pos * half;
    long long blocks = (total + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    k_rope_table<<<(int)blocks, 256, 0, s>>>(tab, max_pos, half, theta, head_dim);
    note_launch(1);
}

// Rotates the pair vectors (row[i0..i0+V), row[i0+d/2..i0+d/2+V)) by `delta` positions:
// (x1, x2) -> (x1 cos - x2 sin, x2 cos + x1 sin); a negative delta flips sin.
template <typename T>
__device__ __forceinline__ void rotate_pair(const T* src, T* dst, int i0, int half, int delta,
                                            const float2* tab) {
    Vec<T> a = ld16(src + i0);
    Vec<T> b = ld16(src + i0 + half);
    const int ad = delta < 0 ? -delta : delta;
    const float sg = delta < 0 ? -1.f : 1.f;
    const float2* cs = tab + (long long)ad * half + i0;
    Vec<T> oa, ob;
#pragma unroll
    for (int e = 0; e < Vec<T>::N; ++e) {
        float2 t = cs[e];
        float c = t.x, s = sg * t.y;
        float x1 = a.get(e), x2 = b.get(e);
        oa.set(e, x1 * c - x2 * s);
        ob.set(e, x2 * c + x1 * s);
    }
    st16(dst + i0, oa);
    st16(dst + i0 + half, ob);
}

// ---------------------------------------------------------------- realign (per-row shift)
template <typename T>
__global__ void k_realign(const T* src, T* dst, int n_rows, const int32_t* delta, long long src_lr,
                          long long dst_lr, int hkv, int d, const float2* tab, int max_pos,
                          int32_t* err) {
    const int layer = blockIdx.y;
    const int row = blockIdx.x;
    if (row >= n_rows) return;
    const int dl = delta[row];
    if (dl <= -max_pos || dl >= max_pos) {
        set_error(err, BLEND_EINVAL);
        return;
    }
    const int half = d / 2;
    const int VN = Vec<T>::N;
    const int per_head = half / VN;
    const long long re = (long long)hkv * d;
    const T* s = src + ((long long)layer * src_lr + row) * re;
    T* o = dst + ((long long)layer * dst_lr + row) * re;
    for (int j = threadIdx.x; j < hkv * per_head; j += blockDim.x) {
        int g = j / per_head, i0 = (j % per_head) * VN;
        rotate_pair(s + g * d, o + g * d, i0, half, dl, tab);
    }
}

void launch_realign(int dtype, const void* src, void* dst, int n_rows, const int32_t* delta,
                    int n_layers, long long src_lr, long long dst_lr, int hkv, int d,
                    const float2* tab, int max_pos, int32_t* err, cudaStream_t s) {
    if (n_rows <= 0 || n_layers <= 0) return;
    dim3 grid(n_rows, n_layers);
    if (dtype == BLEND_BF16)
        k_realign<bf16><<<grid, 128, 0, s>>>((const bf16*)src, (bf16*)dst, n_rows, delta, src_lr,
                                             dst_lr, hkv, d, tab, max_pos, err);
    else
        k_realign<float><<<grid, 128, 0, s>>>((const float*)src, (float*)dst, n_rows, delta,
                                              src_lr, dst_lr, hkv, d, tab, max_pos, err);
    note_launch(1);
}

// ---------------------------------------------------------------- assemble
// Concatenation + prefix drop + key realignment for layers layer0.. of a batch.  The
// segment table lists, in order, the prefix rows of each request (shift 0) and each
// chunk's rows (shift = offset of the chunk among the request's chunks).  One CTA
// handles ASM_ROWS consecutive rows of one layer (layer0 + blockIdx.y).  The pool may
// sit in pinned host memory that the GPU reads directly (on Grace-Blackwell over the
// NVLink chip-to-chip link): the kernel only streams it.
constexpr int ASM_ROWS = 8;

template <typename T>
__global__ void __launch_bounds__(256)
    k_assemble(const __grid_constant__ SegTable segs, const T* __restrict__ pk,
               const T* __restrict__ pv, long long pool_rows, T* __restrict__ ok,
               T* __restrict__ ov, long long out_tokens, int hkv, int d,
               const float2* __restrict__ tab, int max_pos, int32_t* err, int layer0) {
    const int layer = layer0 + blockIdx.y;
    const int half = d / 2;
    const int VN = Vec<T>::N;
    const int per_head = half / VN;
    const int nk = hkv * per_head;  // K pair items per row
    const int nv = hkv * d / VN;    // V vector items per row
    const long long re = (long long)hkv * d;
    for (int rr = 0; rr < ASM_ROWS; ++rr) {
        const int r = blockIdx.x * ASM_ROWS + rr;
        if (r >= segs.total_rows) return;
        int lo = 0, hi = segs.n_seg - 1;  // last segment with row0 <= r
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (segs.s[mid].row0 <= r) lo = mid;
            else hi = mid - 1;
        }
        const Seg sg = segs.s[lo];
        const int k = r - sg.row0;
        const long long srow = (long long)sg.src_row + k;
        const long long drow = (long long)sg.dst_tok + k;
        const int dl = sg.delta;
        if (dl < 0 || dl >= max_pos || srow >= pool_rows || drow >= out_tokens) {
            set_error(err, BLEND_EINVAL);
            continue;
        }
        const T* sk = pk + ((long long)layer * pool_rows + srow) * re;
        const T* sv = pv + ((long long)layer * pool_rows + srow) * re;
        T* dk = ok + ((long long)layer * out_tokens + drow) * re;
        T* dv = ov + ((long long)layer * out_tokens + drow) * re;
        for (int j = threadIdx.x; j < nk + nv; j += blockDim.x) {
            if (j < nk) {
                int g = j / per_head, i0 = (j % per_head) * VN;
                rotate_pair(sk + g * d, dk + g * d, i0, half, dl, tab);
            } else {
                int e = (j - nk) * VN;
                st16(dv + e, ld16(sv + e));
            }
        }
    }
}

void launch_assemble(int dtype, const SegTable& segs, const void* pool_k, const void* pool_v,
                     long long pool_rows, void* out_k, void* out_v, long long out_tokens,
                     int n_layers, int hkv, int d, const float2* tab, int max_pos, int32_t* err,
                     cudaStream_t s, int layer0) {
    if (segs.total_rows <= 0 || n_layers <= 0) return;
    dim3 grid((segs.total_rows + ASM_ROWS - 1) / ASM_ROWS, n_layers);
    const int items = hkv * (d / 2) / (16 / (dtype == BLEND_BF16 ? 2 : 4)) +
                      hkv * d / (16 / (dtype == BLEND_BF16 ? 2 : 4));
    int threads = items >= 256 ? 256 : ((items + 31) / 32) * 32;
    if (dtype == BLEND_BF16)
        k_assemble<bf16><<<grid, threads, 0, s>>>(segs, (const bf16*)pool_k, (const bf16*)pool_v,
                                                  pool_rows, (bf16*)out_k, (bf16*)out_v,
                                                  out_tokens, hkv, d, tab, max_pos, err, layer0);
    else
        k_assemble<float><<<grid, threads, 0, s>>>(segs, (const float*)pool_k,
                                                   (const float*)pool_v, pool_rows, (float*)out_k,
                                                   (float*)out_v, out_tokens, hkv, d, tab, max_pos,
                                                   err, layer0);
    note_launch(1);
}

// EPIC's static selection: the first m tokens of every chunk, written run by run.
__global__ void k_epic_set(const __grid_constant__ EpicTable et, int32_t* __restrict__ set,
                           int32_t* __restrict__ set_n) {
    const int q = blockIdx.x;
    if (q < et.n_run)
        for (int t = threadIdx.x; t < et.count[q]; t += blockDim.x) set[et.out[q] + t] = et.start[q] + t;
    if (q == 0)
        for (int r = threadIdx.x; r < et.n_req; r += blockDim.x) set_n[r] = et.req_n[r];
}

void launch_epic_set(const EpicTable& et, int32_t* set, int32_t* set_n, cudaStream_t s) {
    k_epic_set<<<et.n_run > 0 ? et.n_run : 1, 128, 0, s>>>(et, set, set_n);
    note_launch(1);
}

// Bounded wait on a caller's device flag: one thread polls until *flag != 0, at most
// max_polls times with a short sleep between polls; if the flag never changes the error
// word gets BLEND_ETIMEOUT and the kernel returns (no trap, the context stays usable).
__global__ void k_wait_flag(const int32_t* flag, long long max_polls, int32_t* err) {
    if (threadIdx.x != 0) return;
    const volatile int32_t* f = flag;
    for (long long i = 0; i < max_polls; ++i) {
        if (*f != 0) return;
        __nanosleep(64);
    }
    set_error(err, BLEND_ETIMEOUT);
}

void launch_wait_flag(const int32_t* flag, long long max_polls, int32_t* err, cudaStream_t s) {
    k_wait_flag<<<1, 32, 0, s>>>(flag, max_polls, err);
    note_launch(1);
}

// Token id of every blended token: prefix and chunk rows from the pool, query rows
// from each request's query tokens.
__global__ void k_tokens(const __grid_constant__ SegTable segs,
                         const __grid_constant__ QueryTable qt, const int32_t* pool_tokens,
                         int32_t* out) {
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < segs.total_rows;
         r += gridDim.x * blockDim.x) {
        int lo = 0, hi = segs.n_seg - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (segs.s[mid].row0 <= r) lo = mid;
            else hi = mid - 1;
        }
        const Seg sg = segs.s[lo];
        const int k = r - sg.row0;
        out[sg.dst_tok + k] = pool_tokens[sg.src_row + k];
    }
    for (int q = 0; q < qt.n; ++q)
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < qt.len[q];
             i += gridDim.x * blockDim.x)
            out[qt.dst_tok[q] + i] = qt.ptr[q][i];
}

void launch_tokens(const SegTable& segs, const QueryTable& qt, const int32_t* pool_tokens,
                   int32_t* out_tokens, cudaStream_t s) {
    int blocks = (segs.total_rows + 255) / 256;
    if (blocks < 1) blocks = 1;
    if (blocks > 1024) blocks = 1024;
    k_tokens<<<blocks, 256, 0, s>>>(segs, qt, pool_tokens, out_tokens);
    note_launch(1);
}

// ---------------------------------------------------------------- RMSNorm
// out[row] = x[row] / sqrt(mean(x^2) + eps) * g, x fp32, out in the model dtype.  One
// CTA per row; the row stays in registers (float4, up to RMS_V per thread) between the
// sum of squares and the scaling, so x is read once.  The block sum is a fixed-order
// shuffle tree plus a fixed-order sum of the warp partials (bitwise reproducible).
constexpr int RMS_THREADS = 256;
constexpr int RMS_V = 8;  // H <= 4 * RMS_V * RMS_THREADS = 8192

__device__ __forceinline__ float block_sum_fast(float v, float* warp_part) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x / 32;
    if ((threadIdx.x & 31) == 0) warp_part[w] = v;
    __syncthreads();
    float r = 0.f;
    for (int i = 0; i < (int)(blockDim.x / 32); ++i) r += warp_part[i];
    return r;
}

template <typename T>
__device__ __forceinline__ void store4(T* p, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<float>(float* p, float a, float b, float c, float d) {
    *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
template <>
__device__ __forceinline__ void store4<bf16>(bf16* p, float a, float b, float c, float d) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
}

template <typename T>
__global__ void __launch_bounds__(RMS_THREADS)
    k_rmsnorm(const float* __restrict__ x, const T* __restrict__ g, T* __restrict__ out, int H, float eps,
              const int32_t* M_dev) {
    __shared__ float part[RMS_THREADS / 32];
    const int row = blockIdx.x;
    if (row >= *M_dev) return;
    const float4* xr = reinterpret_cast<const float4*>(x + (long long)row * H);
    const int nv = H / 4;
    float4 v[RMS_V];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < RMS_V; ++k) {
        const int i = threadIdx.x + k * RMS_THREADS;
        v[k] = i < nv ? xr[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
    }
    ss = block_sum_fast(ss, part);
    const float r = rsqrtf(ss / (float)H + eps);
    T* o = out + (long long)row * H;
#pragma unroll
    for (int k = 0; k < RMS_V; ++k) {
        const int i = threadIdx.x + k * RMS_THREADS;
        if (i < nv) {
            const int c = 4 * i;
            store4<T>(o + c, v[k].x * r * to_f<T>(g[c]), v[k].y * r * to_f<T>(g[c + 1]),
                      v[k].z * r * to_f<T>(g[c + 2]), v[k].w * r * to_f<T>(g[c + 3]));
        }
    }
}

void launch_rmsnorm(int dtype, const float* x, const void* g, void* out, int H, float eps,
                    const int32_t* M_dev, int M_max, cudaStream_t s) {
    if (M_max <= 0) return;
    if (dtype == BLEND_BF16)
        k_rmsnorm<bf16><<<M_max, RMS_THREADS, 0, s>>>(x, (const bf16*)g, (bf16*)out, H, eps, M_dev);
    else
        k_rmsnorm<float><<<M_max, RMS_THREADS, 0, s>>>(x, (const float*)g, (float*)out, H, eps, M_dev);
    note_launch(1);
}

// Final norm of every request's query rows (the last Q rows of its block of rows).
template <typename T>
__global__ void __launch_bounds__(256)
    k_final_norm(const float* __restrict__ x, const T* __restrict__ g, T* __restrict__ hidden,
                 int H, float eps, const __grid_constant__ BatchDesc bd, const int32_t* req_row_end) {
    __shared__ float red[256];
    const int r = blockIdx.y;
    const int j = blockIdx.x;
    if (j >= bd.r[r].Q) return;
    const long long row = (long long)req_row_end[r] - bd.r[r].Q + j;
    const float* xr = x + row * H;
    float ss = 0.f;
    for (int c = threadIdx.x; c < H; c += blockDim.x) {
        float v = xr[c];
        ss += v * v;
    }
    ss = block_sum(ss, red);
    const float rr = rsqrtf(ss / (float)H + eps);
    T* o = hidden + ((long long)bd.r[r].q_off + j) * H;
    for (int c = threadIdx.x; c < H; c += blockDim.x) o[c] = from_f<T>(xr[c] * rr * to_f<T>(g[c]));
}

void launch_final_norm(int dtype, const float* x, const void* g, void* hidden, int H, float eps,
                       const BatchDesc& bd, const int32_t* req_row_end, cudaStream_t s) {
    int maxq = 0;
    for (int r = 0; r < bd.n_req; ++r) maxq = bd.r[r].Q > maxq ? bd.r[r].Q : maxq;
    if (maxq == 0) return;
    dim3 grid(maxq, bd.n_req);
    if (dtype == BLEND_BF16)
        k_final_norm<bf16><<<grid, 256, 0, s>>>(x, (const bf16*)g, (bf16*)hidden, H, eps, bd,
                                                req_row_end);
    else
        k_final_norm<float><<<grid, 256, 0, s>>>(x, (const float*)g, (float*)hidden, H, eps, bd,
                                                 req_row_end);
    note_launch(1);
}

// ---------------------------------------------------------------- embeddings, gather
template <typename T>
__global__ void k_embed(const T* __restrict__ embed, const int32_t* __restrict__ tokens,
                        const int32_t* __restrict__ row_tok, float* __restrict__ x, int H, int vocab,
                        const int32_t* M_dev, int32_t* err) {
    const int row = blockIdx.x;
    if (row >= *M_dev) return;
    long long tok = tokens[row_tok[row]];
    if (tok < 0 || tok >= vocab) {  // token id outside the vocabulary: reported, row 0 used
        if (threadIdx.x == 0) set_error(err, BLEND_EDEVICE);
        tok = 0;
    }
    const T* e = embed + tok * H;
    float* o = x + (long long)row * H;
    for (int j = threadIdx.x; j < H; j += blockDim.x) o[j] = to_f<T>(e[j]);
}

void launch_embed(int dtype, const void* embed, const int32_t* tokens, const int32_t* row_tok,
                  float* x, int H, int vocab, const int32_t* M_dev, int M_max, int32_t* err,
                  cudaStream_t s) {
    if (M_max <= 0) return;
    if (dtype == BLEND_BF16)
        k_embed<bf16><<<M_max, 256, 0, s>>>((const bf16*)embed, tokens, row_tok, x, H, vocab, M_dev, err);
    else
        k_embed<float><<<M_max, 256, 0, s>>>((const float*)embed, tokens, row_tok, x, H, vocab, M_dev, err);
    note_launch(1);
}

// dst[i] = src[idx[i]], rows of row_bytes (multiple of 16).  An index outside
// 0..src_rows-1 is reported in err and its destination row is left untouched; a count
// above max_n is reported and clamped (the grid has max_n blocks).
__global__ void k_gather(const uint4* __restrict__ src, long long row_vec, long long src_rows,
                         const int32_t* __restrict__ idx, const int32_t* n_dev, int max_n,
                         uint4* __restrict__ dst, int32_t* err) {
    const int i = blockIdx.x;
    const int n = *n_dev;
    if (i == 0 && threadIdx.x == 0 && (n < 0 || n > max_n)) set_error(err, BLEND_EDEVICE);
    if (i >= n) return;
    const long long r = idx[i];
    if (r < 0 || r >= src_rows) {
        if (threadIdx.x == 0) set_error(err, BLEND_EDEVICE);
        return;
    }
    const long long s = r * row_vec;
    const long long d = (long long)i * row_vec;
    for (long long j = threadIdx.x; j < row_vec; j += blockDim.x) dst[d + j] = src[s + j];
}

void launch_gather(const void* src, long long row_bytes, long long src_rows, const int32_t* idx,
                   const int32_t* n_dev, int max_n, void* dst, int32_t* err, cudaStream_t s) {
    if (max_n <= 0) return;
    long long rv = row_bytes / 16;
    int threads = rv >= 256 ? 256 : (int)(((rv + 31) / 32) * 32);
    k_gather<<<max_n, threads, 0, s>>>((const uint4*)src, rv, src_rows, idx, n_dev, max_n, (uint4*)dst, err);
    note_launch(1);
}

// Two consecutive elements of T (8 bytes of fp32 or 4 of bf16) as floats, and back.
template <typename T> __device__ __forceinline__ float2 load2(const T* p);
template <> __device__ __forceinline__ float2 load2<float>(const float* p) { return *reinterpret_cast<const float2*>(p); }
template <> __device__ __forceinline__ float2 load2<bf16>(const bf16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
template <typename T> __device__ __forceinline__ void store2(T* p, float a, float b);
template <> __device__ __forceinline__ void store2<float>(float* p, float a, float b) {
    *reinterpret_cast<float2*>(p) = make_float2(a, b);
}
template <> __device__ __forceinline__ void store2<bf16>(bf16* p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}

// ---------------------------------------------------------------- fused RoPE + deviation + scatter
// For each recomputed row (one CTA per row): rotate q and k at the row's blended
// position, store q for attention, compare the fresh k, v (fp32, before rounding) with
// the cached rows at that position (deviation, optional), then overwrite the cache rows.
template <typename T>
__global__ void __launch_bounds__(256)
    k_rope_qkv(const float* __restrict__ qkv, const int32_t* __restrict__ row_pos,
               const int32_t* __restrict__ row_tok, const int32_t* __restrict__ row_req,
               const int32_t* M_dev, const __grid_constant__ BatchDesc bd, int hq, int hkv, int d,
               int m_cap, const float2* __restrict__ tab, T* __restrict__ q_out, T* __restrict__ kc,
               T* __restrict__ vc, float* __restrict__ dev_out, int dev_mode, int dev_by_row) {
    __shared__ float red[256];
    const int row = blockIdx.x;
    if (row >= *M_dev) return;
    const int pos = row_pos[row];
    const long long tok = row_tok[row];
    const int half = d / 2;
    const int width = (hq + 2 * hkv) * d;
    const float* src = qkv + (long long)row * width;
    const float2* cs = tab + (long long)pos * half;
    // q layout: per kv head g a slab of [m_cap rows][group][d] (pair = row * group + j).
    // Each thread takes two neighbouring rotate-half pairs (i, i+1) and (i+d/2, i+1+d/2):
    // 8-byte loads of the fp32 projection, one 16-byte (cos, sin) load, paired stores.
    const int group = hq / hkv;
    const int hp = half / 2;  // pairs of pairs per head
    for (int j = threadIdx.x; j < hq * hp; j += blockDim.x) {
        const int h = j / hp, i = 2 * (j % hp);
        const float2 a = *reinterpret_cast<const float2*>(src + h * d + i);
        const float2 b = *reinterpret_cast<const float2*>(src + h * d + i + half);
        const float4 t = *reinterpret_cast<const float4*>(cs + i);  // (cos, sin) of i and i+1
        T* qo = q_out + (((long long)(h / group) * m_cap + row) * group + (h % group)) * d;
        store2<T>(qo + i, a.x * t.x - b.x * t.y, a.y * t.z - b.y * t.w);
        store2<T>(qo + i + half, b.x * t.x + a.x * t.y, b.y * t.z + a.y * t.w);
    }
    float acc = 0.f;
    const float* ks = src + hq * d;
    T* kr = kc + tok * hkv * d;
    for (int j = threadIdx.x; j < hkv * hp; j += blockDim.x) {
        const int g = j / hp, i = 2 * (j % hp);
        const float2 a = *reinterpret_cast<const float2*>(ks + g * d + i);
        const float2 b = *reinterpret_cast<const float2*>(ks + g * d + i + half);
        const float4 t = *reinterpret_cast<const float4*>(cs + i);
        const float r1a = a.x * t.x - b.x * t.y, r1b = a.y * t.z - b.y * t.w;
        const float r2a = b.x * t.x + a.x * t.y, r2b = b.y * t.z + a.y * t.w;
        if (dev_out && dev_mode == BLEND_DEV_KV) {
            const float2 c1 = load2<T>(kr + g * d + i), c2 = load2<T>(kr + g * d + i + half);
            const float o1 = c1.x - r1a, o2 = c1.y - r1b, o3 = c2.x - r2a, o4 = c2.y - r2b;
            acc += o1 * o1 + o2 * o2 + o3 * o3 + o4 * o4;
        }
        store2<T>(kr + g * d + i, r1a, r1b);
        store2<T>(kr + g * d + i + half, r2a, r2b);
    }
    const float* vs = src + (hq + hkv) * d;
    T* vr = vc + tok * hkv * d;
    for (int j = threadIdx.x; j < hkv * d / 2; j += blockDim.x) {
        const float2 v = *reinterpret_cast<const float2*>(vs + 2 * j);
        if (dev_out) {
            const float2 c = load2<T>(vr + 2 * j);
            const float o1 = c.x - v.x, o2 = c.y - v.y;
            acc += o1 * o1 + o2 * o2;
        }
        store2<T>(vr + 2 * j, v.x, v.y);
    }
    if (dev_out) {
        float dv = block_sum(acc, red);
        const ReqDesc rd = bd.r[row_req[row]];
        if (threadIdx.x == 0) {
            if (dev_by_row) dev_out[row] = dv;
            else if (pos >= rd.P && pos < rd.P + rd.n_c) dev_out[rd.nc_off + pos - rd.P] = dv;
        }
    }
}

void launch_rope_qkv(int dtype, const float* qkv, const int32_t* row_pos, const int32_t* row_tok,
                     const int32_t* row_req, const int32_t* M_dev, int M_max, const BatchDesc& bd,
                     int hq, int hkv, int d, int m_cap, const float2* tab, void* q_out, void* k_cache,
                     void* v_cache, float* dev_out, int dev_mode, int dev_by_row, cudaStream_t s) {
    if (M_max <= 0) return;
    if (dtype == BLEND_BF16)
        k_rope_qkv<bf16><<<M_max, 256, 0, s>>>(qkv, row_pos, row_tok, row_req, M_dev, bd, hq, hkv,
                                               d, m_cap, tab, (bf16*)q_out, (bf16*)k_cache,
                                               (bf16*)v_cache, dev_out, dev_mode, dev_by_row);
    else
        k_rope_qkv<float><<<M_max, 256, 0, s>>>(qkv, row_pos, row_tok, row_req, M_dev, bd, hq, hkv,
                                                d, m_cap, tab, (float*)q_out, (float*)k_cache,
                                                (float*)v_cache, dev_out, dev_mode, dev_by_row);
    note_launch(1);
}

// ---------------------------------------------------------------- standalone deviation / scatter
// One warp per row, 16-byte loads of the fresh and the cached rows; each lane adds its
// vectors in order and the lanes are combined by a fixed shuffle tree, so the result
// does not depend on timing.  A position outside 0..n_ctx-1 is reported in err and
// gives dev = 0 without touching the cache; a count above max_rows is reported and
// clamped.
constexpr int DEV_WARPS = 8;
template <typename T>
__global__ void __launch_bounds__(DEV_WARPS * 32)
    k_deviation(const T* __restrict__ kn, const T* __restrict__ vn, const T* __restrict__ kc,
                const T* __restrict__ vc, const int32_t* __restrict__ pos, const int32_t* n_dev,
                int max_rows, long long n_ctx, int kv_elems, int mode, float* __restrict__ dev,
                int32_t* err) {
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * DEV_WARPS + (threadIdx.x >> 5);
    int n = *n_dev;
    if (blockIdx.x == 0 && threadIdx.x == 0 && (n < 0 || n > max_rows)) set_error(err, BLEND_EDEVICE);
    n = min(n, max_rows);
    if (i >= n) return;
    const long long p = pos[i];
    if (p < 0 || p >= n_ctx) {
        if (lane == 0) {
            set_error(err, BLEND_EDEVICE);
            dev[i] = 0.f;
        }
        return;
    }
    constexpr int E = Vec<T>::N;
    const long long a = (long long)i * kv_elems, b = p * kv_elems;
    float acc = 0.f;
    for (int j = lane * E; j < kv_elems; j += 32 * E) {
        const Vec<T> x = ld16(vn + a + j), y = ld16(vc + b + j);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float dv = x.get(e) - y.get(e);
            acc = fmaf(dv, dv, acc);
        }
        if (mode == BLEND_DEV_KV) {
            const Vec<T> xk = ld16(kn + a + j), yk = ld16(kc + b + j);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float dk = xk.get(e) - yk.get(e);
                acc = fmaf(dk, dk, acc);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) dev[i] = acc;
}

void launch_deviation(int dtype, const void* k_new, const void* v_new, const void* k_cache,
                      const void* v_cache, const int32_t* pos, const int32_t* n_dev, int max_rows,
                      long long n_ctx, int kv_elems, int mode, float* dev_out, int32_t* err, cudaStream_t s) {
    if (max_rows <= 0) return;
    const int grid = (max_rows + DEV_WARPS - 1) / DEV_WARPS;
    if (dtype == BLEND_BF16)
        k_deviation<bf16><<<grid, DEV_WARPS * 32, 0, s>>>((const bf16*)k_new, (const bf16*)v_new,
                                                          (const bf16*)k_cache, (const bf16*)v_cache, pos,
                                                          n_dev, max_rows, n_ctx, kv_elems, mode, dev_out, err);
    else
        k_deviation<float><<<grid, DEV_WARPS * 32, 0, s>>>((const float*)k_new, (const float*)v_new,
                                                           (const float*)k_cache, (const float*)v_cache,
                                                           pos, n_dev, max_rows, n_ctx, kv_elems, mode, dev_out,
                                                           err);
    note_launch(1);
}

// k_cache[pos[i]] = k_new[i], v_cache[pos[i]] = v_new[i] in 16-byte vectors; a position
// outside 0..n_ctx-1 is reported in err and that row is not written; a count above
// max_n is reported and clamped.
__global__ void k_scatter(const uint4* __restrict__ kn, const uint4* __restrict__ vn,
                          const int32_t* __restrict__ pos, const int32_t* n_dev, int max_n, long long n_ctx,
                          long long row_vec, uint4* __restrict__ kc, uint4* __restrict__ vc, int32_t* err) {
    const int i = blockIdx.x;
    const int n = *n_dev;
    if (i == 0 && threadIdx.x == 0 && (n < 0 || n > max_n)) set_error(err, BLEND_EDEVICE);
    if (i >= n) return;
    const long long p = pos[i];
    if (p < 0 || p >= n_ctx) {
        if (threadIdx.x == 0) set_error(err, BLEND_EDEVICE);
        return;
    }
    const long long a = (long long)i * row_vec, b = p * row_vec;
    for (long long j = threadIdx.x; j < row_vec; j += blockDim.x) {
        kc[b + j] = kn[a + j];
        vc[b + j] = vn[a + j];
    }
}

void launch_scatter(int dtype, const void* k_new, const void* v_new, const int32_t* pos,
                    const int32_t* n_dev, int max_n, long long n_ctx, int kv_elems, void* k_cache,
                    void* v_cache, int32_t* err, cudaStream_t s) {
    if (max_n <= 0) return;
    long long rv = (long long)kv_elems * (dtype == BLEND_BF16 ? 2 : 4) / 16;
    int threads = rv >= 128 ? 128 : (int)(((rv + 31) / 32) * 32);
    k_scatter<<<max_n, threads, 0, s>>>((const uint4*)k_new, (const uint4*)v_new, pos, n_dev, max_n, n_ctx, rv,
                                        (uint4*)k_cache, (uint4*)v_cache, err);
    note_launch(1);
}

// ---------------------------------------------------------------- importance scores
// SpecCache 2.2: out[i] = mean over layers of the L2 norm of hidden[i][l].  One warp per
// (token, layer) row at a time: 16-byte loads when dim allows, a fixed shuffle tree for
// the sum of squares.  A block of IMP_WARPS warps covers IMP_WARPS / w tokens with w =
// min(n_layers, IMP_WARPS) warps each; the layer norms go to shared memory and are added
// in layer order.
constexpr int IMP_WARPS = 8;
template <typename T>
__global__ void __launch_bounds__(IMP_WARPS * 32) k_importance(const T* __restrict__ h, int n, int n_layers, int dim,
                                                             float* __restrict__ out) {
    extern __shared__ float norms[];  // [tokens per block][n_layers]
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int wpt = n_layers < IMP_WARPS ? n_layers : IMP_WARPS;
    const int per_block = IMP_WARPS / wpt;
    const int tb = warp / wpt;  // token within the block
    const long long i = (long long)blockIdx.x * per_block + tb;
    const bool live = tb < per_block && i < n;
    const bool vec = dim % Vec<T>::N == 0 && ((uintptr_t)h & 15) == 0;
    if (live) {
        for (int l = warp % wpt; l < n_layers; l += wpt) {
            const T* r = h + (i * n_layers + l) * dim;
            float ss = 0.f;
            if (vec) {
#pragma unroll 4
                for (int j = lane * Vec<T>::N; j < dim; j += 32 * Vec<T>::N) {
                    const Vec<T> v = ld16(r + j);
#pragma unroll
                    for (int e = 0; e < Vec<T>::N; ++e) ss = fmaf(v.get(e), v.get(e), ss);
                }
            } else {
                for (int j = lane; j < dim; j += 32) {
                    const float v = to_f<T>(r[j]);
                    ss = fmaf(v, v, ss);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) norms[tb * n_layers + l] = sqrtf(ss);
        }
    }
    __syncthreads();
    if (live && warp % wpt == 0 && lane == 0) {
        float acc = 0.f;
        for (int l = 0; l < n_layers; ++l) acc += norms[tb * n_layers + l];
        out[i] = acc / (float)n_layers;
    }
}

void launch_importance(int dtype, const void* hidden, int n, int n_layers, int dim, float* out,
                       cudaStream_t s) {
    if (n <= 0) return;
    const int wpt = n_layers < IMP_WARPS ? n_layers : IMP_WARPS;
    const int per_block = IMP_WARPS / wpt;
    const int grid = (n + per_block - 1) / per_block;
    const size_t smem = (size_t)per_block * n_layers * sizeof(float);
    if (dtype == BLEND_BF16)
        k_importance<bf16><<<grid, IMP_WARPS * 32, smem, s>>>((const bf16*)hidden, n, n_layers, dim, out);
    else
        k_importance<float><<<grid, IMP_WARPS * 32, smem, s>>>((const float*)hidden, n, n_layers, dim, out);
    note_launch(1);
}

// ---------------------------------------------------------------- row plans
// Rows of request r = its stage set (ascending) followed by its Q query positions;
// requests are laid out one after another.  Also records, for a new plan, the row each
// position held in the previous plan (row_src; the new set is a subset of the old
// one), then updates the position -> row map.  Positions outside a request's chunk
// region (or not increasing) are reported in err and replaced by the first query
// position, so no access leaves the request's rows.
__global__ void __launch_bounds__(1024)
    k_plan(const __grid_constant__ BatchDesc bd, StageDesc st, int32_t* row_pos, int32_t* row_tok,
           int32_t* row_req, int32_t* row_src, int32_t* pos2row, int32_t* M_dev,
           int32_t* req_row_end, const int32_t* old_row_tok, const int32_t* old_M, int32_t* err) {
    __shared__ int off[BLEND_MAX_BATCH + 1];
    __shared__ int cnt[BLEND_MAX_BATCH];
    if (threadIdx.x == 0) {
        off[0] = 0;
        for (int r = 0; r < bd.n_req; ++r) {
            const ReqDesc rd = bd.r[r];
            int cap = st.iota == 2 ? (rd.P + rd.n_c) : rd.n_c;
            if (st.max_count > 0 && cap > st.max_count) cap = st.max_count;
            int n = st.iota ? cap : st.count[r];
            if (n < 0 || n > cap) {
                set_error(err, BLEND_EDEVICE);
                n = n < 0 ? 0 : cap;
            }
            cnt[r] = n;
            off[r + 1] = off[r] + n + rd.Q;
        }
    }
    __syncthreads();
    for (int r = 0; r < bd.n_req; ++r) {
        const ReqDesc rd = bd.r[r];
        const int n = cnt[r];
        for (int i = threadIdx.x; i < n + rd.Q; i += blockDim.x) {
            int pos;
            if (i < n) {
                if (st.iota) {
                    pos = st.iota == 2 ? i : rd.P + i;
                } else {
                    pos = st.set[rd.nc_off + i];
                    bool ok = pos >= rd.P && pos < rd.P + rd.n_c;
                    if (ok && i > 0) ok = st.set[rd.nc_off + i - 1] < pos;
                    if (!ok) {
                        set_error(err, BLEND_EDEVICE);
                        pos = rd.Q > 0 ? rd.P + rd.n_c : rd.P;  // a valid row of this request
                    }
                }
            } else {
                pos = rd.P + rd.n_c + (i - n);
            }
            const int row = off[r] + i;
            const int tok = rd.tok_off + pos;
            row_pos[row] = pos;
            row_tok[row] = tok;
            row_req[row] = r;
            if (old_row_tok) {
                // the new set must be part of the previous one: its row there holds tok
                int src = pos2row[tok];
                if (src < 0 || src >= *old_M || old_row_tok[src] != tok) {
                    set_error(err, BLEND_EDEVICE);
                    src = 0;
                }
                row_src[row] = src;
            }
        }
    }
    __syncthreads();
    for (int r = 0; r < bd.n_req; ++r) {
        const int base = off[r];
        const int m = off[r + 1] - base;
        for (int i = threadIdx.x; i < m; i += blockDim.x) pos2row[row_tok[base + i]] = base + i;
    }
    if (threadIdx.x == 0) {
        *M_dev = off[bd.n_req];
        for (int r = 0; r < bd.n_req; ++r) req_row_end[r] = off[r + 1];
    }
}

void launch_plan(const BatchDesc& bd, const StageDesc& st, int32_t* row_pos, int32_t* row_tok,
                 int32_t* row_req, int32_t* row_src, int32_t* pos2row, int32_t* M_dev,
                 int32_t* req_row_end, const int32_t* old_row_tok, const int32_t* old_M, int32_t* err,
                 cudaStream_t s) {
    k_plan<<<1, 1024, 0, s>>>(bd, st, row_pos, row_tok, row_req, row_src, pos2row, M_dev,
                              req_row_end, old_row_tok, old_M, err);
    note_launch(1);
}

// mask[nc_off + pos - P] = 1 for every position of request r's set (one CTA per request).
__global__ void __launch_bounds__(1024)
    k_set_mask(const __grid_constant__ BatchDesc bd, const int32_t* set, const int32_t* count,
               uint8_t* mask) {
    const ReqDesc rd = bd.r[blockIdx.x];
    for (int i = threadIdx.x; i < rd.n_c; i += blockDim.x) mask[rd.nc_off + i] = 0;
    __syncthreads();
    const int n = count[blockIdx.x];
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int p = set[rd.nc_off + i] - rd.P;
        if (p >= 0 && p < rd.n_c) mask[rd.nc_off + p] = 1;
    }
}

void launch_set_mask(const BatchDesc& bd, const int32_t* set, const int32_t* count, uint8_t* mask,
                     cudaStream_t s) {
    k_set_mask<<<bd.n_req, 1024, 0, s>>>(bd, set, count, mask);
    note_launch(1);
}

__global__ void k_fill_i32(int32_t* p, int32_t v, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        p[i] = v;
}

void launch_fill_i32(int32_t* p, int32_t v, long long n, cudaStream_t s) {
    if (n <= 0) return;
    long long b = (n + 255) / 256;
    if (b > 4096) b = 4096;
    k_fill_i32<<<(int)b, 256, 0, s>>>(p, v, n);
    note_launch(1);
}

// Copies each request's set (and count) from the workspace to the caller's outputs;
// with src == nullptr the set is every chunk row P..P+n_c-1.  Unused slots get -1.
__global__ void k_copy_sets(const __grid_constant__ BatchDesc bd, const int32_t* src,
                            const int32_t* src_n, int32_t* dst, int32_t* dst_n) {
    const ReqDesc rd = bd.r[blockIdx.x];
    const int n = src ? src_n[blockIdx.x] : rd.n_c;
    if (dst)
        for (int i = threadIdx.x; i < rd.n_c; i += blockDim.x)
            dst[rd.nc_off + i] = i < n ? (src ? src[rd.nc_off + i] : rd.P + i) : -1;
    if (dst_n && threadIdx.x == 0) dst_n[blockIdx.x] = n;
}

void launch_copy_sets(const BatchDesc& bd, const int32_t* src, const int32_t* src_n, int32_t* dst,
                      int32_t* dst_n, cudaStream_t s) {
    k_copy_sets<<<bd.n_req, 256, 0, s>>>(bd, src, src_n, dst, dst_n);
    note_launch(1);
}

}  // namespace blend
