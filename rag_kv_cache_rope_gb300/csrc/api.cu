// C ABI of libblend: argument validation, workspace layout and the orchestration of
// blended prefill (assemble -> select -> per-layer selective recompute -> final norm).
// Every argument is checked on the host before the first launch; nothing here
// synchronises the device except blend_device_status.
#include <nvtx3/nvToolsExt.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <string>
#include <vector>

#include "common.cuh"
#include "gemm_tc.cuh"

namespace {
thread_local std::string g_err;
}  // namespace

namespace blend {
static std::atomic<long long> g_launches{0};
void note_launch(int n) { g_launches += n; }
int report_error(int code, const char* msg) {
    g_err = msg;
    return code;
}
}  // namespace blend

using namespace blend;

namespace {

// Stages timed by the profiler (CUDA events on the caller's stream).
enum ProfCat {
    PROF_ASSEMBLE, PROF_SELECT, PROF_PLAN, PROF_NORM, PROF_GEMM_QKV, PROF_ROPE_KV, PROF_ATTN,
    PROF_GEMM_O, PROF_GEMM_GU, PROF_GEMM_DOWN, PROF_FINAL, PROF_N
};
const char* kProfNames[PROF_N] = {"assemble", "select", "plan_gather", "rmsnorm", "gemm_qkv", "rope_kv",
                                  "attention", "gemm_o", "gemm_gate_up", "gemm_down", "final_norm"};
struct ProfRec {
    cudaEvent_t a, b;
    int cat;
    long long launches;
};

int fail(blend_handle* h, int code, const char* fmt, ...);

}  // namespace

struct Plan {
    int32_t* row_pos;
    int32_t* row_tok;
    int32_t* row_req;
    int32_t* M;
    int32_t* req_row_end;
};

struct blend_handle {
    blend_model_cfg cfg;
    blend_weights w;
    blend_limits lim;
    char* ws;
    size_t ws_bytes;
    float2* rope;
    float* x;
    float* x2;
    float* qkv;
    void* xn;
    void* q;
    void* q2;
    void* o;
    void* hmlp;
    Plan plan[2];
    int32_t* row_src;
    int32_t* pos2row;
    int32_t* tokens;
    int32_t* err;
    int32_t* rank;
    unsigned long long* rank_keys;  // selection: sorted 64-bit keys per 2048-position tile
    int32_t* set[3];
    int32_t* set_n[3];
    uint8_t* mask;
    float* dev[2];
    float2* aux_stats;   // aux_attention_scores: softmax (max, sum) per query row, head and key span
    float* ssq;          // folded RMSNorm: per-row partial sums of squares [rows][ssq_parts]
    bool xn_scaled = false;  // xn holds bf16(x * g) of the next layer's attention norm, ssq its partials
    int ssq_parts = 0;
    // host-memory pool: per-layer copies into two staging buffers on a side stream (copy
    // engines), one event per layer, one per staging buffer
    void* stage[4];  // K0, V0, K1, V1
    cudaStream_t side = nullptr;
    cudaEvent_t ev_start = nullptr;
    cudaEvent_t ev_free[2] = {nullptr, nullptr};
    std::vector<cudaEvent_t> ev_layer;
    int use_tc;  // tensor-core GEMM for bf16
    float* split_ws;  // tensor-core GEMM: K-half partials of last-wave tiles
    int host_rc = 0;  // first failure of an internal launch during the current call
    std::string last_error;
    // profiler
    bool prof_on = false;
    uint32_t prof_mask = 0xffffffffu;  // stages recorded while prof_on (bit = stage)
    std::vector<ProfRec> prof;            // events recorded since the last read
    std::vector<cudaEvent_t> ev_pool;     // reusable events
    size_t ev_used = 0;
    ~blend_handle() {
        for (cudaEvent_t e : ev_pool) cudaEventDestroy(e);
        for (cudaEvent_t e : ev_layer) cudaEventDestroy(e);
        if (ev_start) cudaEventDestroy(ev_start);
        for (cudaEvent_t e : ev_free)
            if (e) cudaEventDestroy(e);
        if (side) cudaStreamDestroy(side);
    }
    cudaEvent_t next_event() {
        if (ev_used == ev_pool.size()) {
            cudaEvent_t e;
            if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
            ev_pool.push_back(e);
        }
        return ev_pool[ev_used++];
    }
};

namespace {
// An NVTX range for the lifetime of a scope (shown on a profiler's timeline).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Times the launches made in its lifetime under one profiler category, and marks them as
// an NVTX range named after the stage (a no-op unless a profiler is attached).
struct ProfScope {
    blend_handle* h;
    cudaStream_t s;
    int cat;
    cudaEvent_t a = nullptr;
    long long l0 = 0;
    ProfScope(blend_handle* h_, int cat_, cudaStream_t s_) : h(h_), s(s_), cat(cat_) {
        nvtxRangePushA(kProfNames[cat]);
        if (h && h->prof_on && ((h->prof_mask >> cat) & 1u) && h->prof.size() < 100000) {
            a = h->next_event();
            if (a) cudaEventRecord(a, s);
            l0 = g_launches.load();
        }
    }
    ~ProfScope() {
        if (a) {
            cudaEvent_t b = h->next_event();
            if (b) {
                cudaEventRecord(b, s);
                h->prof.push_back(ProfRec{a, b, cat, g_launches.load() - l0});
            }
        }
        nvtxRangePop();
    }
};
}  // namespace

namespace {

int fail(blend_handle* h, int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (h) h->last_error = buf;
    g_err = buf;
    return code;
}

int check_cuda(blend_handle* h, const char* where) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(h, BLEND_ECUDA, "%s: %s", where, cudaGetErrorString(e));
    return BLEND_OK;
}

// End of a public call: the first internal launch failure, else any CUDA launch error.
int finish(blend_handle* h, const char* where) {
    if (h->host_rc != BLEND_OK) {
        int rc = h->host_rc;
        h->host_rc = BLEND_OK;
        cudaGetLastError();
        return fail(h, rc, "%s: a tensor-core operand could not be described (tensor map)", where);
    }
    return check_cuda(h, where);
}

inline size_t elem_size(int dtype) { return dtype == BLEND_BF16 ? 2 : 4; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int ceil_bp(int rho_bp, int n) { return (int)(((long long)rho_bp * n + 9999) / 10000); }

// Workspace carve-up, shared by blend_workspace_size and blend_init.
struct Layout {
    size_t off[64];
    int n = 0;
    size_t total = 0;
    size_t add(size_t bytes) {
        size_t o = total;
        off[n++] = o;
        total = align_up(total + (bytes ? bytes : 1), 256);
        return o;
    }
};

bool cfg_ok(const blend_model_cfg* c, std::string* why) {
    char b[256];
    if (!c) { *why = "cfg is NULL"; return false; }
    if (c->dtype != BLEND_F32 && c->dtype != BLEND_BF16) { *why = "dtype must be BLEND_F32 or BLEND_BF16"; return false; }
    if (c->n_layers < 1 || c->hidden < 16 || c->hidden % 16 || c->n_q_heads < 1 || c->n_kv_heads < 1 ||
        c->n_q_heads % c->n_kv_heads || c->ffn < 16 || c->ffn % BLEND_GU_BLOCK || c->vocab < 1 ||
        c->max_pos < 1 || !(c->rope_theta > 0) || !(c->rms_eps >= 0)) {
        snprintf(b, sizeof b, "bad model shape (L=%d H=%d hq=%d hkv=%d F=%d vocab=%d max_pos=%d)", c->n_layers,
                 c->hidden, c->n_q_heads, c->n_kv_heads, c->ffn, c->vocab, c->max_pos);
        *why = b;
        return false;
    }
    if (c->head_dim != 64 && c->head_dim != 128) { *why = "head_dim must be 64 or 128"; return false; }
    if (c->n_q_heads / c->n_kv_heads > 32) { *why = "more than 32 query heads per kv head"; return false; }
    if (c->hidden > 8192) { *why = "hidden size above 8192"; return false; }
    return true;
}

bool lim_ok(const blend_limits* l, std::string* why) {
    if (!l) { *why = "limits is NULL"; return false; }
    if (l->max_rows < 1 || l->max_tokens < 1 || l->max_chunk_rows < 1 || l->max_batch < 1 ||
        l->max_batch > BLEND_MAX_BATCH || l->max_chunk_rows > 32768) {
        *why = "bad limits (max_rows, max_tokens >= 1; 1 <= max_chunk_rows <= 32768; 1 <= max_batch <= 64)";
        return false;
    }
    return true;
}

// Folded RMSNorm: at most this many partial sums of squares per row (hidden <= 8192).
constexpr int NORM_PARTS_MAX = 64;

Layout make_layout(const blend_model_cfg* c, const blend_limits* l) {
    Layout L;
    const size_t es = elem_size(c->dtype);
    const size_t M = (size_t)l->max_rows, H = (size_t)c->hidden, d = (size_t)c->head_dim;
    const size_t qd = (size_t)c->n_q_heads * d, kvd = (size_t)c->n_kv_heads * d;
    const size_t nc = (size_t)l->max_batch * l->max_chunk_rows;
    L.add((size_t)c->max_pos * (d / 2) * sizeof(float2));  // 0 rope
    L.add(M * H * 4);                                      // 1 x
    L.add(M * H * 4);                                      // 2 x2
    L.add(M * (qd + 2 * kvd) * 4);                         // 3 qkv
    L.add(M * H * es);                                     // 4 xn
    L.add(M * qd * es);                                    // 5 q
    L.add(M * qd * es);                                    // 6 q2
    L.add(M * qd * es);                                    // 7 o
    L.add(M * (size_t)c->ffn * es);                        // 8 hmlp
    for (int p = 0; p < 2; ++p) {                          // 9..18 plans
        L.add(M * 4);
        L.add(M * 4);
        L.add(M * 4);
        L.add(16);
        L.add(BLEND_MAX_BATCH * 4);
    }
    L.add(M * 4);                                          // 19 row_src
    L.add((size_t)l->max_tokens * 4);                      // 20 pos2row
    L.add((size_t)l->max_tokens * 4);                      // 21 tokens
    L.add(16);                                             // 22 err
    L.add(nc * 4);                                         // 23 rank
    for (int s = 0; s < 3; ++s) L.add(nc * 4);             // 24..26 sets
    for (int s = 0; s < 3; ++s) L.add(BLEND_MAX_BATCH * 4);  // 27..29 set sizes
    L.add(nc);                                             // 30 mask
    L.add(nc * 4);                                         // 31 dev1
    L.add(nc * 4);                                         // 32 dev2
    L.add(M * (size_t)c->n_q_heads * tc_score_spans(l->max_tokens) * sizeof(float2));  // 33 aux score row statistics
    L.add(c->dtype == BLEND_BF16 ? GEMM_SPLIT_WS_FLOATS * 4 : 0);  // 34 GEMM split partials
    for (int b = 0; b < 4; ++b)                            // 35..38 host-pool staging: K, V x 2 buffers
        L.add((size_t)l->max_tokens * kvd * es);
    L.add(M * NORM_PARTS_MAX * sizeof(float));             // 39 folded-RMSNorm partial sums of squares
    L.add((size_t)l->max_batch * ((l->max_chunk_rows + 2047) / 2048 * 2048) * 8);  // 40 sorted rank keys
    return L;
}

const char* ptr_in(const void* p) { return (const char*)p; }

// Per-layer weight pointers.
struct LayerW {
    const void *attn_norm, *w_qkv, *w_o, *mlp_norm, *w_gu, *w_down;
};
LayerW layer_w(const blend_handle* h, int l) {
    const blend_model_cfg& c = h->cfg;
    const size_t es = elem_size(c.dtype);
    const size_t H = c.hidden, d = c.head_dim;
    const size_t qd = (size_t)c.n_q_heads * d, kvd = (size_t)c.n_kv_heads * d, F = c.ffn;
    LayerW r;
    r.attn_norm = ptr_in(h->w.attn_norm) + (size_t)l * H * es;
    r.mlp_norm = ptr_in(h->w.mlp_norm) + (size_t)l * H * es;
    r.w_qkv = ptr_in(h->w.w_qkv) + (size_t)l * (qd + 2 * kvd) * H * es;
    r.w_o = ptr_in(h->w.w_o) + (size_t)l * H * qd * es;
    r.w_gu = ptr_in(h->w.w_gu) + (size_t)l * 2 * F * H * es;
    r.w_down = ptr_in(h->w.w_down) + (size_t)l * H * F * es;
    return r;
}

// C[M, N] (epi) A[M, K] . B[N, K]^T: tensor cores for bf16, CUDA cores for fp32.
bool gemm_on_tc(const blend_handle* h, int K, int N, int epi, int ldc) {
    return h->cfg.dtype == BLEND_BF16 && h->use_tc && tc_gemm_supported(K, N, epi, ldc, h->lim.max_rows);
}

// ne: folded-RMSNorm sides (tensor-core path only; callers pass it only when gemm_on_tc).
void gemm(blend_handle* h, const void* A, int K, const void* B, int N, int epi, void* C, int ldc,
          const int32_t* M_dev, int M_max, cudaStream_t s, const NormEpi* ne = nullptr) {
    if (gemm_on_tc(h, K, N, epi, ldc)) {
        int rc = launch_gemm_tc(A, K, h->lim.max_rows, B, N, M_dev, M_max, epi, C, ldc, h->err, s, nullptr,
                                h->split_ws, ne);
        if (rc != BLEND_OK && h->host_rc == BLEND_OK) h->host_rc = rc;
    } else
        launch_gemm_simt(h->cfg.dtype, A, K, B, K, K, N, M_dev, M_max, epi, C, ldc, s);
}

void attention(blend_handle* h, const Plan& p, int n_req, int M_max, const void* kc, const void* vc,
               long long n_tokens, cudaStream_t s) {
    const blend_model_cfg& c = h->cfg;
    if (c.dtype == BLEND_BF16 && h->use_tc && tc_attn_supported(c.head_dim)) {
        int rc = launch_attn_tc(h->q, h->lim.max_rows, n_req, p.req_row_end, p.row_pos, p.row_tok, M_max, kc, vc,
                                n_tokens, h->o, c.n_q_heads, c.n_kv_heads, c.head_dim, h->err, s);
        if (rc != BLEND_OK && h->host_rc == BLEND_OK) h->host_rc = rc;
        return;
    }
    launch_attn_simt(c.dtype, h->q, h->lim.max_rows, p.row_pos, p.row_tok, p.M, M_max, kc, vc, h->o,
                     c.n_q_heads, c.n_kv_heads, c.head_dim, s);
}

// The part of a layer after the K/V write: attention, O-proj + residual, RMSNorm,
// SwiGLU MLP + residual, on the rows of plan p (x holds those rows).
// Producer and consumer sides of the folded RMSNorm (RMSNorm(x) . W = (1/rms(x)) ((x * g) . W)):
// the residual-add GEMM writes bf16(x * g) and per-tile sums of squares, the next GEMM
// scales its rows.
NormEpi norm_producer(blend_handle* h, const void* g) {
    const int H = h->cfg.hidden;
    NormEpi ne{};
    ne.x_out = (bf16*)h->xn;
    ne.g = (const bf16*)g;
    ne.ssq_out = h->ssq;
    ne.ssq_stride = gemm_tc_norm_parts(H);
    ne.ldx = H;
    return ne;
}
NormEpi norm_consumer(blend_handle* h, int parts) {
    NormEpi ne{};
    ne.ssq_in = h->ssq;
    ne.n_part = parts;
    ne.inv_h = 1.f / (float)h->cfg.hidden;
    ne.eps = h->cfg.rms_eps;
    return ne;
}

// The rest of a layer.  next_follows: the next layer's QKV projection runs right after on
// the same rows, so the down projection may hand it normalised input.
void layer_rest(blend_handle* h, int l, float* x, const Plan& p, int n_req, int M_max, const void* kc,
                const void* vc, long long n_tokens, cudaStream_t s, bool next_follows) {
    const blend_model_cfg& c = h->cfg;
    const LayerW lw = layer_w(h, l);
    const int H = c.hidden, qd = c.n_q_heads * c.head_dim, F = c.ffn;
    const int width = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
    { ProfScope ps(h, PROF_ATTN, s); attention(h, p, n_req, M_max, kc, vc, n_tokens, s); }
    const bool fold_mlp = gemm_on_tc(h, qd, H, EPI_ADD_F32, H) && gemm_on_tc(h, H, 2 * F, EPI_SWIGLU, F) &&
                          gemm_tc_norm_parts(H) <= NORM_PARTS_MAX;
    if (fold_mlp) {
        const NormEpi prod = norm_producer(h, lw.mlp_norm);
        { ProfScope ps(h, PROF_GEMM_O, s); gemm(h, h->o, qd, lw.w_o, H, EPI_ADD_F32, x, H, p.M, M_max, s, &prod); }
        const NormEpi cons = norm_consumer(h, prod.ssq_stride);
        { ProfScope ps(h, PROF_GEMM_GU, s); gemm(h, h->xn, H, lw.w_gu, 2 * F, EPI_SWIGLU, h->hmlp, F, p.M, M_max, s, &cons); }
    } else {
        { ProfScope ps(h, PROF_GEMM_O, s); gemm(h, h->o, qd, lw.w_o, H, EPI_ADD_F32, x, H, p.M, M_max, s); }
        { ProfScope ps(h, PROF_NORM, s); launch_rmsnorm(c.dtype, x, lw.mlp_norm, h->xn, H, c.rms_eps, p.M, M_max, s); }
        { ProfScope ps(h, PROF_GEMM_GU, s); gemm(h, h->xn, H, lw.w_gu, 2 * F, EPI_SWIGLU, h->hmlp, F, p.M, M_max, s); }
    }
    const bool fold_next = next_follows && l + 1 < c.n_layers && gemm_on_tc(h, F, H, EPI_ADD_F32, H) &&
                           gemm_on_tc(h, H, width, EPI_STORE_F32, width) && gemm_tc_norm_parts(H) <= NORM_PARTS_MAX;
    if (fold_next) {
        const NormEpi prod = norm_producer(h, layer_w(h, l + 1).attn_norm);
        { ProfScope ps(h, PROF_GEMM_DOWN, s); gemm(h, h->hmlp, F, lw.w_down, H, EPI_ADD_F32, x, H, p.M, M_max, s, &prod); }
        h->xn_scaled = true;
        h->ssq_parts = prod.ssq_stride;
    } else {
        { ProfScope ps(h, PROF_GEMM_DOWN, s); gemm(h, h->hmlp, F, lw.w_down, H, EPI_ADD_F32, x, H, p.M, M_max, s); }
    }
}

// The part of a layer up to the K/V write: RMSNorm, QKV projection, RoPE, optional
// deviation against the cache, overwrite of the cache rows.
void layer_kv(blend_handle* h, int l, const float* x, const Plan& p, const int32_t* row_req,
              int M_max, const BatchDesc& bd, void* kc, void* vc, float* dev, int dev_mode,
              int dev_by_row, cudaStream_t s) {
    const blend_model_cfg& c = h->cfg;
    const LayerW lw = layer_w(h, l);
    const int H = c.hidden, d = c.head_dim;
    const int width = (c.n_q_heads + 2 * c.n_kv_heads) * d;
    // xn already holds bf16(x * g) from the previous down projection (folded RMSNorm), or
    // the norm runs here
    const bool folded = h->xn_scaled && gemm_on_tc(h, H, width, EPI_STORE_F32, width);
    h->xn_scaled = false;
    NormEpi cons{};
    if (folded)
        cons = norm_consumer(h, h->ssq_parts);
    else {
        ProfScope ps(h, PROF_NORM, s);
        launch_rmsnorm(c.dtype, x, lw.attn_norm, h->xn, H, c.rms_eps, p.M, M_max, s);
    }
    const bool fused = dev == nullptr && c.dtype == BLEND_BF16 && h->use_tc && d == 128 && width % 256 == 0 &&
                       tc_gemm_supported(H, width, EPI_QKV_ROPE, width, h->lim.max_rows);
    if (fused) {
        // projection, RoPE, q layout and the K/V cache write in one kernel
        ProfScope ps(h, PROF_GEMM_QKV, s);
        QkvEpi qe{p.row_pos, p.row_tok, h->rope, (bf16*)h->q, (bf16*)kc, (bf16*)vc, h->lim.max_rows,
                  c.n_q_heads / c.n_kv_heads, c.n_q_heads, c.n_kv_heads};
        int rc = launch_gemm_tc(h->xn, H, h->lim.max_rows, lw.w_qkv, width, p.M, M_max, EPI_QKV_ROPE, nullptr, 0,
                                h->err, s, &qe, nullptr, &cons);
        if (rc != BLEND_OK && h->host_rc == BLEND_OK) h->host_rc = rc;
        return;
    }
    {
        ProfScope ps(h, PROF_GEMM_QKV, s);
        gemm(h, h->xn, H, lw.w_qkv, width, EPI_STORE_F32, h->qkv, width, p.M, M_max, s, folded ? &cons : nullptr);
    }
    ProfScope ps(h, PROF_ROPE_KV, s);
    launch_rope_qkv(c.dtype, h->qkv, p.row_pos, p.row_tok, row_req, p.M, M_max, bd, c.n_q_heads,
                    c.n_kv_heads, d, h->lim.max_rows, h->rope, h->q, kc, vc, dev, dev_mode, dev_by_row, s);
}

}  // namespace

extern "C" {

size_t blend_workspace_size(const blend_model_cfg* cfg, const blend_limits* lim) {
    std::string why;
    if (!cfg_ok(cfg, &why) || !lim_ok(lim, &why)) return 0;
    return make_layout(cfg, lim).total;
}

const char* blend_last_error(const blend_handle* h) {
    return h ? h->last_error.c_str() : g_err.c_str();
}

int blend_init(const blend_model_cfg* cfg, const blend_weights* w, const blend_limits* lim,
               void* workspace, size_t ws_bytes, void* stream, blend_handle** out) {
    std::string why;
    if (!out) return fail(nullptr, BLEND_EINVAL, "out is NULL");
    *out = nullptr;
    if (!cfg_ok(cfg, &why) || !lim_ok(lim, &why)) return fail(nullptr, BLEND_EINVAL, "%s", why.c_str());
    if (!w || !w->embed || !w->attn_norm || !w->w_qkv || !w->w_o || !w->mlp_norm || !w->w_gu ||
        !w->w_down || !w->final_norm)
        return fail(nullptr, BLEND_EINVAL, "a weight pointer is NULL");
    if (!workspace || ((uintptr_t)workspace & 255))
        return fail(nullptr, BLEND_EINVAL, "workspace must be non-NULL and 256-byte aligned");
    Layout L = make_layout(cfg, lim);
    if (ws_bytes < L.total)
        return fail(nullptr, BLEND_ENOMEM, "workspace has %zu bytes, needs %zu", ws_bytes, L.total);
    blend_handle* h = new blend_handle();
    h->cfg = *cfg;
    h->w = *w;
    h->lim = *lim;
    h->ws = (char*)workspace;
    h->ws_bytes = ws_bytes;
    char* b = h->ws;
    int i = 0;
    h->rope = (float2*)(b + L.off[i++]);
    h->x = (float*)(b + L.off[i++]);
    h->x2 = (float*)(b + L.off[i++]);
    h->qkv = (float*)(b + L.off[i++]);
    h->xn = b + L.off[i++];
    h->q = b + L.off[i++];
    h->q2 = b + L.off[i++];
    h->o = b + L.off[i++];
    h->hmlp = b + L.off[i++];
    for (int p = 0; p < 2; ++p) {
        h->plan[p].row_pos = (int32_t*)(b + L.off[i++]);
        h->plan[p].row_tok = (int32_t*)(b + L.off[i++]);
        h->plan[p].row_req = (int32_t*)(b + L.off[i++]);
        h->plan[p].M = (int32_t*)(b + L.off[i++]);
        h->plan[p].req_row_end = (int32_t*)(b + L.off[i++]);
    }
    h->row_src = (int32_t*)(b + L.off[i++]);
    h->pos2row = (int32_t*)(b + L.off[i++]);
    h->tokens = (int32_t*)(b + L.off[i++]);
    h->err = (int32_t*)(b + L.off[i++]);
    h->rank = (int32_t*)(b + L.off[i++]);
    for (int s = 0; s < 3; ++s) h->set[s] = (int32_t*)(b + L.off[i++]);
    for (int s = 0; s < 3; ++s) h->set_n[s] = (int32_t*)(b + L.off[i++]);
    h->mask = (uint8_t*)(b + L.off[i++]);
    h->dev[0] = (float*)(b + L.off[i++]);
    h->dev[1] = (float*)(b + L.off[i++]);
    h->aux_stats = (float2*)(b + L.off[i++]);
    h->split_ws = cfg->dtype == BLEND_BF16 ? (float*)(b + L.off[i]) : nullptr;
    ++i;
    for (int q = 0; q < 4; ++q) h->stage[q] = b + L.off[i++];
    h->ssq = (float*)(b + L.off[i++]);
    h->rank_keys = (unsigned long long*)(b + L.off[i++]);
    h->use_tc = cfg->dtype == BLEND_BF16 ? tc_available() : 0;
    cudaStream_t s = (cudaStream_t)stream;
    cudaMemsetAsync(h->err, 0, 16, s);
    launch_rope_table(h->rope, cfg->max_pos, cfg->head_dim, cfg->rope_theta, s);
    int rc = check_cuda(h, "blend_init");
    if (rc != BLEND_OK) {
        g_err = h->last_error;
        delete h;
        return rc;
    }
    *out = h;
    return BLEND_OK;
}

int blend_destroy(blend_handle* h) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    delete h;
    return BLEND_OK;
}

// Synchronises `stream`, then reports (and clears) the handle's device error word.
int blend_device_status(blend_handle* h, void* stream) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return check_cuda(h, "blend_device_status");
    int32_t e = 0;
    if (cudaMemcpy(&e, h->err, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return check_cuda(h, "blend_device_status");
    if (e != 0) {
        cudaMemset(h->err, 0, 4);
        return fail(h, e == BLEND_ETIMEOUT ? BLEND_ETIMEOUT : BLEND_EDEVICE,
                    "device-side check failed (code %d)", e);
    }
    return BLEND_OK;
}

int blend_wait_flag(blend_handle* h, const int32_t* flag, int64_t max_polls, void* stream) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    if (!flag) return fail(h, BLEND_EINVAL, "flag is NULL");
    if (((uintptr_t)flag & 3) != 0) return fail(h, BLEND_EINVAL, "flag must be 4-byte aligned");
    if (max_polls < 0 || max_polls > BLEND_MAX_WAIT_POLLS)
        return fail(h, BLEND_EINVAL, "max_polls=%lld outside 0..%lld", (long long)max_polls,
                    (long long)BLEND_MAX_WAIT_POLLS);
    launch_wait_flag(flag, (long long)max_polls, h->err, (cudaStream_t)stream);
    return check_cuda(h, "blend_wait_flag");
}

int blend_set_tensor_cores(blend_handle* h, int on) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    h->use_tc = (on && h->cfg.dtype == BLEND_BF16 && tc_available()) ? 1 : 0;
    return h->use_tc;
}

int blend_profile(blend_handle* h, int enable) {
    return blend_profile_stages(h, enable != 0 ? 0xffffffffu : 0u);
}

int blend_profile_stages(blend_handle* h, uint32_t stage_mask) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    h->prof.clear();
    h->ev_used = 0;
    h->prof_on = stage_mask != 0;
    h->prof_mask = stage_mask;
    return BLEND_OK;
}

int blend_profile_read(blend_handle* h, double* ms, int64_t* launches, int32_t n) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    if (n < 0 || (n > 0 && (!ms || !launches))) return fail(h, BLEND_EINVAL, "bad output arrays");
    for (int i = 0; i < n && i < PROF_N; ++i) {
        ms[i] = 0.0;
        launches[i] = 0;
    }
    for (const ProfRec& r : h->prof) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) return check_cuda(h, "blend_profile_read");
        float t = 0.f;
        cudaEventElapsedTime(&t, r.a, r.b);
        if (r.cat < n) {
            ms[r.cat] += t;
            launches[r.cat] += r.launches;
        }
    }
    h->prof.clear();
    h->ev_used = 0;
    return PROF_N;
}

const char* blend_profile_name(int32_t i) { return (i >= 0 && i < PROF_N) ? kProfNames[i] : ""; }

int64_t blend_launch_count(void) { return g_launches.load(); }

int rope_realign(blend_handle* h, const void* k_src, void* k_dst, int32_t n_rows,
                 const int32_t* delta, int32_t n_layers, int64_t src_layer_rows,
                 int64_t dst_layer_rows, void* stream) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    if (!k_src || !k_dst || !delta) return fail(h, BLEND_EINVAL, "NULL pointer");
    if (n_rows < 0 || n_layers < 0 || src_layer_rows < n_rows || dst_layer_rows < n_rows)
        return fail(h, BLEND_EINVAL, "bad sizes");
    if (((uintptr_t)k_src | (uintptr_t)k_dst) & 15) return fail(h, BLEND_EINVAL, "k_src/k_dst must be 16-byte aligned");
    launch_realign(h->cfg.dtype, k_src, k_dst, n_rows, delta, n_layers, src_layer_rows,
                   dst_layer_rows, h->cfg.n_kv_heads, h->cfg.head_dim, h->rope, h->cfg.max_pos,
                   h->err, (cudaStream_t)stream);
    return check_cuda(h, "rope_realign");
}

int kv_deviation(blend_handle* h, const void* k_new, const void* v_new, const void* k_cache,
                 const void* v_cache, const int32_t* pos, const int32_t* n_rows, int32_t max_rows,
                 int64_t n_ctx, int32_t mode, float* dev_out, void* stream) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    if (!k_new || !v_new || !k_cache || !v_cache || !pos || !n_rows || !dev_out)
        return fail(h, BLEND_EINVAL, "NULL pointer");
    if (max_rows < 0 || n_ctx < 0 || (mode != BLEND_DEV_KV && mode != BLEND_DEV_V))
        return fail(h, BLEND_EINVAL, "bad mode or size");
    if (((uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)k_cache | (uintptr_t)v_cache) & 15)
        return fail(h, BLEND_EINVAL, "K/V pointers must be 16-byte aligned");
    launch_deviation(h->cfg.dtype, k_new, v_new, k_cache, v_cache, pos, n_rows, max_rows, n_ctx,
                     h->cfg.n_kv_heads * h->cfg.head_dim, mode, dev_out, h->err, (cudaStream_t)stream);
    return check_cuda(h, "kv_deviation");
}

int topk_select_dilate(blend_handle* h, const float* scores, int32_t n, int32_t base,
                       int32_t budget, int32_t window, int32_t tau, int32_t budget_mode,
                       const uint8_t* allowed, int32_t* idx_out, int32_t* n_out, void* stream) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    if (!scores || !idx_out || !n_out) return fail(h, BLEND_EINVAL, "NULL pointer");
    if (n < 0 || n > 32768 || (long long)n > (long long)h->lim.max_batch * h->lim.max_chunk_rows)
        return fail(h, BLEND_EINVAL, "n=%d outside 0..min(32768, workspace capacity)", n);
    if (budget < 0 || window < 1 || window > BLEND_MAX_WINDOW || tau < 1 || tau > window)
        return fail(h, BLEND_EINVAL, "bad budget/window/tau (%d/%d/%d)", budget, window, tau);
    if (budget_mode != BLEND_BUDGET_FINAL && budget_mode != BLEND_BUDGET_CANDIDATE)
        return fail(h, BLEND_EINVAL, "bad budget_mode");
    SelectBatch sb;
    memset(&sb, 0, sizeof sb);
    sb.n_job = 1;
    sb.window = window;
    sb.tau = tau;
    sb.budget_mode = budget_mode;
    sb.j[0] = SelectJob{scores, allowed, idx_out, n_out, n, base, budget, 0};
    launch_select(sb, h->rank, h->rank_keys, n, (cudaStream_t)stream);
    return check_cuda(h, "topk_select_dilate");
}

int span_select(blend_handle* h, const float* scores, int32_t n, int32_t base, int32_t budget, int32_t cap,
                float tau_smooth, int32_t tau_cover_bp, int32_t max_span, int32_t budget_mode,
                int32_t* idx_out, int32_t* n_out, void* stream) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    if (!scores || !idx_out || !n_out) return fail(h, BLEND_EINVAL, "NULL pointer");
    if (n < 0 || n > 32768 || (long long)n > (long long)h->lim.max_batch * h->lim.max_chunk_rows)
        return fail(h, BLEND_EINVAL, "n=%d outside 0..min(32768, workspace capacity)", n);
    if (budget < 0 || cap < 0 || !std::isfinite(tau_smooth) || tau_smooth < 0.f || tau_cover_bp < 1 ||
        tau_cover_bp > 10000 || max_span < 1 || max_span > BLEND_MAX_SPAN)
        return fail(h, BLEND_EINVAL, "bad budget/cap/tau_smooth/tau_cover_bp/max_span");
    if (budget_mode != BLEND_BUDGET_FINAL && budget_mode != BLEND_BUDGET_CANDIDATE)
        return fail(h, BLEND_EINVAL, "bad budget_mode");
    SelectBatch sb;
    memset(&sb, 0, sizeof sb);
    sb.n_job = 1;
    sb.window = 1;
    sb.tau = 1;
    sb.budget_mode = budget_mode;
    sb.rule = BLEND_GROUP_SPAN;
    sb.tau_smooth = tau_smooth;
    sb.tau_cover_bp = tau_cover_bp;
    sb.max_span = max_span;
    sb.j[0] = SelectJob{scores, nullptr, idx_out, n_out, n, base, budget, 0, cap};
    launch_select(sb, h->rank, h->rank_keys, n, (cudaStream_t)stream);
    return check_cuda(h, "span_select");
}

int align_expand(blend_handle* h, const int32_t* sel, const int32_t* n_sel, int32_t max_sel, int32_t sel_base,
                 const int32_t* a_start, const int32_t* a_end, int32_t n_spec, int32_t n_target,
                 int32_t out_base, int32_t* idx_out, int32_t* n_out, void* stream) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    if (!sel || !n_sel || !idx_out || !n_out || (n_spec > 0 && (!a_start || !a_end)))
        return fail(h, BLEND_EINVAL, "NULL pointer");
    if (max_sel < 0 || n_spec < 0 || n_target < 0 || n_target > BLEND_MAX_ALIGN_TARGETS)
        return fail(h, BLEND_EINVAL, "bad sizes (max_sel %d, n_spec %d, n_target %d)", max_sel, n_spec, n_target);
    launch_align_expand(sel, n_sel, max_sel, sel_base, a_start, a_end, n_spec, n_target, out_base, idx_out, n_out,
                        h->err, (cudaStream_t)stream);
    return check_cuda(h, "align_expand");
}

int blend_ratio_controller(double full_prefill_s, double kv_bytes, double load_bytes_per_s, int32_t floor_bp,
                           int32_t* rho_bp) {
    if (!rho_bp) return fail(nullptr, BLEND_EINVAL, "rho_bp is NULL");
    if (!(std::isfinite(full_prefill_s) && full_prefill_s > 0) || !(std::isfinite(kv_bytes) && kv_bytes > 0) ||
        !(std::isfinite(load_bytes_per_s) && load_bytes_per_s > 0) || floor_bp < 0 || floor_bp > 10000)
        return fail(nullptr, BLEND_EINVAL, "controller inputs must be positive and finite, floor in 0..10000");
    const double load_s = kv_bytes / load_bytes_per_s;
    const double r = std::ceil(10000.0 * (load_s / full_prefill_s));
    const double v = r > 10000.0 ? 10000.0 : (r < (double)floor_bp ? (double)floor_bp : r);
    *rho_bp = (int32_t)v;
    return BLEND_OK;
}

int blend_pick_storage(double full_prefill_s, double kv_bytes, int32_t floor_bp, int32_t n_dev,
                       const double* bytes_per_s, const double* cost_per_byte, int32_t* best) {
    if (!best || n_dev < 0 || (n_dev > 0 && (!bytes_per_s || !cost_per_byte)))
        return fail(nullptr, BLEND_EINVAL, "NULL pointer or negative device count");
    if (!(std::isfinite(full_prefill_s) && full_prefill_s > 0) || !(std::isfinite(kv_bytes) && kv_bytes > 0) ||
        floor_bp < 0 || floor_bp > 10000)
        return fail(nullptr, BLEND_EINVAL, "controller inputs must be positive and finite, floor in 0..10000");
    const double budget_s = ((double)floor_bp / 10000.0) * full_prefill_s;
    *best = -1;
    for (int32_t i = 0; i < n_dev; ++i) {
        if (!(bytes_per_s[i] > 0) || !std::isfinite(cost_per_byte[i]))
            return fail(nullptr, BLEND_EINVAL, "device %d: throughput must be positive, cost finite", i);
        const double load_s = kv_bytes / bytes_per_s[i];
        if (load_s <= budget_s && (*best < 0 || cost_per_byte[i] < cost_per_byte[*best])) *best = i;
    }
    return BLEND_OK;
}

int gather_rows(blend_handle* h, const void* src, int64_t row_bytes, int64_t src_rows, const int32_t* idx,
                const int32_t* n, int32_t max_n, void* dst, void* stream) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    if (!src || !idx || !n || !dst) return fail(h, BLEND_EINVAL, "NULL pointer");
    if (row_bytes <= 0 || row_bytes % 16 || max_n < 0 || src_rows < 0)
        return fail(h, BLEND_EINVAL, "row_bytes must be a positive multiple of 16, max_n and src_rows >= 0");
    if (((uintptr_t)src | (uintptr_t)dst) & 15) return fail(h, BLEND_EINVAL, "src/dst must be 16-byte aligned");
    launch_gather(src, row_bytes, src_rows, idx, n, max_n, dst, h->err, (cudaStream_t)stream);
    return check_cuda(h, "gather_rows");
}

int scatter_kv(blend_handle* h, const void* k_new, const void* v_new, const int32_t* pos,
               const int32_t* n, int32_t max_n, int64_t n_ctx, void* k_cache, void* v_cache, void* stream) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    if (!k_new || !v_new || !pos || !n || !k_cache || !v_cache) return fail(h, BLEND_EINVAL, "NULL pointer");
    if (max_n < 0 || n_ctx < 0) return fail(h, BLEND_EINVAL, "bad max_n or n_ctx");
    if (((uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)k_cache | (uintptr_t)v_cache) & 15)
        return fail(h, BLEND_EINVAL, "pointers must be 16-byte aligned");
    launch_scatter(h->cfg.dtype, k_new, v_new, pos, n, max_n, n_ctx, h->cfg.n_kv_heads * h->cfg.head_dim,
                   k_cache, v_cache, h->err, (cudaStream_t)stream);
    return check_cuda(h, "scatter_kv");
}

int importance_scores(const void* hidden, int32_t n, int32_t n_layers, int32_t dim, int32_t dtype,
                      float* out, void* stream) {
    if (!hidden || !out) return fail(nullptr, BLEND_EINVAL, "NULL pointer");
    if (n < 0 || n_layers < 1 || n_layers > 4096 || dim < 1 || (dtype != BLEND_F32 && dtype != BLEND_BF16))
        return fail(nullptr, BLEND_EINVAL, "bad sizes or dtype");
    launch_importance(dtype, hidden, n, n_layers, dim, out, (cudaStream_t)stream);
    return check_cuda(nullptr, "importance_scores");
}

int selective_layer(blend_handle* h, int32_t layer, float* x, const int32_t* pos, const int32_t* n,
                    int32_t max_n, void* k_cache, void* v_cache, int32_t n_ctx, float* dev_out, int32_t dev_mode,
                    void* stream) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    const blend_model_cfg& c = h->cfg;
    if (!x || !pos || !n || !k_cache || !v_cache) return fail(h, BLEND_EINVAL, "NULL pointer");
    if (layer < 0 || layer >= c.n_layers) return fail(h, BLEND_EINVAL, "layer %d out of range", layer);
    if (max_n < 0 || max_n > h->lim.max_rows || n_ctx < 0 || n_ctx > c.max_pos || n_ctx > h->lim.max_tokens)
        return fail(h, BLEND_EINVAL, "max_n=%d / n_ctx=%d outside the handle's limits", max_n, n_ctx);
    if (dev_mode != BLEND_DEV_KV && dev_mode != BLEND_DEV_V) return fail(h, BLEND_EINVAL, "bad dev_mode");
    if (max_n == 0) return BLEND_OK;
    cudaStream_t s = (cudaStream_t)stream;
    BatchDesc bd;
    memset(&bd, 0, sizeof bd);
    bd.n_req = 1;
    bd.r[0] = ReqDesc{0, 0, n_ctx, 0, 0, 0};
    // rows = the given positions, in order; the device count is checked against max_n and n_ctx
    StageDesc st{pos, n, 0, max_n};
    Plan& p = h->plan[0];
    launch_plan(bd, st, p.row_pos, p.row_tok, p.row_req, h->row_src, h->pos2row, p.M, p.req_row_end,
                nullptr, nullptr, h->err, s);
    h->xn_scaled = false;
    layer_kv(h, layer, x, p, p.row_req, max_n, bd, k_cache, v_cache, dev_out, dev_mode, 1, s);
    layer_rest(h, layer, x, p, 1, max_n, k_cache, v_cache, n_ctx, s, false);
    return finish(h, "selective_layer");
}

}  // extern "C"

// ------------------------------------------------------------------ blended prefill
namespace {

struct ReqInfo {
    int P, n_c, Q, N, B, k1, max_rows, cap;
    int stage_rows[3];  // most chunk rows each stage can hold (stage 0 = max_rows - Q)
};

int validate_batch(blend_handle* h, int n_req, const blend_request* reqs, const blend_pool* pool,
                   const blend_outputs* out, std::vector<ReqInfo>* info, bool check_rows = true) {
    const blend_model_cfg& c = h->cfg;
    if (n_req < 1 || n_req > h->lim.max_batch) return fail(h, BLEND_EINVAL, "n_req=%d outside 1..%d", n_req, h->lim.max_batch);
    if (!reqs || !pool || !out) return fail(h, BLEND_EINVAL, "NULL reqs/pool/out");
    if (!pool->entry_len || !pool->entry_row || !pool->k || !pool->v || !pool->tokens || pool->n_entries < 1 ||
        pool->prefix_len < 0 || pool->n_rows < 1)
        return fail(h, BLEND_EINVAL, "bad pool description");
    if (pool->n_rows >= (1LL << 31)) return fail(h, BLEND_EUNSUPPORTED, "pool rows per layer must be < 2^31");
    if (pool->location != BLEND_POOL_DEVICE && pool->location != BLEND_POOL_HOST)
        return fail(h, BLEND_EINVAL, "bad pool location %d", pool->location);
    if (pool->location == BLEND_POOL_HOST) {
        // the GPU reads the pool in place: it must be pinned (page-locked, mapped) host memory
        const void* ptrs[3] = {pool->k, pool->v, pool->tokens};
        for (const void* ptr : ptrs) {
            cudaPointerAttributes a;
            if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess || a.type != cudaMemoryTypeHost ||
                a.devicePointer != ptr) {
                cudaGetLastError();
                return fail(h, BLEND_EINVAL, "a host pool must be pinned host memory the GPU can address directly");
            }
        }
    }
    if (!out->k || !out->v || !out->hidden) return fail(h, BLEND_EINVAL, "outputs k, v and hidden are required");
    if (((uintptr_t)out->k | (uintptr_t)out->v | (uintptr_t)pool->k | (uintptr_t)pool->v) & 15)
        return fail(h, BLEND_EINVAL, "caches must be 16-byte aligned");
    const int mode = reqs[0].mode;
    long long tot_tok = 0, tot_rows = 0, n_seg = 0;
    for (int r = 0; r < n_req; ++r) {
        const blend_request& q = reqs[r];
        if (q.mode != mode || q.window != reqs[0].window || q.tau != reqs[0].tau ||
            q.budget_mode != reqs[0].budget_mode || q.dev_mode != reqs[0].dev_mode ||
            q.group_rule != reqs[0].group_rule)
            return fail(h, BLEND_EINVAL, "requests of one batch must share mode, window, tau, budget, deviation and grouping rule");
        if (q.group_rule != BLEND_GROUP_WINDOW && q.group_rule != BLEND_GROUP_SPAN)
            return fail(h, BLEND_EINVAL, "request %d: bad group_rule %d", r, q.group_rule);
        if (q.focus_bp != reqs[0].focus_bp || q.focus_layer != reqs[0].focus_layer)
            return fail(h, BLEND_EINVAL, "requests of one batch must share focus_layer and focus_bp");
        if (q.focus_bp < 0 || q.focus_bp > 10000)
            return fail(h, BLEND_EINVAL, "request %d: focus_bp must be in 0..10000", r);
        if (q.focus_bp > 0 && ((mode != BLEND_SEL_EXT && mode != BLEND_SEL_EPIC) || q.focus_layer < 0 ||
                               q.focus_layer >= c.n_layers))
            return fail(h, BLEND_EINVAL, "request %d: focus filtering needs EXT or EPIC mode and 0 <= focus_layer < L", r);
        if (q.group_rule == BLEND_GROUP_SPAN) {
            if (mode != BLEND_SEL_EXT) return fail(h, BLEND_EINVAL, "the span rule applies to EXT mode only");
            if (q.tau_smooth != reqs[0].tau_smooth || q.tau_cover_bp != reqs[0].tau_cover_bp ||
                q.max_span != reqs[0].max_span)
                return fail(h, BLEND_EINVAL, "requests of one batch must share the span parameters");
            if (!std::isfinite(q.tau_smooth) || q.tau_smooth < 0.f || q.tau_cover_bp < 1 || q.tau_cover_bp > 10000 ||
                q.max_span < 1 || q.max_span > BLEND_MAX_SPAN)
                return fail(h, BLEND_EINVAL, "request %d: bad tau_smooth/tau_cover_bp/max_span", r);
            if (q.budget_mode == BLEND_BUDGET_CANDIDATE && (q.cap_bp < q.rho_bp || q.cap_bp > 10000))
                return fail(h, BLEND_EINVAL, "request %d: cap_bp must be in rho_bp..10000", r);
        }
        if (mode < BLEND_SEL_EXT || mode > BLEND_SEL_EPIC) return fail(h, BLEND_EINVAL, "bad mode %d", mode);
        if (q.n_chunks < 1 || !q.chunk_ids || q.query_len < 1 || !q.query_tokens)
            return fail(h, BLEND_EINVAL, "request %d: needs >= 1 chunk and a non-empty query", r);
        if (q.rho_bp < 0 || q.rho_bp > 10000 || q.window < 1 || q.window > BLEND_MAX_WINDOW || q.tau < 1 ||
            q.tau > q.window)
            return fail(h, BLEND_EINVAL, "request %d: bad rho/window/tau (%d/%d/%d)", r, q.rho_bp, q.window, q.tau);
        if (q.budget_mode != BLEND_BUDGET_FINAL && q.budget_mode != BLEND_BUDGET_CANDIDATE)
            return fail(h, BLEND_EINVAL, "bad budget_mode");
        if (q.dev_mode != BLEND_DEV_KV && q.dev_mode != BLEND_DEV_V) return fail(h, BLEND_EINVAL, "bad dev_mode");
        ReqInfo ri{};
        ri.P = pool->prefix_len;
        long long nc = 0;
        for (int j = 0; j < q.n_chunks; ++j) {
            int e = q.chunk_ids[j];
            if (e < 0 || e >= pool->n_entries) return fail(h, BLEND_EINVAL, "request %d: chunk id %d not in the pool", r, e);
            if (pool->present && !pool->present[e]) return fail(h, BLEND_EMISS, "request %d: pool entry %d has no cache", r, e);
            if (pool->entry_len[e] < 1 || pool->entry_row[e] < 0 ||
                pool->entry_row[e] + pool->prefix_len + pool->entry_len[e] > pool->n_rows)
                return fail(h, BLEND_EINVAL, "pool entry %d lies outside the pool rows", e);
            nc += pool->entry_len[e];
        }
        n_seg += q.n_chunks + 1;
        if (nc > h->lim.max_chunk_rows) return fail(h, BLEND_ENOMEM, "request %d: %lld chunk rows > limit %d", r, nc, h->lim.max_chunk_rows);
        ri.n_c = (int)nc;
        ri.Q = q.query_len;
        ri.N = ri.P + ri.n_c + ri.Q;
        if (ri.N > c.max_pos) return fail(h, BLEND_EINVAL, "request %d: %d tokens > max_pos %d", r, ri.N, c.max_pos);
        ri.B = ceil_bp(q.rho_bp, ri.n_c);
        int chunk_rows = 0;
        if (mode == BLEND_SEL_EXT) {
            if (!q.scores) return fail(h, BLEND_EINVAL, "request %d: EXT mode needs scores", r);
            if (q.budget_mode == BLEND_BUDGET_FINAL) {
                chunk_rows = ri.B < ri.n_c ? ri.B : ri.n_c;
            } else if (q.group_rule == BLEND_GROUP_SPAN) {
                ri.cap = ceil_bp(q.cap_bp, ri.n_c);
                chunk_rows = ri.cap < ri.n_c ? ri.cap : ri.n_c;
            } else {
                chunk_rows = ri.n_c;
            }
        } else if (mode == BLEND_SEL_HKVD) {
            if (q.r1_bp < q.rho_bp || q.r1_bp > 10000) return fail(h, BLEND_EINVAL, "request %d: r1_bp must be in rho_bp..10000", r);
            ri.k1 = ceil_bp(q.r1_bp, ri.n_c);
            chunk_rows = ri.n_c;
            // C1 holds exactly k1 rows; S lies within C1 and, with the final budget, holds at most B
            ri.stage_rows[1] = ri.k1;
            ri.stage_rows[2] = q.budget_mode == BLEND_BUDGET_FINAL && ri.B < ri.k1 ? ri.B : ri.k1;
        } else if (mode == BLEND_SEL_FORCED) {
            if (q.n_stages < 1 || q.n_stages > 3 || q.stage_layer[0] != 0)
                return fail(h, BLEND_EINVAL, "request %d: FORCED needs 1..3 stages, the first at layer 0", r);
            for (int s = 0; s < q.n_stages; ++s) {
                if (q.stage_n[s] < 0 || q.stage_n[s] > ri.n_c || (q.stage_n[s] > 0 && !q.stage_pos[s]))
                    return fail(h, BLEND_EINVAL, "request %d: bad stage %d", r, s);
                if (s > 0 && (q.stage_layer[s] <= q.stage_layer[s - 1] || q.stage_n[s] > q.stage_n[s - 1] ||
                              q.stage_layer[s] != reqs[0].stage_layer[s]))
                    return fail(h, BLEND_EINVAL, "request %d: stages must start on increasing layers (same for every request) and shrink", r);
                if (q.n_stages != reqs[0].n_stages) return fail(h, BLEND_EINVAL, "requests must have the same number of stages");
            }
            chunk_rows = q.stage_n[0];
            for (int s = 1; s < q.n_stages; ++s) ri.stage_rows[s] = q.stage_n[s];
        } else if (mode == BLEND_SEL_EPIC) {
            if (q.epic_m < 0) return fail(h, BLEND_EINVAL, "request %d: epic_m must be >= 0", r);
            for (int j = 0; j < q.n_chunks; ++j) {
                const int L = pool->entry_len[q.chunk_ids[j]];
                chunk_rows += q.epic_m < L ? q.epic_m : L;
            }
        } else {
            chunk_rows = ri.P + ri.n_c;
        }
        ri.max_rows = chunk_rows + ri.Q;
        ri.stage_rows[0] = chunk_rows;
        if (mode != BLEND_SEL_HKVD && mode != BLEND_SEL_FORCED) ri.stage_rows[1] = ri.stage_rows[2] = chunk_rows;
        tot_tok += ri.N;
        tot_rows += ri.max_rows;
        info->push_back(ri);
    }
    if (n_seg > BLEND_MAX_CHUNKS + BLEND_MAX_BATCH) return fail(h, BLEND_EUNSUPPORTED, "too many chunks in one call");
    if (tot_tok > h->lim.max_tokens) return fail(h, BLEND_ENOMEM, "%lld blended tokens > limit %d", tot_tok, h->lim.max_tokens);
    if (check_rows && tot_rows > h->lim.max_rows)
        return fail(h, BLEND_ENOMEM, "%lld recomputed rows > limit %d", tot_rows, h->lim.max_rows);
    return BLEND_OK;
}

}  // namespace

namespace {
// Segment table (prefix rows once, then each chunk's rows with its shift) and query table
// of a validated batch.
void build_segments(int n_req, const blend_request* reqs, const blend_pool* pool, const std::vector<ReqInfo>& info,
                    SegTable& segs, QueryTable& qt, int* tok_out) {
    memset(&qt, 0, sizeof qt);
    segs.n_seg = 0;
    int row = 0, tok = 0;
    for (int r = 0; r < n_req; ++r) {
        const blend_request& q = reqs[r];
        const int P = info[r].P;
        if (P > 0) {
            const int e0 = q.chunk_ids[0];
            segs.s[segs.n_seg++] = Seg{row, (int32_t)pool->entry_row[e0], tok, P, 0};
            row += P;
        }
        int off = 0;
        for (int j = 0; j < q.n_chunks; ++j) {
            const int e = q.chunk_ids[j];
            const int L = pool->entry_len[e];
            segs.s[segs.n_seg++] = Seg{row, (int32_t)(pool->entry_row[e] + P), tok + P + off, L, off};
            row += L;
            off += L;
        }
        qt.ptr[qt.n] = q.query_tokens;
        qt.dst_tok[qt.n] = tok + P + off;
        qt.len[qt.n] = q.query_len;
        qt.n++;
        tok += info[r].N;
    }
    segs.total_rows = row;
    *tok_out = tok;
}

// Host-pool staging: merged runs of pool rows [start, end) and their first staging row.
struct Run {
    long long start, end, stage;
};
thread_local SegTable hp_segs;
thread_local QueryTable hp_qt;
thread_local std::vector<Run> hp_runs;
thread_local int hp_tok = 0;
thread_local long long hp_staged = 0;

// Copy engines: layer l's pool rows (every run, K and V) into staging buffer l % 2 on the
// side stream, then mark layer l as landed.
void stage_layer_copy(blend_handle* h, const blend_pool* pool, int l) {
    const blend_model_cfg& c = h->cfg;
    const size_t row_bytes = (size_t)c.n_kv_heads * c.head_dim * elem_size(c.dtype);
    const char* pk = (const char*)pool->k + (size_t)l * pool->n_rows * row_bytes;
    const char* pv = (const char*)pool->v + (size_t)l * pool->n_rows * row_bytes;
    char* sk = (char*)h->stage[2 * (l & 1)];
    char* sv = (char*)h->stage[2 * (l & 1) + 1];
    for (const Run& r : hp_runs) {
        const size_t n = (size_t)(r.end - r.start) * row_bytes;
        cudaMemcpyAsync(sk + r.stage * row_bytes, pk + r.start * row_bytes, n, cudaMemcpyHostToDevice, h->side);
        cudaMemcpyAsync(sv + r.stage * row_bytes, pv + r.start * row_bytes, n, cudaMemcpyHostToDevice, h->side);
    }
    cudaEventRecord(h->ev_layer[l], h->side);
}

// Side stream and per-layer events of the host-pool pipeline (created on first use).
int ensure_pipeline(blend_handle* h) {
    if (!h->side && cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess)
        return check_cuda(h, "pipeline stream");
    if (!h->ev_start && cudaEventCreateWithFlags(&h->ev_start, cudaEventDisableTiming) != cudaSuccess)
        return check_cuda(h, "pipeline event");
    for (cudaEvent_t& e : h->ev_free)
        if (!e && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
            return check_cuda(h, "pipeline event");
    while ((int)h->ev_layer.size() < h->cfg.n_layers) {
        cudaEvent_t e;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return check_cuda(h, "pipeline event");
        h->ev_layer.push_back(e);
    }
    return BLEND_OK;
}
}  // namespace

extern "C" int blend_assemble(blend_handle* h, int32_t n_req, const blend_request* reqs,
                              const blend_pool* pool, const blend_outputs* out, void* stream) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    std::vector<ReqInfo> info;
    int rc = validate_batch(h, n_req, reqs, pool, out, &info, false);
    if (rc != BLEND_OK) return rc;
    const blend_model_cfg& c = h->cfg;
    cudaStream_t s = (cudaStream_t)stream;
    static thread_local SegTable segs;
    static thread_local QueryTable qt;
    int tok = 0;
    build_segments(n_req, reqs, pool, info, segs, qt, &tok);
    launch_assemble(c.dtype, segs, pool->k, pool->v, pool->n_rows, out->k, out->v, tok, c.n_layers,
                    c.n_kv_heads, c.head_dim, h->rope, c.max_pos, h->err, s);
    launch_tokens(segs, qt, pool->tokens, h->tokens, s);
    return check_cuda(h, "blend_assemble");
}

extern "C" int blend_prefill(blend_handle* h, int32_t n_req, const blend_request* reqs,
                             const blend_pool* pool, const blend_outputs* out, void* stream) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    std::vector<ReqInfo> info;
    int rc = validate_batch(h, n_req, reqs, pool, out, &info);
    if (rc != BLEND_OK) return rc;
    NvtxRange call_range("blend_prefill");
    const blend_model_cfg& c = h->cfg;
    cudaStream_t s = (cudaStream_t)stream;
    const int mode = reqs[0].mode;

    // ---- batch layout
    BatchDesc bd;
    memset(&bd, 0, sizeof bd);
    bd.n_req = n_req;
    int tok = 0, nc = 0, qo = 0, M_max = 0;
    int M_stage[3] = {0, 0, 0};  // most rows of each stage over the batch (launch sizes)
    for (int r = 0; r < n_req; ++r) {
        bd.r[r] = ReqDesc{tok, info[r].P, info[r].n_c, info[r].Q, nc, qo};
        tok += info[r].N;
        nc += info[r].n_c;
        qo += info[r].Q;
        M_max += info[r].max_rows;
        for (int st = 0; st < 3; ++st) M_stage[st] += info[r].stage_rows[st] + info[r].Q;
    }
    const int nc_total = nc;
    const size_t layer_elems = (size_t)tok * c.n_kv_heads * c.head_dim;
    const size_t es = elem_size(c.dtype);

    // ---- 1. cache preparation (all layers) and token ids
    const bool host_pool = pool->location == BLEND_POOL_HOST;
    if (!host_pool) {
        ProfScope ps(h, PROF_ASSEMBLE, s);
        rc = blend_assemble(h, n_req, reqs, pool, out, stream);
    } else {
        rc = ensure_pipeline(h);
        if (rc != BLEND_OK) return rc;
        build_segments(n_req, reqs, pool, info, hp_segs, hp_qt, &hp_tok);
        launch_tokens(hp_segs, hp_qt, pool->tokens, h->tokens, s);
        // the pool rows this batch reads, as merged runs; each segment is re-pointed at its
        // rows in the staging buffer
        std::vector<std::pair<long long, long long>> iv;
        for (int q = 0; q < hp_segs.n_seg; ++q)
            iv.push_back({hp_segs.s[q].src_row, (long long)hp_segs.s[q].src_row + hp_segs.s[q].n_rows});
        std::sort(iv.begin(), iv.end());
        hp_runs.clear();
        long long staged = 0;
        for (auto& a : iv) {
            if (!hp_runs.empty() && a.first <= hp_runs.back().end) {
                if (a.second > hp_runs.back().end) {
                    staged += a.second - hp_runs.back().end;
                    hp_runs.back().end = a.second;
                }
            } else {
                hp_runs.push_back(Run{a.first, a.second, staged});
                staged += a.second - a.first;
            }
        }
        if (staged > h->lim.max_tokens)
            return fail(h, BLEND_ENOMEM, "%lld pool rows to stage > max_tokens %d", staged, h->lim.max_tokens);
        hp_staged = staged;
        for (int q = 0; q < hp_segs.n_seg; ++q) {
            const long long src = hp_segs.s[q].src_row;
            const Run* run = &hp_runs[0];
            for (const Run& x : hp_runs)
                if (x.start <= src && src < x.end) run = &x;
            hp_segs.s[q].src_row = (int32_t)(run->stage + (src - run->start));
        }
        cudaEventRecord(h->ev_start, s);
        cudaStreamWaitEvent(h->side, h->ev_start, 0);
        for (int l = 0; l < c.n_layers && l < 2; ++l) stage_layer_copy(h, pool, l);
        rc = check_cuda(h, "blend_prefill (pool loading)");
    }
    if (rc != BLEND_OK) return rc;

    // ---- 2. stage-0 rows
    StageDesc st0{h->set[0], h->set_n[0], 0};
    int n_stage = 1;
    int stage_layer[3] = {0, 1 << 30, 1 << 30};
    if (mode == BLEND_SEL_EXT) {
        SelectBatch sb;
        memset(&sb, 0, sizeof sb);
        sb.n_job = n_req;
        sb.window = reqs[0].window;
        sb.tau = reqs[0].tau;
        sb.budget_mode = reqs[0].budget_mode;
        sb.rule = reqs[0].group_rule;
        sb.tau_smooth = reqs[0].tau_smooth;
        sb.tau_cover_bp = reqs[0].tau_cover_bp;
        sb.max_span = reqs[0].max_span;
        int max_n = 0;
        for (int r = 0; r < n_req; ++r) {
            sb.j[r] = SelectJob{reqs[r].scores, nullptr, h->set[0] + bd.r[r].nc_off, h->set_n[0] + r,
                                info[r].n_c, info[r].P, info[r].B, bd.r[r].nc_off, info[r].cap};
            max_n = info[r].n_c > max_n ? info[r].n_c : max_n;
        }
        ProfScope ps(h, PROF_SELECT, s);
        launch_select(sb, h->rank, h->rank_keys, max_n, s);
    } else if (mode == BLEND_SEL_HKVD) {
        st0.iota = 1;
        n_stage = 3;
        stage_layer[1] = 1;
        stage_layer[2] = 2;
    } else if (mode == BLEND_SEL_FULL) {
        st0.iota = 2;
    } else if (mode == BLEND_SEL_EPIC) {
        static thread_local EpicTable et;
        et.n_run = 0;
        et.n_req = n_req;
        for (int r = 0; r < n_req; ++r) {
            int off = 0, cnt = 0;
            for (int j = 0; j < reqs[r].n_chunks; ++j) {
                const int L = pool->entry_len[reqs[r].chunk_ids[j]];
                const int m = reqs[r].epic_m < L ? reqs[r].epic_m : L;
                if (m > 0) {
                    et.start[et.n_run] = info[r].P + off;
                    et.count[et.n_run] = m;
                    et.out[et.n_run] = bd.r[r].nc_off + cnt;
                    ++et.n_run;
                }
                cnt += m;
                off += L;
            }
            et.req_n[r] = cnt;
        }
        launch_epic_set(et, h->set[0], h->set_n[0], s);
    } else {
        n_stage = reqs[0].n_stages;
        for (int sidx = 0; sidx < n_stage; ++sidx) {
            stage_layer[sidx] = reqs[0].stage_layer[sidx];
            for (int r = 0; r < n_req; ++r) {
                if (reqs[r].stage_n[sidx] > 0)
                    cudaMemcpyAsync(h->set[sidx] + bd.r[r].nc_off, reqs[r].stage_pos[sidx],
                                    (size_t)reqs[r].stage_n[sidx] * 4, cudaMemcpyDeviceToDevice, s);
                launch_fill_i32(h->set_n[sidx] + r, reqs[r].stage_n[sidx], 1, s);
            }
        }
    }
    const bool focus = reqs[0].focus_bp > 0;
    static thread_local FocusTable ft;
    int max_nc = 0;
    if (focus) {
        n_stage = 2;
        stage_layer[1] = reqs[0].focus_layer;
        ft.n_req = n_req;
        int ci = 0;
        for (int r = 0; r < n_req; ++r) {
            ft.chunk0[r] = ci;
            ft.n_chunks[r] = reqs[r].n_chunks;
            int off = 0;
            for (int j = 0; j < reqs[r].n_chunks; ++j, ++ci) {
                const int L = pool->entry_len[reqs[r].chunk_ids[j]];
                ft.start[ci] = info[r].P + off;
                ft.len[ci] = L;
                off += L;
            }
            max_nc = info[r].n_c > max_nc ? info[r].n_c : max_nc;
        }
    }
    int cur = 0;
    {
        ProfScope ps(h, PROF_PLAN, s);
        launch_plan(bd, st0, h->plan[0].row_pos, h->plan[0].row_tok, h->plan[0].row_req, h->row_src,
                    h->pos2row, h->plan[0].M, h->plan[0].req_row_end, nullptr, nullptr, h->err, s);
        launch_embed(c.dtype, h->w.embed, h->tokens, h->plan[0].row_tok, h->x, c.hidden, c.vocab,
                     h->plan[0].M, M_max, h->err, s);
    }

    const bool checks = mode == BLEND_SEL_HKVD || mode == BLEND_SEL_FORCED;
    if (checks) {
        cudaMemsetAsync(h->dev[0], 0, (size_t)nc_total * 4, s);
        cudaMemsetAsync(h->dev[1], 0, (size_t)nc_total * 4, s);
    }
    // ---- 3. layers
    h->xn_scaled = false;
    float* x = h->x;
    float* x_alt = h->x2;
    int M_cur = M_stage[0];  // bound of the current stage's rows (sizes the launches)
    for (int l = 0; l < c.n_layers; ++l) {
        char layer_name[24];
        snprintf(layer_name, sizeof layer_name, "layer %d", l);
        NvtxRange layer_range(layer_name);
        void* kc = (char*)out->k + (size_t)l * layer_elems * es;
        void* vc = (char*)out->v + (size_t)l * layer_elems * es;
        const Plan& p = h->plan[cur];
        if (host_pool) {
            // this layer's pool rows have landed in staging buffer l % 2: realign them into the
            // blended cache, free the buffer, and start the copy of layer l + 2 into it
            cudaStreamWaitEvent(s, h->ev_layer[l], 0);
            {
                ProfScope ps(h, PROF_ASSEMBLE, s);
                launch_assemble(c.dtype, hp_segs, h->stage[2 * (l & 1)], h->stage[2 * (l & 1) + 1], hp_staged, kc, vc,
                                tok, 1, c.n_kv_heads, c.head_dim, h->rope, c.max_pos, h->err, s, 0);
            }
            cudaEventRecord(h->ev_free[l & 1], s);
            if (l + 2 < c.n_layers) {
                cudaStreamWaitEvent(h->side, h->ev_free[l & 1], 0);
                stage_layer_copy(h, pool, l + 2);
            }
        }
        float* dev = (checks && (l == 1 || l == 2)) ? h->dev[l - 1] : nullptr;
        layer_kv(h, l, x, p, p.row_req, M_cur, bd, kc, vc, dev, reqs[0].dev_mode, 0, s);
        int new_stage = -1;
        for (int sidx = 1; sidx < n_stage; ++sidx)
            if (stage_layer[sidx] == l) new_stage = sidx;
        if (new_stage > 0) {
            if (mode == BLEND_SEL_HKVD) {
                SelectBatch sb;
                memset(&sb, 0, sizeof sb);
                sb.n_job = n_req;
                int max_n = 0;
                if (new_stage == 1) {
                    sb.window = 1;
                    sb.tau = 1;
                    sb.budget_mode = BLEND_BUDGET_CANDIDATE;
                } else {
                    ProfScope ps(h, PROF_SELECT, s);
                    launch_set_mask(bd, h->set[1], h->set_n[1], h->mask, s);
                    sb.window = reqs[0].window;
                    sb.tau = reqs[0].tau;
                    sb.budget_mode = reqs[0].budget_mode;
                }
                for (int r = 0; r < n_req; ++r) {
                    const int budget = new_stage == 1 ? info[r].k1 : info[r].B;
                    sb.j[r] = SelectJob{h->dev[new_stage - 1] + bd.r[r].nc_off,
                                        new_stage == 1 ? nullptr : h->mask + bd.r[r].nc_off,
                                        h->set[new_stage] + bd.r[r].nc_off, h->set_n[new_stage] + r,
                                        info[r].n_c, info[r].P, budget, bd.r[r].nc_off};
                    max_n = info[r].n_c > max_n ? info[r].n_c : max_n;
                }
                ProfScope ps(h, PROF_SELECT, s);
                launch_select(sb, h->rank, h->rank_keys, max_n, s);
            } else if (focus) {
                // the query rows' attention at this layer, per chunk: their q (into the free
                // attention-output buffer), column means over chunk tokens, then the filter
                ProfScope ps(h, PROF_SELECT, s);
                launch_gather_qlast(c.dtype, h->q, h->lim.max_rows, c.n_q_heads / c.n_kv_heads, c.n_kv_heads,
                                    c.head_dim, bd, h->plan[cur].req_row_end, h->o, qo, s);
                launch_aux_scores(c.dtype, h->o, kc, bd, c.n_q_heads, c.n_kv_heads, c.head_dim, qo, max_nc,
                                  h->aux_stats, tc_score_spans(h->lim.max_tokens), h->dev[0], h->err, h->use_tc != 0, s);
                launch_focus_filter(bd, ft, h->dev[0], reqs[0].focus_bp, h->set[0], h->set_n[0], h->set[1],
                                    h->set_n[1], s);
            }
            ProfScope ps(h, PROF_PLAN, s);
            StageDesc st{h->set[new_stage], h->set_n[new_stage], 0};
            Plan& np = h->plan[1 - cur];
            launch_plan(bd, st, np.row_pos, np.row_tok, np.row_req, h->row_src, h->pos2row, np.M,
                        np.req_row_end, h->plan[cur].row_tok, h->plan[cur].M, h->err, s);
            // the new set is at most as large as its stage's bound (the focus filter only
            // removes rows of the current stage)
            if (!focus) M_cur = M_stage[new_stage];
            launch_gather(x, (long long)c.hidden * 4, h->lim.max_rows, h->row_src, np.M, M_cur, x_alt, h->err, s);
            {
                // q is stored per kv head: compact each head's slab of [rows][group][d]
                const int group = c.n_q_heads / c.n_kv_heads;
                const size_t slab = (size_t)h->lim.max_rows * group * c.head_dim * es;
                for (int g = 0; g < c.n_kv_heads; ++g)
                    launch_gather((const char*)h->q + g * slab, (long long)group * c.head_dim * es,
                                  h->lim.max_rows, h->row_src, np.M, M_cur, (char*)h->q2 + g * slab, h->err, s);
            }
            float* tx = x;
            x = x_alt;
            x_alt = tx;
            void* tq = h->q;
            h->q = h->q2;
            h->q2 = tq;
            cur = 1 - cur;
        }
        if (l == c.n_layers - 1 && out->q_last)
            launch_gather_qlast(c.dtype, h->q, h->lim.max_rows, c.n_q_heads / c.n_kv_heads, c.n_kv_heads,
                                c.head_dim, bd, h->plan[cur].req_row_end, out->q_last, qo, s);
        layer_rest(h, l, x, h->plan[cur], n_req, M_cur, kc, vc, tok, s, true);
    }
    // ---- 4. final norm of the query rows
    ProfScope ps_final(h, PROF_FINAL, s);
    launch_final_norm(c.dtype, x, h->w.final_norm, out->hidden, c.hidden, c.rms_eps, bd,
                      h->plan[cur].req_row_end, s);
    // ---- 5. sets and deviations out
    int last = 0;
    for (int sidx = 1; sidx < n_stage; ++sidx)
        if (stage_layer[sidx] < c.n_layers) last = sidx;
    if (out->sel || out->n_sel) {
        if (last == 0 && st0.iota)
            launch_copy_sets(bd, nullptr, nullptr, out->sel, out->n_sel, s);  // every chunk row
        else
            launch_copy_sets(bd, h->set[last], h->set_n[last], out->sel, out->n_sel, s);
    }
    if ((out->c1 || out->n_c1) && mode == BLEND_SEL_HKVD && stage_layer[1] < c.n_layers)
        launch_copy_sets(bd, h->set[1], h->set_n[1], out->c1, out->n_c1, s);
    if (checks && out->dev1) cudaMemcpyAsync(out->dev1, h->dev[0], (size_t)nc_total * 4, cudaMemcpyDeviceToDevice, s);
    if (checks && out->dev2) cudaMemcpyAsync(out->dev2, h->dev[1], (size_t)nc_total * 4, cudaMemcpyDeviceToDevice, s);
    return finish(h, "blend_prefill");
}

extern "C" int aux_attention_scores(blend_handle* h, int32_t n_req, const blend_request* reqs, const blend_pool* pool,
                         const blend_outputs* out, float* scores, void* stream) {
    if (!h) return fail(nullptr, BLEND_EINVAL, "handle is NULL");
    if (!out || !out->q_last || !scores) return fail(h, BLEND_EINVAL, "out->q_last and scores are required");
    std::vector<ReqInfo> info;
    int rc = validate_batch(h, n_req, reqs, pool, out, &info, false);
    if (rc != BLEND_OK) return rc;
    const blend_model_cfg& c = h->cfg;
    BatchDesc bd;
    memset(&bd, 0, sizeof bd);
    bd.n_req = n_req;
    int tok = 0, nc = 0, qo = 0, max_nc = 0;
    for (int r = 0; r < n_req; ++r) {
        bd.r[r] = ReqDesc{tok, info[r].P, info[r].n_c, info[r].Q, nc, qo};
        tok += info[r].N;
        nc += info[r].n_c;
        qo += info[r].Q;
        max_nc = info[r].n_c > max_nc ? info[r].n_c : max_nc;
    }
    if (qo > h->lim.max_rows) return fail(h, BLEND_ENOMEM, "%d query rows > limit %d", qo, h->lim.max_rows);
    const size_t layer_elems = (size_t)tok * c.n_kv_heads * c.head_dim;
    const void* k_last = (const char*)out->k + (size_t)(c.n_layers - 1) * layer_elems * elem_size(c.dtype);
    launch_aux_scores(c.dtype, out->q_last, k_last, bd, c.n_q_heads, c.n_kv_heads, c.head_dim, qo, max_nc,
                      h->aux_stats, tc_score_spans(h->lim.max_tokens), scores, h->err, h->use_tc != 0,
                      (cudaStream_t)stream);
    return check_cuda(h, "aux_attention_scores");
}
