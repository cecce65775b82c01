/*
 * blend.h - C ABI of libblend: selective KV-recompute ("blended") prefill for RAG
 * on one GB300 (sm_103a).
 *
 * The method (CacheBlend blog, "Selective KV recompute" and "Picking the tokens to
 * recompute"; CacheClip blog, "6. How CacheClip works"; SpecCache notes, 2.2):
 * precomputed per-chunk KV caches, each encoded behind one shared prefix, are
 * concatenated with a single prefix copy and their keys rotated to their new
 * positions; a subset of chunk rows (plus the query) is then recomputed on every
 * layer against the full blended KV and written back into it.  The problem the
 * calls solve is the pages' own: given precomputed chunk caches, a query and a
 * recompute ratio, hand over a finished KV cache and the query's first-token
 * state (CacheBlend blog, "The system": the engine receives a finished KV cache).
 *
 * Conventions
 *   - Every call returns an int status (BLEND_OK or a negative BLEND_E* code).
 *     Arguments are validated on the host before anything is launched; a call that
 *     fails validation launches nothing and leaves every buffer untouched.
 *   - Tensors are caller-owned device pointers (allocated by the caller, e.g. with
 *     PyTorch).  The library never frees or reallocates them.  "host" in a comment
 *     marks a host pointer.  Only the workspace given to blend_init is used as
 *     scratch by the handle; it must stay allocated until blend_destroy.
 *   - All work is enqueued on the caller's stream (`stream` is a cudaStream_t;
 *     NULL is the legacy default stream).  Calls do not synchronise the device.
 *     Counts produced on the device (set sizes) stay on the device.
 *   - Row-major layouts.  Per-layer caches are [layer][token][kv_head][head_dim].
 *     The storage type of weights, activations and caches is the model's dtype
 *     (BLEND_F32 or BLEND_BF16); accumulation is fp32.
 *   - Positions are absolute positions in the blended sequence of one request:
 *     prefix rows 0..P-1, chunk rows P..P+N_c-1, query rows P+N_c..N-1.
 *   - Errors from CUDA are returned as BLEND_ECUDA; blend_last_error() gives the
 *     text.  A bounded device-side wait that expired sets BLEND_ETIMEOUT.
 */
#ifndef BLEND_H
#define BLEND_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------- */
#define BLEND_OK 0
#define BLEND_EINVAL (-1)       /* bad argument (null pointer, bad size or mode) */
#define BLEND_ENOMEM (-2)       /* workspace too small for the request */
#define BLEND_ECUDA (-3)        /* a CUDA call or launch failed */
#define BLEND_EMISS (-4)        /* a requested pool entry has no cache (fetch miss) */
#define BLEND_ETIMEOUT (-5)     /* a bounded device wait expired */
#define BLEND_EDEVICE (-6)      /* a device-side check failed (error word set) */
#define BLEND_EUNSUPPORTED (-7) /* shape or dtype the library does not handle */

/* ---- enums ----------------------------------------------------------------- */
#define BLEND_F32 0
#define BLEND_BF16 1

#define BLEND_SEL_EXT 0    /* one set for all layers from external scores */
#define BLEND_SEL_HKVD 1   /* KV-deviation gradual filtering (checks on layers 1 and 2) */
#define BLEND_SEL_FORCED 2 /* caller-given stage sets */
#define BLEND_SEL_FULL 3   /* recompute every row (full prefill through the same path) */
#define BLEND_SEL_EPIC 4   /* static: the first epic_m tokens of every chunk (EPIC, as SpecCache
                            * describes it) */

#define BLEND_BUDGET_FINAL 0     /* at most ceil(rho*N_c) rows after grouping */
#define BLEND_BUDGET_CANDIDATE 1 /* ceil(rho*N_c) candidates, then grouping */

/* EXT selection rule applied after TopK: CacheClip window grouping (window, tau) or
 * SpecCache span completion (tau_smooth, tau_cover_bp, max_span, cap_bp). */
#define BLEND_GROUP_WINDOW 0
#define BLEND_GROUP_SPAN 1

#define BLEND_POOL_DEVICE 0
#define BLEND_POOL_HOST 1

#define BLEND_DEV_KV 0 /* deviation = |k-k'|^2 + |v-v'|^2 */
#define BLEND_DEV_V 1  /* deviation = |v-v'|^2 */

#define BLEND_MAX_BATCH 64
#define BLEND_MAX_CHUNKS 1024 /* chunks over all requests of one call */
#define BLEND_MAX_WINDOW 64
#define BLEND_MAX_SPAN 64              /* longest span of the span rule */
#define BLEND_MAX_ALIGN_TARGETS 131072 /* target tokens of one align_expand call */
#define BLEND_GU_BLOCK 16 /* gate/up row interleave of w_gu, see blend_weights */

/* ---- model ----------------------------------------------------------------- */
typedef struct {
    int32_t n_layers;
    int32_t hidden;     /* H */
    int32_t n_q_heads;  /* hq */
    int32_t n_kv_heads; /* hkv; hq % hkv == 0 */
    int32_t head_dim;   /* d: 64 or 128 */
    int32_t ffn;        /* F: multiple of BLEND_GU_BLOCK */
    int32_t vocab;
    int32_t dtype;      /* BLEND_F32 | BLEND_BF16 */
    double rope_theta;  /* RoPE base; pairs (i, i+d/2), angle pos * theta^(-2i/d) */
    float rms_eps;
    int32_t max_pos;    /* positions 0..max_pos-1 are supported (RoPE table size) */
} blend_model_cfg;

/* Device pointers to the stacked per-layer weights (non-owning; they must stay valid
 * while the handle is used).  Linear weights are [out_features][in_features]. */
typedef struct {
    const void* embed;      /* [vocab][H] */
    const void* attn_norm;  /* [L][H] RMSNorm gain before attention */
    const void* w_qkv;      /* [L][(hq+2*hkv)*d][H]: rows of q heads, then k heads, then v heads */
    const void* w_o;        /* [L][H][hq*d] */
    const void* mlp_norm;   /* [L][H] */
    const void* w_gu;       /* [L][2F][H]: rows 32j..32j+15 = gate rows 16j..16j+15,
                               rows 32j+16..32j+31 = up rows 16j..16j+15 */
    const void* w_down;     /* [L][H][F] */
    const void* final_norm; /* [H] */
} blend_weights;

/* Capacity a handle is built for (sizes its workspace). */
typedef struct {
    int32_t max_rows;   /* rows recomputed in one layer, summed over a batch */
    int32_t max_tokens; /* blended tokens (sum of N over a batch) */
    int32_t max_chunk_rows; /* N_c of one request */
    int32_t max_batch;  /* requests per blend_prefill call (<= BLEND_MAX_BATCH) */
} blend_limits;

typedef struct blend_handle blend_handle;

/* ---- chunk-KV pool --------------------------------------------------------- */
/* Offline precompute (CacheClip "4.1 KV Cache Calibration with Shared Prefix"):
 * entry c holds [prefix + chunk_c] encoded at positions 0..P+L_c-1 (keys after RoPE).
 * Entries are packed along rows: entry c occupies rows entry_row[c]..+P+L_c. */
typedef struct {
    int32_t n_entries;
    int32_t prefix_len;        /* P */
    const int32_t* entry_len;  /* host [n_entries]: chunk length L_c (without prefix) */
    const int64_t* entry_row;  /* host [n_entries]: first row of each entry */
    const uint8_t* present;    /* host [n_entries] or NULL; 0 = cache missing -> BLEND_EMISS */
    int64_t n_rows;            /* rows per layer in k, v, tokens */
    const void* k;             /* device [L][n_rows][hkv][d] */
    const void* v;             /* device [L][n_rows][hkv][d] */
    const int32_t* tokens;     /* device [n_rows] token id of each row */
    /* BLEND_POOL_DEVICE: k, v, tokens in device memory.  BLEND_POOL_HOST: in pinned host
     * memory (cudaHostAlloc / cudaHostRegister).  blend_prefill then copies each layer's
     * pool rows into one of two staging buffers with the copy engines on a side stream,
     * two layers ahead, and realigns them into the blended cache just before that layer's
     * recompute, which waits only for its own layer (CacheBlend blog, "Making the
     * recompute free": loading and recompute overlap).  The pool rows one call reads must
     * fit max_tokens (BLEND_ENOMEM otherwise). */
    int32_t location;
} blend_pool;

/* ---- one request ----------------------------------------------------------- */
typedef struct {
    int32_t n_chunks;
    const int32_t* chunk_ids;    /* host [n_chunks]: pool entries in request order */
    int32_t query_len;           /* Q >= 1 */
    const int32_t* query_tokens; /* device [Q] */
    int32_t mode;                /* BLEND_SEL_* */
    int32_t rho_bp;              /* recompute ratio of chunk rows, basis points (0..10000) */
    int32_t r1_bp;               /* HKVD: first-stage ratio, basis points (>= rho_bp) */
    int32_t window;              /* grouping window w (1..BLEND_MAX_WINDOW); 1 = none */
    int32_t tau;                 /* grouping density threshold (1..w) */
    int32_t budget_mode;         /* BLEND_BUDGET_* */
    int32_t dev_mode;            /* BLEND_DEV_* */
    const float* scores;         /* EXT: device [N_c] per chunk-row score (higher = recompute) */
    /* FORCED: stage s applies from layer stage_layer[s] (stage 0 from layer 0);
     * stage_pos[s] = device sorted absolute positions in [P, P+N_c), stage_n[s] of them. */
    int32_t n_stages;
    int32_t stage_layer[3];
    const int32_t* stage_pos[3];
    int32_t stage_n[3];
    /* EXT only: BLEND_GROUP_WINDOW (0, the fields window/tau above) or BLEND_GROUP_SPAN
     * (SpecCache 2.3: spans of smooth importance, completed when covered enough). */
    int32_t group_rule;
    float tau_smooth;            /* SPAN: merge while the relative change is below this (0.4) */
    int32_t tau_cover_bp;        /* SPAN: complete a span at this coverage, basis points (7000) */
    int32_t max_span;            /* SPAN: longest span, 1..BLEND_MAX_SPAN (16) */
    int32_t cap_bp;              /* SPAN + CANDIDATE: most rows kept after completion, basis
                                  * points of N_c (rho_bp..10000); FINAL: the budget is the cap */
    int32_t epic_m;              /* EPIC: tokens recomputed at the start of every chunk (>= 0) */
    /* Early termination for unfocused chunks (Cache-Craft notes, 3.2.2), EXT and EPIC modes:
     * with focus_bp > 0, at layer focus_layer (after its K/V projection) each chunk's share
     * of the query rows' attention is measured (mean over query rows and heads of the
     * softmax weight on its tokens, summed over the chunk); chunks whose share of the total
     * is below focus_bp basis points stop being recomputed from that layer's attention on.
     * The set after the filter is what out->sel receives. */
    int32_t focus_layer;
    int32_t focus_bp;
} blend_request;

/* Outputs of a batch.  Request r owns tokens tok_r .. tok_r+N_r-1 of k, v with
 * tok_r = sum of N over earlier requests; chunk rows nc_r .. of sel/dev with
 * nc_r = sum of N_c over earlier requests; query rows q_r .. of hidden. */
typedef struct {
    void* k;           /* device [L][sum N][hkv][d]: the finished blended cache */
    void* v;           /* device [L][sum N][hkv][d] */
    void* hidden;      /* device [sum Q][H]: final RMSNorm of the query rows (model dtype) */
    int32_t* sel;      /* device [sum N_c] or NULL: set used from the last stage on */
    int32_t* n_sel;    /* device [n_req] or NULL */
    int32_t* c1;       /* device [sum N_c] or NULL: HKVD first-stage set */
    int32_t* n_c1;     /* device [n_req] or NULL */
    float* dev1;       /* device [sum N_c] or NULL: deviation at layer 1 (0 = not checked) */
    float* dev2;       /* device [sum N_c] or NULL: deviation at layer 2 */
    void* q_last;      /* device [sum Q][hq][d] or NULL: the query rows' last-layer q after RoPE
                        * (model dtype), read by aux_attention_scores */
} blend_outputs;

/* ---- handle ---------------------------------------------------------------- */
/* Bytes of device workspace a handle needs for `cfg` and `lim`. 0 on bad input. */
size_t blend_workspace_size(const blend_model_cfg* cfg, const blend_limits* lim);

/* Create a handle.  `workspace` (device, >= blend_workspace_size bytes, 256-byte
 * aligned) is owned by the caller and used by the handle until blend_destroy.
 * Builds the RoPE table (angles in fp64, cos/sin stored fp32) on `stream`. */
int blend_init(const blend_model_cfg* cfg, const blend_weights* w, const blend_limits* lim,
               void* workspace, size_t ws_bytes, void* stream, blend_handle** out);
int blend_destroy(blend_handle* h);
/* Text of the last error on this handle (or of the last handle-less call when h is NULL). */
const char* blend_last_error(const blend_handle* h);
/* Synchronises `stream`, then returns BLEND_OK, or BLEND_EDEVICE / BLEND_ETIMEOUT if a
 * device-side check of an earlier call on this handle failed (bad positions in a
 * caller-given set, an out-of-range shift, an expired bounded wait).  Clears the word. */
int blend_device_status(blend_handle* h, void* stream);
/* Bounded device-side wait (the pages have no counterpart): enqueues on the stream a wait
 * until *flag (device int32, 4-byte aligned) is nonzero, polling at most max_polls times
 * with a short sleep (~64 ns) between polls.  If the flag stays 0 the handle's error word
 * gets BLEND_ETIMEOUT and the wait ends: blend_device_status then returns BLEND_ETIMEOUT
 * (and clears the word), and the handle and the CUDA context stay usable.  Every
 * device-side wait inside the library's kernels is bounded the same way; this call lets
 * a caller (or a test) exercise that timeout path on purpose, without a trap or a hang.
 * The flag must be set by something that does not need the GPU's SMs to progress (a
 * copy, or the host through mapped memory); a kernel queued behind this wait on the
 * same stream never sets it.
 * Errors: BLEND_EINVAL for a NULL handle or flag, an unaligned flag, or max_polls
 * outside 0..BLEND_MAX_WAIT_POLLS (nothing is launched). */
#define BLEND_MAX_WAIT_POLLS (1ll << 24)
int blend_wait_flag(blend_handle* h, const int32_t* flag, int64_t max_polls, void* stream);

/* Turns the tcgen05 tensor-core GEMM/attention on (1) or off (0) for a bf16 handle;
 * off uses the CUDA-core kernels.  Returns the setting in effect (0 for fp32 handles
 * and on GPUs without tcgen05). */
int blend_set_tensor_cores(blend_handle* h, int on);

/* Allocation-free variant of topk_select_dilate (same arguments, same result, no
 * handle).  The pages have no counterpart: this call exists for callers that cannot
 * allocate device memory when they select tokens - for example a serving loop that
 * reserves all HBM for its KV pool at start-up, or one that must not call cudaMalloc /
 * cudaFree on its hot path because those calls can synchronise the device or fail
 * under fragmentation.  The call uses fixed scratch arrays in device memory (32768 ranks
 * and 32768 sorted 64-bit keys, 384 KB) that every GPU which loads the library holds
 * until the process exits; it never allocates or frees memory.
 *   - n above 32768 is rejected with BLEND_EINVAL (nothing is launched).
 *   - Every call looks up the arrays' device addresses on the current device (a
 *     host-side query; the first one on a device may load the library's device code, so
 *     make the first call on each device before any stream capture).
 *   - Every call shares the one set of arrays: calls whose work overlaps on the GPU (on
 *     different streams, or on several host threads) race and give wrong sets.
 *     Each call rewrites every scratch entry it reads, so nothing needs clearing.
 * Errors: as topk_select_dilate; the text is in blend_last_error(NULL). */
int topk_select_dilate_noalloc(const float* scores, int32_t n, int32_t base, int32_t budget,
                               int32_t window, int32_t tau, int32_t budget_mode,
                               const uint8_t* allowed, int32_t* idx_out, int32_t* n_out,
                               void* stream);

/* ---- tracing --------------------------------------------------------------- */
/* Per-stage timing with CUDA events recorded on the caller's stream around each stage
 * of blend_prefill / selective_layer (assemble, select, plan_gather, rmsnorm,
 * gemm_qkv, rope_kv, attention, gemm_o, gemm_gate_up, gemm_down, final_norm).
 * blend_profile(h, 1) clears the record and starts recording; (h, 0) stops.
 * blend_profile_stages(h, mask) does the same for only the stages whose bit
 * (1 << stage index, the order above) is set in mask (0 stops): every recorded stage
 * adds an event pair on the stream, so timing one stage this way disturbs the step
 * least.  blend_profile_read waits for the recorded events, writes per-stage total ms and
 * kernel launch counts for the first n stages, clears the record and returns the
 * number of stages.  blend_launch_count() is the process-wide number of kernels the
 * library has launched.  Errors: BLEND_EINVAL for a NULL handle. */
int blend_profile(blend_handle* h, int enable);
int blend_profile_stages(blend_handle* h, uint32_t stage_mask);
int blend_profile_read(blend_handle* h, double* ms, int64_t* launches, int32_t n);
const char* blend_profile_name(int32_t i);
int64_t blend_launch_count(void);

/* ---- step calls ------------------------------------------------------------ */

/* RoPE realignment (CacheBlend blog, "Selective KV recompute", footnote on positional
 * correctness: moving a chunk multiplies its keys by a rotation once).  For each
 * layer l < n_layers and row i < n_rows: dst[l][i] = R(delta[i]) src[l][i], where
 * rows are [hkv][d] and delta (device [n_rows] int32, |delta| < max_pos) is the
 * position shift.  src and dst layer strides are in rows.  src == dst is allowed. */
int rope_realign(blend_handle* h, const void* k_src, void* k_dst, int32_t n_rows,
                 const int32_t* delta, int32_t n_layers, int64_t src_layer_rows,
                 int64_t dst_layer_rows, void* stream);

/* Cache preparation for a batch (CacheClip blog 6.1 and paper 4.1): writes out->k,
 * out->v for every layer: prefix rows from the first chunk's entry only, chunk j of
 * request r at positions P+off_j.. with keys rotated by off_j (values copied).  Query
 * rows are left as they are (they are written by the first layer's recompute). */
int blend_assemble(blend_handle* h, int32_t n_req, const blend_request* reqs,
                   const blend_pool* pool, const blend_outputs* out, void* stream);

/* KV deviation (CacheBlend blog, "Selective KV recompute"): for row i < *n_rows,
 * dev[i] = sum over [hkv][d] of (k_new[i]-k_cache[pos[i]])^2 + (v_new[i]-v_cache[pos[i]])^2
 * (v only for BLEND_DEV_V), accumulated in fp32 in a fixed order.  k_new, v_new:
 * [rows][hkv][d]; caches: [n_ctx][hkv][d] (one layer); every K/V pointer 16-byte aligned.
 * n_rows is a device scalar, at most max_rows (host) rows are read.  Device-side checks:
 * a position outside 0..n_ctx-1 gives dev[i] = 0 without reading the cache, and a count
 * outside 0..max_rows is clamped; both are reported by blend_device_status as
 * BLEND_EDEVICE.  Host errors: BLEND_EINVAL for NULL or unaligned pointers, negative
 * sizes or a bad mode (nothing is launched). */
int kv_deviation(blend_handle* h, const void* k_new, const void* v_new, const void* k_cache,
                 const void* v_cache, const int32_t* pos, const int32_t* n_rows, int32_t max_rows,
                 int64_t n_ctx, int32_t mode, float* dev_out, void* stream);

/* Token selection: top-k by score then sliding-window grouping (CacheClip blog 6.3,
 * rule list and Figure 6; SpecCache 2.2 TopK).  scores: device [n] fp32 for positions
 * base..base+n-1; ranked by score descending, ties by position ascending, -0 == +0,
 * NaN last.  Candidates = top k; every window [t, t+w) with t <= n-w that starts on a
 * candidate and holds >= tau candidates joins the set.  k = min(budget, #allowed) in
 * CANDIDATE mode; in FINAL mode the largest k <= budget whose set has <= budget rows.
 * allowed: device [n] uint8 or NULL (0 = may be neither candidate nor output).
 * Writes the set ascending (absolute positions) to idx_out (device [n]) and its size to
 * *n_out (device).  Uses the handle's workspace; calls on one handle must not overlap. */
int topk_select_dilate(blend_handle* h, const float* scores, int32_t n, int32_t base,
                       int32_t budget, int32_t window, int32_t tau, int32_t budget_mode,
                       const uint8_t* allowed, int32_t* idx_out, int32_t* n_out, void* stream);

/* SpecCache selection (SpecCache notes, "2.2 Importance score estimation" TopK and
 * "2.3 Semantic span completion" with its global budget control).  scores: device [n]
 * fp32 for positions base..base+n-1, ranked as in topk_select_dilate.  Normalised
 * scores n~ = (s - min)/(max - min) (fp32, -0 as +0, NaN skipped by min/max); token i+1
 * joins token i's span while |n~(i+1) - n~(i)| / n~(i) < tau_smooth (each step one fp32
 * operation; a NaN or infinite change ends the span), at most max_span tokens per span.
 * A span joins the set when (#TopK members in it) * 10000 >= tau_cover_bp * length.
 * CANDIDATE: TopK size = budget, then at most `cap` tokens, those of highest score.
 * FINAL: the largest TopK size <= budget whose completed set has <= budget tokens
 * (`cap` unused).  Writes the set ascending (absolute positions) to idx_out (device [n])
 * and its size to *n_out (device).  n <= 32768 and within the handle's chunk-row
 * capacity; 0 <= tau_smooth (finite), 1 <= tau_cover_bp <= 10000,
 * 1 <= max_span <= BLEND_MAX_SPAN, cap >= 0, else BLEND_EINVAL.  Uses the handle's
 * workspace; calls on one handle must not overlap. */
int span_select(blend_handle* h, const float* scores, int32_t n, int32_t base, int32_t budget, int32_t cap,
                float tau_smooth, int32_t tau_cover_bp, int32_t max_span, int32_t budget_mode,
                int32_t* idx_out, int32_t* n_out, void* stream);

/* Cross-tokenizer alignment (SpecCache notes, "2.4 Cross-tokenizer alignment"): the
 * selected speculative-model tokens sel[0..*n_sel) (device, values sel_base..sel_base+
 * n_spec-1; *n_sel clamped to 0..max_sel) are expanded to every target-model token
 * a_start[i]..a_end[i]-1 (device [n_spec] each) of token i = sel[k] - sel_base; the
 * distinct target tokens are written ascending, plus out_base, to idx_out (device,
 * room for n_target) and their count to *n_out (device).  0 <= n_target <=
 * BLEND_MAX_ALIGN_TARGETS.  A selected index or a range outside its bounds is skipped
 * and reported by blend_device_status as BLEND_EDEVICE. */
int align_expand(blend_handle* h, const int32_t* sel, const int32_t* n_sel, int32_t max_sel, int32_t sel_base,
                 const int32_t* a_start, const int32_t* a_end, int32_t n_spec, int32_t n_target,
                 int32_t out_base, int32_t* idx_out, int32_t* n_out, void* stream);

/* Auxiliary-model importance scores (CacheClip blog, "6.2 Auxiliary-model-guided token
 * selection", steps 3-5, and its formula score(j) = (1/|Q|) sum over query rows i of
 * A_last[i, j]; CacheClip paper 4.2).  Call it after blend_prefill on the auxiliary model's
 * handle with the same reqs, pool and out, where out->q_last was set: each request is one
 * [prefix + chunk(s) + query] sequence, typically FORCED with an empty stage so that only
 * the query rows are computed over the chunk's cached rows.  For every request r and chunk
 * column j (the request's tokens P..P+N_c-1) writes scores[nc_r + j] = mean over its query
 * rows and the model's hq heads of the last layer's softmax weight on key j, the softmax
 * covering every key the row sees (prefix, chunks, query rows up to itself; fp32, scale
 * 1/sqrt(d)).  scores: device [sum N_c] fp32.  Deterministic (fixed summation order). */
int aux_attention_scores(blend_handle* h, int32_t n_req, const blend_request* reqs, const blend_pool* pool,
                         const blend_outputs* out, float* scores, void* stream);

/* CacheBlend's loading controller (CacheBlend blog, "Making the recompute free").  The
 * recompute delay is rho x full_prefill_s (the offline-profiled full prefill of the
 * context); the load delay is kv_bytes / load_bytes_per_s.  rho is the ratio where the
 * two are equal, raised to the quality floor floor_bp (15 % on the pages) and capped at
 * 100 %: *rho_bp = min(10000, max(floor_bp, ceil(10000 * load / full_prefill_s)))
 * (double arithmetic in that order).  Host arithmetic only; BLEND_EINVAL unless every
 * time, size and rate is positive and finite and 0 <= floor_bp <= 10000. */
int blend_ratio_controller(double full_prefill_s, double kv_bytes, double load_bytes_per_s, int32_t floor_bp,
                           int32_t* rho_bp);
/* The same estimators run backwards (CacheBlend blog, "Making the recompute free"): at
 * the floor ratio, keep the storage devices whose load delay kv_bytes / bytes_per_s[i]
 * is at most floor x full_prefill_s, and return in *best the index of the cheapest
 * (lowest cost_per_byte[i]; the lower index on a tie), or -1 if none qualifies.  Host
 * arrays of n_dev entries; host arithmetic only. */
int blend_pick_storage(double full_prefill_s, double kv_bytes, int32_t floor_bp, int32_t n_dev,
                       const double* bytes_per_s, const double* cost_per_byte, int32_t* best);

/* Row gather (CacheBlend blog, "Selective KV recompute": the layer input is reduced to
 * the selected rows): dst[i] = src[idx[i]] for i < *n (device scalar, at most max_n rows),
 * rows of row_bytes (a positive multiple of 16; src, dst 16-byte aligned); src holds
 * src_rows rows.  Device-side checks: an index outside 0..src_rows-1 leaves dst[i]
 * untouched and a count outside 0..max_n is clamped; both are reported by
 * blend_device_status(h) as BLEND_EDEVICE.  The handle is used only for that error word.
 * Host errors: BLEND_EINVAL (nothing is launched). */
int gather_rows(blend_handle* h, const void* src, int64_t row_bytes, int64_t src_rows, const int32_t* idx,
                const int32_t* n, int32_t max_n, void* dst, void* stream);

/* KV scatter (CacheClip blog 6.3: the global KV cache entries are overwritten):
 * k_cache[pos[i]] = k_new[i], v_cache[pos[i]] = v_new[i] for i < *n (one layer; caches
 * [n_ctx][hkv][d], rows [hkv][d]; 16-byte aligned pointers).  Device-side checks: a
 * position outside 0..n_ctx-1 is not written and a count outside 0..max_n is clamped;
 * both are reported by blend_device_status as BLEND_EDEVICE.  Host errors: BLEND_EINVAL. */
int scatter_kv(blend_handle* h, const void* k_new, const void* v_new, const int32_t* pos,
               const int32_t* n, int32_t max_n, int64_t n_ctx, void* k_cache, void* v_cache, void* stream);

/* One selective decoder layer (CacheBlend blog, "Selective KV recompute": mask the
 * input to the selected rows, project Q/K/V, expand K/V with the reused rows, run
 * attention and the rest of the layer) for one request.
 * x: device fp32 [max_n][H] residual rows (in/out); the first *n of them (n: device
 * scalar, so a set size produced on the device needs no host round trip) are the rows at
 * strictly ascending positions pos (device [*n], each in 0..n_ctx-1).  k_cache, v_cache:
 * this layer's [n_ctx][hkv][d]; their rows pos[i] are overwritten with the fresh K/V
 * before attention.  dev_out: device [max_n] or NULL, the deviation of each row against
 * the cache before the overwrite.  max_n (host) <= the handle's max_rows bounds *n and
 * sizes the launches; n_ctx <= max_tokens.  Device-side checks: a count above
 * min(max_n, n_ctx) is clamped and a position out of range or out of order is replaced by
 * a valid one; both are reported by blend_device_status as BLEND_EDEVICE. */
int selective_layer(blend_handle* h, int32_t layer, float* x, const int32_t* pos, const int32_t* n,
                    int32_t max_n, void* k_cache, void* v_cache, int32_t n_ctx, float* dev_out,
                    int32_t dev_mode, void* stream);

/* The whole blended prefill for a batch of requests (all layers; assemble, select,
 * recompute, final norm).  Rows of all requests share each weight pass. */
int blend_prefill(blend_handle* h, int32_t n_req, const blend_request* reqs,
                  const blend_pool* pool, const blend_outputs* out, void* stream);

/* SpecCache 2.2 importance scores: out[i] = (1/n_layers) * sum_l ||hidden[i][l]||_2
 * for hidden device [n][n_layers][dim] of dtype (BLEND_F32 | BLEND_BF16); out fp32.
 * BLEND_EINVAL for a NULL pointer, n < 0, dim < 1, n_layers outside [1, 4096] or
 * another dtype.  Any alignment of hidden is accepted (16-byte aligned rows read faster). */
int importance_scores(const void* hidden, int32_t n, int32_t n_layers, int32_t dim,
                      int32_t dtype, float* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* BLEND_H */
