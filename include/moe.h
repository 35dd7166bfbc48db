/*
 * moe.h -- C ABI of libmoe.so: forward pass of a top-k routed Mixture-of-Experts
 * SwiGLU FFN layer with optional shared experts, on one B300 GPU (sm_103a).
 *
 * The operation is the one defined on the page "混合专家 MoE" (ai-infra-handbooks,
 * Transformer 解剖), sections "结构" and "实现：逐 token 与按专家分组":
 *     y_t = sum_{i in TopK(softmax(x_t W_r^T))} w_i(x_t) Expert_i(x_t) + sum_s Shared_s(x_t)
 *     Expert(x) = W_down (silu(W_gate x) * (W_up x))          (no biases)
 * with the k weights renormalised to sum to 1, computed in the expert-grouped
 * organisation of that section (flatten (token, slot), stable sort by expert,
 * histogram + prefix sum, one grouped GEMM per projection, weighted scatter back).
 * The capacity limit follows "混合专家模型 (MoE)：大规模稀疏条件计算的架构与工程实践",
 * section 三.1: each expert takes at most C = ceil(CF * N * k / E) assignments;
 * an overflowing assignment skips the expert (the token keeps the residual path,
 * which is the caller's job: out does not include x).
 *
 * Conventions for every call
 *   - Pointers named x, W_*, out, idx, ... are DEVICE pointers owned by the caller;
 *     pointers named *_host are host pointers.  The library never allocates device
 *     memory: scratch comes from a caller-provided workspace of moe_workspace_size()
 *     bytes (256-byte aligned), initialised once with moe_workspace_init().
 *   - Layouts are row-major with the last index contiguous (nn.Linear weight
 *     layout: out x in).  Every row start must be 16-byte aligned, i.e. d, d_ff and
 *     d_ff_shared are multiples of 8 (bf16) or 4 (fp32); base pointers 16-byte aligned.
 *   - Dtypes: act_dtype MOE_BF16 means x, expert weights, intermediates and out are
 *     bf16 with fp32 accumulation; MOE_F32 means all of them are fp32.  The router
 *     weight W_r, its bias b_r, the routing weights w and probabilities are always fp32.
 *   - stream is a cudaStream_t passed as void*.  Calls enqueue work on it and return
 *     after host-side validation; only moe_stats and moe_device_error synchronise.
 *   - Host-detected problems return a moe_status and launch nothing.  Problems found
 *     on the device (an expert index outside [0,E), a bounded wait that ran out) set
 *     bits of a sticky error word in the workspace; read it with moe_device_error().
 *     Kernels never trap.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,    /* null pointer, negative size, misaligned pointer, k > E ... */
    MOE_ERR_UNSUPPORTED = 2,    /* valid but not implemented (E > 1024, k > 16, ...) */
    MOE_ERR_CUDA = 3,           /* a CUDA runtime call failed */
    MOE_ERR_DEVICE_BOUNDS = 4,  /* device saw an expert index outside [0, E) */
    MOE_ERR_DEVICE_TIMEOUT = 5, /* a device-side bounded wait ran out */
    MOE_ERR_WORKSPACE = 6       /* workspace missing, too small or misaligned */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Layer configuration ("混合专家 MoE", 实现 section: MoE(d, d_ff, n_experts, top_k, n_shared)). */
typedef struct {
    int64_t N;                /* tokens in the batch, >= 0 */
    int32_t d;                /* model dim */
    int32_t d_ff;             /* routed expert hidden dim F */
    int32_t E;                /* routed experts, 1..1024 */
    int32_t k;                /* experts per token, 1..min(E, 16) */
    int32_t n_shared;         /* shared experts S, 0..8 (always active, weight 1) */
    int32_t d_ff_shared;      /* shared expert hidden dim F_s (ignored when S = 0) */
    double capacity_factor;   /* <= 0: no capacity limit; else C = ceil(CF * N * k / E) in fp64 */
    int32_t renorm;           /* 1: renormalise the k weights to sum to 1 (the pages' form) */
    int32_t bias_mode;        /* 0: no router bias; 1: b_r added to the logits before softmax;
                                 2: b_r added to the probabilities for the top-k choice only
                                 (weights and P stay unbiased: the DeepSeek-V3 balancing bias,
                                 "混合专家 MoE" 负载均衡 section) */
    int32_t act_dtype;        /* moe_dtype */
} moe_cfg;

/* Device-side error bits of the sticky error word. */
#define MOE_DEVERR_BOUNDS 1
#define MOE_DEVERR_TIMEOUT 2

/* Near-tie threshold: a token whose k-th and (k+1)-th router probabilities differ by
 * less than this is reported by moe_stats (its expert set is not numerically unique). */
#define MOE_TIE_EPS 1e-6f

/* ------------------------------------------------------------------ workspace */

/* Bytes of device workspace needed by every call below for this cfg. */
MOE_API moe_status moe_workspace_size(const moe_cfg *cfg, size_t *bytes_host);

/* Clears the sticky device error word.  Call once after allocating the workspace. */
MOE_API moe_status moe_workspace_init(const moe_cfg *cfg, void *ws, size_t ws_bytes, void *stream);

/* Rows of the expert-grouped buffers: min(N*k, E*C) (N*k without capacity). */
MOE_API int64_t moe_grouped_rows(const moe_cfg *cfg);

/*
 * moe_router_prepare -- prepares the router weight once for many calls ("混合专家 MoE", 实现
 * section, MoE.route: the router is a fixed linear layer d -> E between weight updates).  For
 * bf16 layers with E > 32 the router runs on the tensor cores on an exact three-way bf16 split
 * of the fp32 W_r (hi + mid + lo == W_r bit for bit); this call writes that split into the
 * workspace and records, in host memory, that the workspace now holds the split of this W_r
 * pointer.  moe_route, moe_forward and moe_forward_traced called with the same workspace and
 * the same W_r pointer then skip the split.  Other layers: nothing to prepare (MOE_OK).
 *   W_r [E,d] fp32 in (device); ws as for moe_forward; asynchronous on stream.
 * The caller must call it again after changing W_r's contents (the record is keyed on the
 * pointer, not the values); moe_workspace_init forgets the record.  Calls that pass another
 * W_r pointer split their own weight as usual.
 */
MOE_API moe_status moe_router_prepare(const moe_cfg *cfg, const float *W_r, void *ws,
                                      size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------ steps */

/*
 * moe_route -- router ("混合专家 MoE", 实现 section, MoE.route): logits l = x W_r^T (+ b_r),
 * probabilities p = softmax(l) over all E experts (fp32), the k largest p per token in
 * descending order (ties to the lower expert index), and w = p_sel / sum(p_sel).
 *   x [N,d] act dtype; W_r [E,d] fp32; b_r [E] fp32 (used when bias_mode != 0, else ignored)
 *   idx [N,k] int32 out; w [N,k] fp32 out;
 *   P_sum [E] fp32 out: sum over tokens of p[t,e] (the load-balance P_e times N);
 *   gap [N] fp32 out, nullable: s_(k) - s_(k+1) of the selection scores s (= p, or p + b_r
 *   with bias_mode 2; +inf when k == E).
 * Also writes each token's log-sum-exp of its logits into the workspace (moe_buffers.lse).
 */
MOE_API moe_status moe_route(const moe_cfg *cfg, const void *x, const float *W_r, const float *b_r,
                     int32_t *idx, float *w, float *P_sum, float *gap,
                     void *ws, size_t ws_bytes, void *stream);

/*
 * moe_permute -- grouping by expert ("混合专家 MoE", 实现 section, forward_grouped and the
 * remark after it: counts are a histogram, segment starts a prefix sum) with the capacity
 * rule of "混合专家模型 (MoE)" section 三.1.  Slot f = t*k + j.
 *   idx [N,k] int32 in; w [N,k] fp32 in; x [N,d] act dtype in.
 *   counts [E], offsets [E+1], kept [E], kept_offsets [E+1] int32 out;
 *   perm [N*k] int32 out: slots stably sorted by expert (bit-identical to a stable sort);
 *   pos [N*k] int32 out: grouped row of slot f, or -1 when dropped by the capacity;
 *   row_token [R] int32, row_weight [R] fp32 out: token and routing weight of grouped row r;
 *   x_perm [R,d] act dtype out: row r = x[row_token[r]].   R = moe_grouped_rows(cfg).
 * Grouped rows are expert-major; within an expert, kept slots in increasing f.
 */
MOE_API moe_status moe_permute(const moe_cfg *cfg, const int32_t *idx, const float *w, const void *x,
                       int32_t *counts, int32_t *offsets, int32_t *kept, int32_t *kept_offsets,
                       int32_t *perm, int32_t *pos, int32_t *row_token, float *row_weight,
                       void *x_perm, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_permute_noalloc -- moe_permute without a workspace, for callers that cannot allocate
 * device memory where they run this step (a plugin interface with no workspace argument, or a
 * process whose device memory belongs to another allocator, where a cudaMalloc mid-run would
 * fail under fragmentation or synchronise the device).  Nothing in the pages corresponds to
 * this call: it is an interface convenience around the same grouping kernels.
 * Same arguments and results as moe_permute, except:
 *   - no ws / ws_bytes: the per-block tables live in a fixed 1 MiB array inside the library
 *     (held by every GPU that loads it until exit), which caps ceil(N*k / 2048) * E at 131072;
 *     larger calls return MOE_ERR_WORKSPACE.  The call allocates nothing.
 *   - err [1] int32, nullable, device: MOE_DEVERR_* bits are OR-ed into it (caller clears it).
 *   - all calls share the array: calls that overlap on the GPU race.  The first call on each
 *     device looks up the array's address and keeps it; make it before any stream capture.  A
 *     device reset (cudaDeviceReset) after that first call is not supported.
 */
MOE_API moe_status moe_permute_noalloc(const moe_cfg *cfg, const int32_t *idx, const float *w,
                                       const void *x, int32_t *counts, int32_t *offsets,
                                       int32_t *kept, int32_t *kept_offsets, int32_t *perm,
                                       int32_t *pos, int32_t *row_token, float *row_weight,
                                       void *x_perm, int32_t *err, void *stream);

/*
 * moe_grouped_ffn -- every routed expert's SwiGLU FFN on its grouped rows as grouped GEMMs
 * ("混合专家 MoE", 实现 section: after grouping, a single grouped GEMM serves all experts;
 * Expert.forward):
 *   h_r = silu(W_gate[e] x_r) * (W_up[e] x_r),   y_r = row_weight[r] * (W_down[e] h_r)
 * for rows r in [kept_offsets[e], kept_offsets[e] + kept[e]).
 *   x_perm [R,d]; W_gate, W_up [E,F,d]; W_down [E,d,F] act dtype;
 *   kept [E], kept_offsets [E+1] int32; row_weight [R] fp32, nullable (weight 1);
 *   y_perm [R,d] act dtype out.  h is kept in the workspace (bf16 or fp32).
 */
MOE_API moe_status moe_grouped_ffn(const moe_cfg *cfg, const void *x_perm, const int32_t *kept,
                           const int32_t *kept_offsets, const float *row_weight,
                           const void *W_gate, const void *W_up, const void *W_down,
                           void *y_perm, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_combine -- weighted scatter back to token order plus the shared experts
 * ("混合专家 MoE", 结构 section y = sum w_i Expert_i(x); forward_naive/forward_grouped
 * "+ sum(s(x) for s in shared)"):
 *   out_t = sum_{j : pos[t*k+j] >= 0} y_perm[pos[t*k+j]] + sum_s Shared_s(x_t)
 * summed in fp32 in slot order then shared order, rounded once to the act dtype.
 *   y_perm [R,d] (weights already applied); pos [N*k]; x [N,d];
 *   Ws_gate, Ws_up [S,F_s,d], Ws_down [S,d,F_s] (NULL when S = 0); out [N,d] out.
 */
MOE_API moe_status moe_combine(const moe_cfg *cfg, const void *y_perm, const int32_t *pos, const void *x,
                       const void *Ws_gate, const void *Ws_up, const void *Ws_down,
                       void *out, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------ whole layer */

/*
 * moe_forward -- the whole layer: moe_route, moe_permute, moe_grouped_ffn, moe_combine on
 * one stream with no host synchronisation; intermediates live in the workspace (see
 * moe_forward_buffers).  Arguments as in the step calls; out [N,d] act dtype.
 * For a bf16 batch of at most 128 tokens with shared experts, the shared experts run on a stream
 * owned by the library, forked from `stream` when the call starts (after all work already on
 * `stream`) and joined back before the combine (also when the call returns an error after the
 * fork): the call stays ordered on `stream`, including under stream capture.  That stream
 * belongs to the calling host thread (one per device and thread, kept until exit), so calls
 * from different threads, capturing or not, never share it.  Larger batches use `stream`
 * only.  The same holds for moe_forward_traced and moe_forward_w4a16; there the "shared" phase
 * then measures the wait for the join.
 */
MOE_API moe_status moe_forward(const moe_cfg *cfg, const void *x, const float *W_r, const float *b_r,
                       const void *W_gate, const void *W_up, const void *W_down,
                       const void *Ws_gate, const void *Ws_up, const void *Ws_down,
                       void *out, void *ws, size_t ws_bytes, void *stream);

/* Phases timed by moe_forward_traced: events[i] is recorded after phase i-1 ends. */
#define MOE_TRACE_EVENTS 7  /* start, route, permute, gate/up, down, shared, combine */

/*
 * moe_forward_traced -- moe_forward that also records events[0..6] (cudaEvent_t as void*,
 * created by the caller) on stream: before routing and after routing, permutation,
 * routed gate/up GEMM, routed down GEMM, shared experts and combine.  A NULL entry skips that
 * record (e.g. only events[2] and events[3] to time the gate/up GEMM alone).
 */
MOE_API moe_status moe_forward_traced(const moe_cfg *cfg, const void *x, const float *W_r,
                              const float *b_r, const void *W_gate, const void *W_up,
                              const void *W_down, const void *Ws_gate, const void *Ws_up,
                              const void *Ws_down, void *out, void *ws, size_t ws_bytes,
                              void *stream, void *const *events);

/* Device pointers of the intermediates moe_forward leaves in the workspace. */
typedef struct {
    int32_t *idx;          /* [N,k] */
    float *w;              /* [N,k] */
    float *gap;            /* [N] */
    float *P_sum;          /* [E] */
    int32_t *counts;       /* [E] */
    int32_t *offsets;      /* [E+1] */
    int32_t *kept;         /* [E] */
    int32_t *kept_offsets; /* [E+1] */
    int32_t *perm;         /* [N*k] */
    int32_t *pos;          /* [N*k] */
    int32_t *row_token;    /* [R] */
    float *row_weight;     /* [R] */
    void *x_perm;          /* [R,d] */
    void *y_perm;          /* [R,d] */
    float *lse;            /* [N] log-sum-exp of each token's router logits (for the z-loss) */
} moe_buffers;

MOE_API moe_status moe_forward_buffers(const moe_cfg *cfg, void *ws, size_t ws_bytes, moe_buffers *out_host);

/* ------------------------------------------------------------------ W4A16 expert weights */

/*
 * W4A16 ("混合专家模型 (MoE)：大规模稀疏条件计算的架构与工程实践", section 五.1, the VRAM wall:
 * only the expert layers are quantised, weights to INT4 with 16-bit activations, and the
 * arithmetic runs on dequantised values).  The page fixes no format; this library's is symmetric
 * per-group INT4: for a weight matrix [rows, cols] (cols a multiple of MOE_W4_GROUP), each row's
 * groups of MOE_W4_GROUP consecutive columns share one fp32 scale s = max|w| / 7 (fp32
 * division), stored group-major: s[g * rows + r] for row r, group g; a weight's code is
 * q = w / s rounded half to even and clamped to [-8, 7] (0 when s == 0), stored as a
 * two's-complement nibble, two per byte, the even column in the low nibble.  The dequantised
 * weight is q * s.  Activations, h and the output stay bf16 (act_dtype MOE_BF16
 * only); d, d_ff and d_ff_shared must be multiples of MOE_W4_GROUP.
 */
#define MOE_W4_GROUP 128

typedef struct {
    const uint8_t *q;   /* device, [rows, cols/2] packed codes, 16-byte aligned */
    const float *s;     /* device, [cols/MOE_W4_GROUP, rows] fp32 scales, 16-byte aligned */
} moe_w4;

/* The quantised expert weights of a layer, in the layouts of moe_forward's bf16 weights
 * (rows x cols): gate, up [E*d_ff, d]; down [E*d, d_ff]; shared_gate, shared_up [S*d_ff_shared, d];
 * shared_down [S*d, d_ff_shared] (shared_* ignored when n_shared == 0). */
typedef struct {
    moe_w4 gate, up, down;
    moe_w4 shared_gate, shared_up, shared_down;
} moe_w4_layer;

/*
 * moe_quantize_w4 -- W [rows, cols] bf16 (device) -> q [rows, cols/2], s [cols/128, rows]
 * (device, caller-owned) in the format above; codes are bit-exact with its definition.
 * cols must be a positive multiple of MOE_W4_GROUP (else MOE_ERR_INVALID_ARG); rows >= 0.
 * Asynchronous on stream.
 */
MOE_API moe_status moe_quantize_w4(const void *W, int64_t rows, int32_t cols, uint8_t *q,
                                   float *s, void *stream);

/*
 * moe_grouped_ffn_w4a16 -- moe_grouped_ffn with W4A16 routed-expert weights (W->gate, up,
 * down; the shared_* members are not read).  Arguments otherwise as in moe_grouped_ffn.
 * Returns MOE_ERR_UNSUPPORTED unless act_dtype is MOE_BF16 and d, d_ff are multiples of 128.
 */
MOE_API moe_status moe_grouped_ffn_w4a16(const moe_cfg *cfg, const void *x_perm,
                                         const int32_t *kept, const int32_t *kept_offsets,
                                         const float *row_weight, const moe_w4_layer *W_host,
                                         void *y_perm, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_forward_w4a16 -- moe_forward with W4A16 expert weights (routed and shared), the router
 * unchanged (fp32 W_r).  W_host is a host pointer to the struct of device pointers.
 * events: NULL, or MOE_TRACE_EVENTS events recorded as in moe_forward_traced.
 */
MOE_API moe_status moe_forward_w4a16(const moe_cfg *cfg, const void *x, const float *W_r,
                                     const float *b_r, const moe_w4_layer *W_host, void *out,
                                     void *ws, size_t ws_bytes, void *stream,
                                     void *const *events);

/* ------------------------------------------------------------------ backward pass */

/*
 * moe_backward -- gradients of
 *     L = sum_t <dout_t, out_t> + aux_coef * L_aux + z_coef * L_z
 * for the layer moe_forward just computed, by the chain rule through page "混合专家 MoE"
 * (实现: MoE.route, Expert.forward; 负载均衡: aux_loss = E sum f_e P_e) and the z-loss of
 * "混合专家模型 (MoE)" section 三.3 (L_z = mean_t lse_t^2, see moe_router_stats).  Readings: the
 * top-k choice and capacity drops carry no gradient (piecewise constant); f_e is a count; the
 * selection-only bias (bias_mode 2) gets none (db = 0); the bf16 rounding of h passes the
 * gradient.  The routing weight w_j = p_ij / sum_sel p gives dp_ij = (dw_j - sum w dw) / sum_sel
 * p with dw_j = <dout_t, y_j>; softmax backward; dW_r = dl^T x, db = sum_t dl (bias_mode 1).
 *   Inputs as for moe_forward (the same pointers), dout [N,d] bf16.
 *   ws: the forward's workspace, unchanged since that moe_forward (the router is rerun, bit
 *   for bit, to get the probabilities); bws: moe_backward_workspace_size() bytes, 256-aligned.
 *   Outputs fp32, overwritten: dx [N,d]; dW_r [E,d]; db [E] (nullable); dW_gate, dW_up [E,F,d];
 *   dW_down [E,d,F]; dWs_gate, dWs_up [S,F_s,d], dWs_down [S,d,F_s] (ignored when S = 0).
 * bf16 layers only, with d a multiple of 64 and d_ff, d_ff_shared multiples of 128 (else
 * MOE_ERR_UNSUPPORTED).  Asynchronous; deterministic (no floating-point atomics).
 */
MOE_API moe_status moe_backward_workspace_size(const moe_cfg *cfg, size_t *bytes_host);
MOE_API moe_status moe_backward(const moe_cfg *cfg, const void *x, const float *W_r,
                                const float *b_r, const void *W_gate, const void *W_up,
                                const void *W_down, const void *Ws_gate, const void *Ws_up,
                                const void *Ws_down, const void *dout, double aux_coef,
                                double z_coef, float *dx, float *dW_r, float *db, float *dW_gate,
                                float *dW_up, float *dW_down, float *dWs_gate, float *dWs_up,
                                float *dWs_down, void *ws, size_t ws_bytes, void *bws,
                                size_t bws_bytes, void *stream);

/* ------------------------------------------------------------------ statistics */

/* Load-balance statistics ("混合专家 MoE", 负载均衡 section, aux_loss). */
typedef struct {
    float aux;                 /* L_aux = E * sum_e f_e P_e */
    int32_t device_error;      /* the sticky device error word */
    int64_t dropped;           /* assignments dropped by the capacity */
    int64_t fully_dropped;     /* tokens with every assignment dropped */
    int64_t near_tie;          /* tokens with gap < MOE_TIE_EPS */
    int64_t touched_experts;   /* experts with >= 1 kept row */
    int64_t kept_rows;         /* sum of kept */
} moe_stats_summary;

/*
 * moe_stats -- f_e = counts_e / (N*k) (before dropping), P_e = P_sum_e / N,
 * L_aux = E * sum_e f_e P_e, and the counters above.  Synchronises the stream.
 *   counts [E], kept [E], pos [N*k] int32; P_sum [E] fp32; gap [N] fp32 (nullable);
 *   f_host [E], P_host [E] fp32 host out (nullable); summary_host host out.
 */
MOE_API moe_status moe_stats(const moe_cfg *cfg, const int32_t *counts, const int32_t *kept,
                     const float *P_sum, const int32_t *pos, const float *gap,
                     float *f_host, float *P_host, moe_stats_summary *summary_host,
                     void *ws, size_t ws_bytes, void *stream);

/*
 * moe_selftest_wait_timeout -- failure-path check of the device-side bounded waits (the pages
 * have no counterpart): launches one block that waits, with the same bounded mbarrier waits as
 * the tensor-core kernels (single-thread and warp-wide forms), on a barrier nothing completes;
 * both give up after timeout_us (1 .. 2,000,000) and set MOE_DEVERR_TIMEOUT in the workspace
 * error word.  The context stays usable.  Asynchronous; read the result with moe_device_error.
 */
MOE_API moe_status moe_selftest_wait_timeout(void *ws, size_t ws_bytes, uint32_t timeout_us,
                                             void *stream);

/* Router statistics the pages name for training ("混合专家模型 (MoE)：大规模稀疏条件计算的架构与
 * 工程实践": section 二.2 importance loss, section 三.3 z-loss; the formulas are lost there). */
typedef struct {
    double z_loss;             /* (1/N) sum_t lse_t^2, lse_t = log sum_e exp(logit_t,e) */
    double importance_cv2;     /* Var(Imp) / Mean(Imp)^2 over experts (population variance) */
    double importance_mean;    /* Mean(Imp) = sum of all routing weights / E */
} moe_router_summary;

/*
 * moe_router_stats -- z-loss and importance of one routed batch.  Imp_e = sum of the routing
 * weights w (renormalised top-k) of the assignments to expert e, counted before any capacity
 * drop; the z-loss uses the raw logits before top-k (with the bias when bias_mode == 1, without
 * the selection-only bias of bias_mode 2).  Both sums are deterministic (fixed order, fp64).
 *   lse [N] fp32 (moe_forward_buffers().lse, written by moe_route / moe_forward);
 *   w [N,k] fp32; perm [N*k], offsets [E+1] int32 (moe_permute);
 *   importance_host [E] fp32 host out, nullable; summary_host host out.
 * Synchronises the stream.
 */
MOE_API moe_status moe_router_stats(const moe_cfg *cfg, const float *lse, const float *w,
                                    const int32_t *perm, const int32_t *offsets,
                                    float *importance_host, moe_router_summary *summary_host,
                                    void *ws, size_t ws_bytes, void *stream);

/*
 * moe_selftest_gemm -- check of the backward pass's tcgen05 GEMM engine (the pages have no
 * counterpart): C [M,N] fp32 = sum_k A(m,k) B(n,k) for one group, with A stored [M,K] (a_mn 0,
 * K-major) or [K,M] (a_mn 1, M-major) and B stored [N,K] (b_mn 0) or [K,N] (b_mn 1), bf16.
 * The K-contiguous or MN-contiguous dimension must be a multiple of 8, N of 4.  Uses 512 bytes
 * of ws (the error word and a plan).  Asynchronous.
 */
MOE_API moe_status moe_selftest_gemm(int32_t a_mn, int32_t b_mn, int32_t M, int32_t N, int32_t K,
                                     const void *A, const void *B, float *C, void *ws,
                                     size_t ws_bytes, void *stream);

/* Synchronises the stream and reads the sticky device error word (MOE_DEVERR_* bits). */
MOE_API moe_status moe_device_error(void *ws, size_t ws_bytes, int32_t *code_host, void *stream);

MOE_API const char *moe_status_string(moe_status s);
/* The same string under the short name. */
MOE_API const char *moe_status_str(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
