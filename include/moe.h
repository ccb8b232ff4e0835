/*
 * moe.h -- C ABI of the B300 (sm_103a) forward pass of a token-choice sparse
 * Mixture-of-Experts FFN layer.
 *
 * The layer, for T tokens x[T, d], E experts, top-k, expert width F:
 *   logits = x W_r^T (+ logit_bias)              router linear, no bias term
 *   probs  = softmax(logits) over the E experts
 *   idx    = top-k of (probs + select_bias)       (bias for selection only)
 *   w      = probs[idx] / sum probs[idx]          renormalised gate weights
 *   capacity C = ceil(cf * T * k / E); per expert the first C assignments in
 *   flattened (t*k + j) order are kept, the rest dropped (contribute zero)
 *   y[t]   = sum_j keep * w[t,j] * FFN_{idx[t,j]}(x[t]) + shared(x[t])
 *   FFN_e  = W2_e (silu(W1_e x) * W3_e x)  (SwiGLU)  or  W2_e relu(W1_e x)
 *   f_e = count_e / (T k), p_e = mean_t probs[t,e], aux = E sum_e f_e p_e
 *
 * Sources (page title, section):
 *   "Mixture of Experts", LLM Transformer book (waylandz.com) ch. 30:
 *     §30.2.3 router, §30.2.4 expert FFN, §30.2.6 load-balancing loss,
 *     §30.4.5 shared expert, §30.6.1 MoELayer.
 *   "Mixture of Experts (MoE) memo" (iwashi.co): auxiliary loss worked
 *     example; DeepSeek-V3 aux-loss-free selection bias; Kimi K3 quantile
 *     balancing.
 *   "混合エキスパートモデル（MoE）実践" (deepseekmodel.com): TopKRouter
 *     (softmax, top-k, renormalise, capacity), capacity factor and token
 *     dropping, load_balance_loss, BiasBalancedRouter, grouping tokens by
 *     expert for a grouped GEMM (expert parallelism section).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers, row-major and dense, owned by
 *     the caller.  The library never allocates or frees device memory and
 *     never synchronises the stream, except moe_device_status().
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and enqueues kernels only.
 *   - Arguments are validated on the host before any launch; a call that
 *     returns an error has enqueued nothing.  Launch failures are reported
 *     as MOE_ERR_CUDA.
 *   - Layouts: x [T, d] in cfg->dtype; W_r [E, d] fp32 (nn.Linear
 *     [out, in]); W1, W3 [E, F, d] and W2 [E, d, F] in cfg->dtype; shared
 *     expert Ws1, Ws3 [Fs, d], Ws2 [d, Fs]; topk_idx [T, k] int32;
 *     topk_w [T, k] fp32; probs [T, E] fp32.
 *   - Results are bitwise reproducible run to run (no floating-point
 *     atomics; fixed reduction orders).
 *   - Pointers must be 16-byte aligned (cudaMalloc and torch allocations
 *     are); d and F must be multiples of 8 for bf16 and of 4 for fp32.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* identical to cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,    /* null/misaligned pointer, bad size */
    MOE_ERR_UNSUPPORTED = -2,    /* a shape or option this build does not run */
    MOE_ERR_WORKSPACE = -3,      /* workspace smaller than moe_workspace_size() */
    MOE_ERR_CUDA = -4,           /* a CUDA runtime/launch error */
    MOE_ERR_DEVICE_TIMEOUT = -5, /* a kernel gave up a bounded wait (see
                                    moe_device_status) */
    MOE_ERR_TOO_LARGE = -6       /* problem needs more than the fixed scratch
                                    of moe_dispatch_static */
} moe_status;

enum { MOE_ACT_RELU = 0, MOE_ACT_SWIGLU = 1 };
enum { MOE_DTYPE_FP32 = 0, MOE_DTYPE_BF16 = 1 };
enum { MOE_SELECT_PROBS = 0, MOE_SELECT_LOGITS = 1 };
/* Token choice: each token picks its top-k experts (the layer above).
 * Expert choice: each expert picks its top-C tokens by router probability,
 * C = capacity (cf * T * k / E, k the average experts per token); see
 * moe_layer_forward. */
enum { MOE_ROUTING_TOKEN_CHOICE = 0, MOE_ROUTING_EXPERT_CHOICE = 1 };

typedef struct {
    int32_t T;                /* tokens (batch * seq flattened), >= 0 */
    int32_t d_model;          /* d */
    int32_t n_experts;        /* E, 1..1024 */
    int32_t top_k;            /* k, 1..min(E, 16) */
    int32_t d_ff;             /* F, routed expert width */
    int32_t act;              /* MOE_ACT_* */
    int32_t dtype;            /* MOE_DTYPE_* of x and expert weights */
    float capacity_factor;    /* <= 0: no capacity limit */
    int32_t d_ff_shared;      /* Fs; 0: no shared expert (SwiGLU when > 0) */
    int32_t select_space;     /* MOE_SELECT_*: where select_bias is added */
    int32_t quantile_balance; /* 1: select_bias = -Q_{1-k/E}(probs[:, e]) */
    int32_t out_dtype;        /* dtype of y: MOE_DTYPE_FP32 or MOE_DTYPE_BF16 */
    int32_t reroute_rounds;   /* capacity overflow: 0 = dropped; R > 0 = sent to
                                 the next-best experts in up to R rounds (see
                                 moe_dispatch_reroute); needs capacity_factor > 0
                                 and k * (1 + R) <= 32 */
    int32_t routing;          /* MOE_ROUTING_*: who chooses */
} moe_config;

/* Capacity C = ceil(cf * T * k / E), or T*k when cf <= 0 (no limit).
 * Source: deepseekmodel.com page, section "capacity factor、token dropping". */
int64_t moe_capacity(const moe_config *cfg);

/* Bytes of device workspace moe_layer_forward() needs for `cfg`; the stage
 * calls that take a workspace need at most this much.  0 on invalid cfg. */
size_t moe_workspace_size(const moe_config *cfg);

/* Router: x W_r^T (+ logit_bias), softmax, top-k of (score + select_bias),
 * renormalisation of the selected unbiased probabilities.
 * Sources: ch. 30 §30.2.3 steps 1-4; deepseekmodel.com TopKRouter and
 * BiasBalancedRouter; iwashi.co aux-loss-free and quantile sections.
 *   x           [T, d] cfg->dtype
 *   w_r         [E, d] fp32
 *   logit_bias  [E] fp32 or NULL: added to the logits (part of the router)
 *   select_bias [E] fp32 or NULL: added to probs (select_space PROBS) or to
 *               logits (LOGITS) for selection only; ignored when
 *               cfg->quantile_balance
 *   topk_idx    [T, k] int32 out: experts by descending selection score,
 *               exactly equal scores ordered by lower expert index
 *   topk_w      [T, k] fp32 out: renormalised gate weights
 *   probs       [T, E] fp32 out or NULL
 *   p_mean      [E] fp32 out or NULL: p_e = mean_t probs[t, e]
 *   select_bias_out [E] fp32 out: the quantile bias; required iff
 *               cfg->quantile_balance, else may be NULL
 *   ws, ws_bytes: workspace (>= moe_workspace_size(cfg)) */
int moe_router_topk(const moe_config *cfg, const void *x, const float *w_r,
                    const float *logit_bias, const float *select_bias,
                    int32_t *topk_idx, float *topk_w, float *probs,
                    float *p_mean, float *select_bias_out, void *ws,
                    size_t ws_bytes, moe_stream_t stream);

/* Dispatch: group the T*k assignments by expert (stable in t*k+j order),
 * apply capacity.  Source: deepseekmodel.com expert-parallel dispatch
 * (stable argsort by expert, bincount) and capacity section.
 *   topk_idx  [T, k] int32 in, values in [0, E)
 *   counts    [E] int32 out: assignments per expert before drops
 *   offsets   [E+1] int32 out: exclusive scan of min(counts, C)
 *   perm      [T*k] int32 out: perm[s] = t*k+j of sorted row s, for
 *             s < offsets[E]; later entries untouched
 *   inv       [T*k] int32 out: sorted row of slot t*k+j, or -1 if dropped
 *   n_dropped [1] int32 out */
int moe_dispatch(const moe_config *cfg, const int32_t *topk_idx,
                 int32_t *counts, int32_t *offsets, int32_t *perm,
                 int32_t *inv, int32_t *n_dropped, void *ws, size_t ws_bytes,
                 moe_stream_t stream);

/* Dispatch with capacity overflow redirected to the next-best experts
 * (cfg->reroute_rounds = R > 0).  Source: ch. 30 §30.5.2 (tokens beyond an
 * expert's capacity are dropped or sent to the next best expert).
 *   Round 0 is the rule of moe_dispatch: slots in flattened (t*k + j) order
 *   are served by their expert while it has fewer than C rows.  In each of
 *   the R further rounds every unserved slot takes its token's next unused
 *   expert down the token's ranking (the token's unserved slots, in j order,
 *   take consecutive candidates) and the slots are served in (t*k + j)
 *   order by experts that still have room.  Slots unserved after round R
 *   are dropped.  An expert's rows are grouped in the order served.
 *   topk_idx, topk_w [T, k]: the router's top-k and renormalised weights
 *   cand_idx  [T, nc] int32: each token's experts ranked after its top k,
 *             best first, nc = moe_reroute_candidates(cfg)
 *             = min(E - k, k * R)
 *   cand_w    [T, nc] fp32: their gate weights, p[t, e] over the token's
 *             top-k probability sum (capacity never rescales other slots)
 *   counts [E] (first-choice assignments before capacity), offsets [E+1],
 *   perm [T*k], inv [T*k], n_dropped [1]: as moe_dispatch
 *   slot_expert [T, k] int32, slot_w [T, k] fp32 (or NULL): the expert that
 *             serves each slot and its weight (-1 and 0 when dropped) */
int moe_dispatch_reroute(const moe_config *cfg, const int32_t *topk_idx,
                         const float *topk_w, const int32_t *cand_idx,
                         const float *cand_w, int32_t *counts, int32_t *offsets,
                         int32_t *perm, int32_t *inv, int32_t *slot_expert,
                         float *slot_w, int32_t *n_dropped, void *ws,
                         size_t ws_bytes, moe_stream_t stream);

/* Number of candidate experts per token that redirection uses (see
 * moe_dispatch_reroute), or -1 on an invalid cfg. */
int64_t moe_reroute_candidates(const moe_config *cfg);

/* How the tensor-core grouped GEMMs of one expert FFN will run for cfg: a
 * host-only query (no device work, no GPU needed), chosen from the config
 * alone.  shared = 0: the routed experts; 1: the shared expert.
 *   rows_per_tile  up projection: 0 = 128 token rows on the MMA's M side;
 *                  16/32/64 = weights on the M side and that many token rows
 *                  on the N side (swap-AB, a few rows per expert); 256 = up
 *                  to 256 rows per tile with the MMA N set per tile
 *   up_splits, down_splits  reduction split over CTAs (partial sums added in
 *                  split order)
 *   up_n, down_n   MMA N of 128-row tiles (256, or 128 with few tiles)
 *   down_rows_per_tile  as rows_per_tile for the down projection, or 256:
 *                  up to 256 rows per tile with the MMA N set per tile
 *   down_halves    1, or 2: 256-row down tiles of two M = 128 MMAs
 *   up_pair, down_pair  1: 256-row tiles on a pair of SMs (a cluster of
 *                  two CTAs running one M = 256 MMA, cta_group::2); the
 *                  down projection then reports down_halves = 2
 * Returns MOE_OK, MOE_ERR_INVALID_ARG for an invalid cfg, or
 * MOE_ERR_UNSUPPORTED when the layer does not run on the tensor cores (fp32,
 * or no shared expert for shared = 1); out untouched then. */
typedef struct {
    int32_t rows_per_tile, up_splits, down_splits, up_n, down_n;
    int32_t down_rows_per_tile, down_halves;
    int32_t up_pair, down_pair;
} moe_ffn_plan_info;
int moe_ffn_plan(const moe_config *cfg, int32_t shared, moe_ffn_plan_info *out);

/* Expert-choice routing (cfg->routing = MOE_ROUTING_EXPERT_CHOICE).
 * Sources: deepseekmodel.com TopKRouter discussion (each expert picks the
 * top-C tokens for its capacity, so every expert is exactly full);
 * iwashi.co routing table (expert choice).  Expert e takes the
 * Cn = moe_expert_choice_rows(cfg) = min(C, T) tokens with the largest
 * router probability probs[t, e], exactly equal values by lower token
 * index; the gate weight is probs[t, e] (not renormalised); a token may be
 * taken by any number of experts, including none.  In moe_layer_forward the
 * router's probabilities are used (selection bias and topk_idx/topk_w do
 * not apply and are not written); counts = Cn per expert; n_dropped = the
 * tokens no expert took (their routed output is 0).
 *   probs_t   [E, T] fp32 expert-major router probabilities
 *   perm      [E*Cn] int32 out: token of grouped row e*Cn + i, ascending in t
 *   row_w     [E*Cn] fp32 out: its gate weight
 *   counts [E], offsets [E+1] (e*Cn) out
 *   tok_start [T+1], tok_rows [E*Cn] int32 out: the rows of token t are
 *             tok_rows[tok_start[t] .. tok_start[t+1]), experts ascending
 *   n_unchosen [1] int32 out */
int64_t moe_expert_choice_rows(const moe_config *cfg);
int moe_expert_choice(const moe_config *cfg, const float *probs_t,
                      int32_t *perm, float *row_w, int32_t *counts,
                      int32_t *offsets, int32_t *tok_start, int32_t *tok_rows,
                      int32_t *n_unchosen, void *ws, size_t ws_bytes,
                      moe_stream_t stream);

/* Combine over per-token row lists (expert choice):
 * y[t] = sum_{i in [tok_start[t], tok_start[t+1])} row_w[r_i] out_sorted[r_i]
 *        + shared_out[t], in list order, fp32 accumulation.
 * out_sorted [rows, d] fp32; shared_out [T, d] fp32 or NULL. */
int moe_combine_rows(const moe_config *cfg, const float *out_sorted,
                     const float *row_w, const int32_t *tok_start,
                     const int32_t *tok_rows, const float *shared_out, void *y,
                     moe_stream_t stream);

/* Same results as moe_dispatch, for callers that cannot allocate device
 * memory.  The pages have no counterpart: this is a deployment variant.
 * Some callers have no way to get a workspace: code running inside a host
 * framework that hands it only its inputs and outputs, or a service that
 * forbids device allocations after start-up so that its memory footprint
 * stays fixed.  For them this call takes no workspace and allocates nothing:
 * its scratch (per-chunk histograms and bases) is a fixed
 * MOE_DISPATCH_STATIC_SCRATCH_BYTES array compiled into the library, which
 * every GPU that loads the library holds until the process exits.
 *   - Limit: 2 * ceil(T*k / 1024) * E * 4 bytes must fit in the scratch;
 *     larger problems return MOE_ERR_TOO_LARGE before any launch.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first
 *     call before any stream capture on the device.
 *   - All calls share the one array and it keeps the last call's contents
 *     (every entry a call reads is written by that call first), so calls
 *     that overlap on the GPU (other streams, other host threads) race:
 *     serialise them.
 * Arguments, layouts and results are those of moe_dispatch. */
#define MOE_DISPATCH_STATIC_SCRATCH_BYTES (2u << 20)
int moe_dispatch_static(const moe_config *cfg, const int32_t *topk_idx,
                        int32_t *counts, int32_t *offsets, int32_t *perm,
                        int32_t *inv, int32_t *n_dropped, moe_stream_t stream);

/* Per-expert FFN on the grouped rows: out_sorted[s] = FFN_e(x[perm[s] / k])
 * for offsets[e] <= s < offsets[e+1] (expert choice: x[perm[s]]).
 * Source: ch. 30 §30.2.4 / §30.6.1.  fp32 accumulation; in a bf16 layer the
 * activation h, the bf16 operand of the down projection, is rounded once to
 * the nearest bf16; the output row is fp32.
 *   x          [T, d]; perm, offsets as produced by moe_dispatch (or
 *              moe_dispatch_reroute, moe_expert_choice)
 *   w1, w3, w2 expert weights (w3 NULL for ReLU)
 *   out_sorted [rows, d] fp32 out, rows = T*k (expert choice: E * Cn);
 *              rows >= offsets[E] untouched */
int moe_expert_ffn(const moe_config *cfg, const void *x, const int32_t *perm,
                   const int32_t *offsets, const void *w1, const void *w3,
                   const void *w2, float *out_sorted, void *ws,
                   size_t ws_bytes, moe_stream_t stream);

/* Combine: y[t] = sum_j [inv[t*k+j] >= 0] w[t,j] out_sorted[inv[t*k+j]]
 *               + shared_out[t].   Source: ch. 30 §30.6.1 (weighted
 * accumulate), §30.4.5 (routed + shared).  fp32 accumulation in j order.
 *   out_sorted [*, d] fp32; inv [T*k]; topk_w [T, k]
 *   shared_out [T, d] fp32 or NULL;  y [T, d] in cfg->out_dtype */
int moe_combine(const moe_config *cfg, const float *out_sorted,
                const int32_t *inv, const float *topk_w,
                const float *shared_out, void *y, moe_stream_t stream);

/* Load statistics from (probs, indices), the inputs of the pages'
 * load_balance_loss: f_e = count_e/(T k), p_e = mean_t probs[t,e],
 * aux = E sum f_e p_e (no coefficient), load_max_over_mean =
 * max_e count_e / (T k / E).  Sources: ch. 30 §30.2.6; iwashi.co worked
 * example; deepseekmodel.com load_balance_loss.
 *   probs [T, E] fp32; topk_idx [T, k]; f, p [E] out; aux, load [1] out;
 *   counts [E] int32 out or NULL */
int moe_load_stats(const moe_config *cfg, const int32_t *topk_idx,
                   const float *probs, int32_t *counts, float *f, float *p,
                   float *aux, float *load_max_over_mean, void *ws,
                   size_t ws_bytes, moe_stream_t stream);

/* Weights of one layer (device pointers; see layouts above). */
typedef struct {
    const float *w_r;          /* [E, d] fp32 */
    const float *logit_bias;   /* [E] or NULL */
    const float *select_bias;  /* [E] or NULL */
    const void *w1, *w3, *w2;  /* routed experts (w3 NULL for ReLU) */
    const void *ws1, *ws3, *ws2; /* shared expert, NULL when d_ff_shared = 0 */
} moe_layer_weights;

/* Outputs of one layer call (device pointers; NULL = not wanted, except y). */
typedef struct {
    void *y;                   /* [T, d] cfg->out_dtype, required */
    int32_t *topk_idx;         /* [T, k] */
    float *topk_w;             /* [T, k] */
    int32_t *counts;           /* [E] assignments before drops */
    int32_t *n_dropped;        /* [1] */
    float *f;                  /* [E] */
    float *p;                  /* [E] */
    float *aux;                /* [1] */
    float *load_max_over_mean; /* [1] */
    float *select_bias_out;    /* [E] quantile bias (quantile_balance only) */
    int32_t *counts_unbiased;  /* [E] counts of the plain top-k, no bias */
    int32_t *slot_expert;      /* [T, k] expert that served each slot after
                                  capacity (and redirection), -1 if dropped */
    float *slot_w;             /* [T, k] gate weight the combine used for it */
    int32_t *offsets;          /* [E+1] the grouped layout: expert e's rows are
                                  offsets[e] .. offsets[e+1]) */
    int32_t *perm;             /* [rows] source of each grouped row: flat slot
                                  t*k+j (token choice) or token t (expert
                                  choice); rows = T*k, or E * Cn (see
                                  moe_expert_choice_rows); rows >= offsets[E]
                                  are not written */
    int32_t *cand_idx;         /* [T, nc] with redirection (reroute_rounds > 0):
                                  each token's experts ranked after its top k,
                                  best first, nc = moe_reroute_candidates(cfg);
                                  not written otherwise */
} moe_layer_outputs;

/* The whole forward pass (router, dispatch, experts, shared expert,
 * combine, statistics) on one stream, with no host synchronisation.
 * Source: ch. 30 §30.6.1 MoELayer.forward returning (output, aux_loss).
 * Precision: fp32 accumulation throughout; in a bf16 layer the activation h
 * is stored in bf16 (rounded once to nearest even), and every expert output
 * row (routed and shared) is kept in fp32 for the weighted combine: the
 * results of the stage calls moe_expert_ffn and moe_combine. */
int moe_layer_forward(const moe_config *cfg, const void *x,
                      const moe_layer_weights *wts,
                      const moe_layer_outputs *out, void *ws,
                      size_t ws_bytes, moe_stream_t stream);

/* The monitoring set the deepseekmodel.com page asks every MoE deployment
 * to log ("エキスパート間のスケールドリフト": drop ratio, per-expert load,
 * per-expert output scale, size of the bias term, gate entropy).  Device
 * pointers; NULL = not wanted.  Per-expert load is moe_layer_outputs.counts. */
typedef struct {
    float *drop_ratio;          /* [1] n_dropped / (T k) */
    float *gate_entropy;        /* [1] mean over tokens of -sum_e p ln p (nats) */
    float *bias_mean_abs;       /* [1] mean |b_e| of the selection bias in effect
                                       (the caller's or the quantile bias; 0 without) */
    float *bias_max_abs;        /* [1] max |b_e| */
    float *expert_out_mean;     /* [E] mean over all elements of expert e's output
                                       rows (its kept rows' FFN outputs, before the
                                       gate weight); 0 for an expert without rows */
    float *expert_out_std;      /* [E] population standard deviation of the same */
    float *expert_out_max_abs;  /* [E] largest magnitude of the same */
} moe_observability;

/* moe_layer_forward plus the observability set `obs` (may be NULL, which is
 * exactly moe_layer_forward).  The entropy is summed inside the router
 * kernels; the expert output scale costs one extra read of the expert
 * outputs (T*k*d fp32). */
int moe_layer_forward_observed(const moe_config *cfg, const void *x,
                               const moe_layer_weights *wts,
                               const moe_layer_outputs *out,
                               const moe_observability *obs, void *ws,
                               size_t ws_bytes, moe_stream_t stream);

/* The observability set from stored tensors (the stage form):
 *   probs      [T, E] fp32 router probabilities, or NULL (no entropy)
 *   out_sorted [rows, d] fp32 expert outputs grouped by expert and
 *   offsets    [E+1] int32 their row ranges, or both NULL (no output scale)
 *   select_bias [E] fp32 or NULL; n_dropped [1] int32 or NULL
 * Fields of `obs` whose inputs are NULL are set to 0. */
int moe_observe(const moe_config *cfg, const float *probs,
                const float *out_sorted, const int32_t *offsets,
                const float *select_bias, const int32_t *n_dropped,
                const moe_observability *obs, void *ws, size_t ws_bytes,
                moe_stream_t stream);

/* Synchronises `stream`, then returns and clears the device error word that
 * kernels set when a bounded wait gave up (MOE_ERR_DEVICE_TIMEOUT), or
 * MOE_OK.  The only call that blocks the host. */
int moe_device_status(moe_stream_t stream);

/* Static description of an error code. */
const char *moe_strerror(int status);

/* Number of kernels this library has launched in this process (all entry
 * points, all devices); a monotone counter for launch accounting. */
int64_t moe_kernel_launches(void);

/* Test hook of the failure detection (no counterpart on the pages): every
 * mbarrier wait in the tensor-core GEMM is bounded, and on expiry the kernel
 * sets the error word that moe_device_status returns as
 * MOE_ERR_DEVICE_TIMEOUT, lets its issued copies and MMAs finish, frees its
 * tensor memory and returns.  This sets, on the current device, the limit of
 * the main-loop waits (default 2e9 ns; the waits that drain an aborted CTA
 * keep 2 s) and, with stall_mma = 1, makes the MMA issuer of every GEMM CTA
 * first wait on a barrier phase that nothing completes, so the bounded wait
 * runs out without any fault.  Synchronous; call it with no library work in
 * flight and restore (2000000000, 0) afterwards.  MOE_ERR_INVALID_ARG for a
 * zero limit or stall_mma outside {0, 1}. */
int moe_debug_set_wait_hooks(uint64_t main_loop_limit_ns, int32_t stall_mma);

/* Tuning and test switch of the 256-row SM-pair tiles (see
 * moe_ffn_plan_info.up_pair): 0 (default) the library's rule (experts
 * averaging at least 512 rows, or loads balanced by quantile balancing or expert
 * choice), -1 never (128-row or one-SM 256-row tiles
 * instead), 1 for every projection that runs token rows on the MMA's M side
 * (rows_per_tile = 0; its N is then 256).  Host-only; it applies to the calls
 * planned after it, on every device.  MOE_ERR_INVALID_ARG outside {-1, 0, 1}. */
int moe_debug_set_pair_tiles(int32_t policy);

/* Tuning and test switch of the up projection's per-tile-width geometry
 * (moe_ffn_plan_info.rows_per_tile = 256: weights on the MMA's M side, up to
 * 256 of one expert's rows on its N side, the N rounded up to 16 per tile):
 * 1 wherever the experts average more than 64 rows; 0 (default) and -1
 * never (the library does not choose it by itself: on the workloads
 * measured, token-row tiles ran the up projection faster).  The down
 * projection keeps its own rule.  Host-only; it applies to the calls planned
 * after it, on every device.  MOE_ERR_INVALID_ARG outside {-1, 0, 1}. */
int moe_debug_set_var_up_tiles(int32_t policy);

/* The architecture the library's kernels were compiled for, as the CUDA
 * runtime reports it for one of them on the current device (binaryVersion:
 * major * 10 + minor, 103 for sm_103a) into *version.  Needs a GPU;
 * MOE_ERR_CUDA when the runtime cannot load the kernel there. */
int moe_kernel_binary_version(int32_t *version);

/* Stages of moe_layer_forward that per-stage timing separates. */
enum {
    MOE_STAGE_ROUTER = 0,   /* router, softmax, top-k (+ quantile bias) */
    MOE_STAGE_DISPATCH,     /* histogram, scan, stable scatter */
    MOE_STAGE_STATS,        /* f, p, aux, load max/mean */
    MOE_STAGE_GATHER,       /* rows into the grouped layout */
    MOE_STAGE_UP,           /* grouped up projection + activation */
    MOE_STAGE_DOWN,         /* grouped down projection */
    MOE_STAGE_SHARED,       /* shared expert */
    MOE_STAGE_COMBINE,      /* weighted combine */
    MOE_NUM_STAGES
};

/* Optional per-stage timing of moe_layer_forward: while enabled, each call
 * records a CUDA event on its stream before and after every stage (events
 * are created on first use; no device memory is allocated).  Disabled by
 * default; enabling or disabling discards pending records. */
int moe_stage_timing_enable(int on);

/* Waits for the recorded events, writes the summed milliseconds of each
 * stage into stage_ms[MOE_NUM_STAGES] and the number of timed calls into
 * *calls.  The records are kept until the next moe_stage_timing_enable().
 * A call captured into a CUDA graph while timing is on captures its event
 * records; every replay records those events again, so a read after a
 * replay returns the times of that replay.  Blocks the host. */
int moe_stage_timing_read(double *stage_ms, int64_t *calls);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
