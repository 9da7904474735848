/*
 * moe.h -- C ABI of the B300 (sm_103a) sparse Mixture-of-Experts FFN forward.
 *
 * The layer (one GPU, one CUDA stream, no host synchronisation):
 *
 *   logits = x W_r^T + b_r                         router GEMM
 *   idx, w = select(logits)                        top-k in one of three modes
 *   offsets, row_of_slot, x_perm = dispatch(idx)   histogram, scan, stable
 *                                                  permutation, capacity drop
 *   h = act(x_perm W1^T [, x_perm W3^T])           grouped expert GEMM (up)
 *   y = h W2^T (+ b2)                              grouped expert GEMM (down)
 *   S = sum_s SwiGLU_s(x)                          always-on shared experts
 *   out[t] = sum_j w[t,j] y[row_of_slot[t,j]] + S[t]   weighted combine
 *   balance = coef * sum_e (count_e / N) * (mean_t p[t,e])
 *
 * Sources (page titles and sections):
 *   - "Hands-on build guide: pure-Python MoE router with load-balanced top-k
 *     gating", Architecture Overview and steps 2 and 5 (gate, combine).
 *   - "Expert Networks > Code Implementation", In[7] (SiLU-MLP expert with
 *     bias) and In[10] (capacity = int(cf * (N // E)), token-order drop).
 *   - "DeepSeek 5.7: MoE from scratch", sections 1-4 (SwiGLU expert, sigmoid
 *     selection with a selection-only balancing bias, dispatch/combine,
 *     shared experts) and Failure modes (empty expert batches are legal).
 *   - "Tutorial -- MoE SER Expert Routing", sections 3-4 (tokens per expert,
 *     load-balancing statistic).
 *   - "Implementing Mixed Expert (MoE) layers", Core Algorithmic Steps
 *     (topk on raw gate scores, softmax over the k, grouping by expert,
 *     SwiGLU expert, index_add_ combine).
 *
 * Conventions for every entry point
 *   - Pointers named "device" point to GPU memory of the current device; the
 *     caller allocates and frees all of it.  Entry points never allocate,
 *     free or synchronise (moe_read_device_error is the one exception: it
 *     waits for the stream to read one word back).
 *   - All work is enqueued on `stream` (a cudaStream_t, NULL = legacy
 *     default stream) and is asynchronous; results are valid once the
 *     stream has reached that point.
 *   - Tensors are dense row-major.  Weights use the PyTorch Linear layout
 *     [out, in], stacked over experts.  Every device pointer must be 16-byte
 *     aligned.  x, weights, biases (except sel_bias), the hidden activations
 *     h and out are in the layer dtype (fp32 or bf16); logits, w, sel_bias,
 *     the expert outputs y and the shared-expert sum S are fp32; indices are
 *     int32.
 *   - Accumulation is fp32, and it runs from the down projection through
 *     the weighted combine: y is not rounded to bf16, the layer output is
 *     rounded once.  bf16 tensors are rounded to nearest even.
 *   - A status other than MOE_OK is returned before anything is enqueued
 *     when arguments are invalid (MOE_ERR_INVALID_ARG / _UNSUPPORTED /
 *     _WORKSPACE); MOE_ERR_CUDA reports a failed launch.  Problems found on
 *     the device (an expert index outside [0, E), group offsets that
 *     decrease or overrun the grouped buffer, a bounded wait that ran out)
 *     set a sticky error word at the start of the workspace instead; read it
 *     with moe_read_device_error.  A GEMM given inconsistent offsets computes
 *     nothing.
 *   - The workspace `ws` must be zero-filled once when it is allocated (its
 *     first word is the device error word; the selection totals live there
 *     too and every call leaves them zero); after that no call needs it
 *     cleared, except after a call that returned MOE_ERR_CUDA.  Calls that
 *     share a workspace must be ordered on one stream.
 *   - n_tokens == 0 is legal: outputs are empty, counts/kept/dropped are
 *     zero-filled, balance is 0.
 */
#ifndef MOE_B300_H_
#define MOE_B300_H_

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

/* ---- status codes ---------------------------------------------------- */
typedef int32_t moe_status_t;
#define MOE_OK                 0
#define MOE_ERR_INVALID_ARG   -1  /* bad size, null or misaligned pointer */
#define MOE_ERR_UNSUPPORTED   -2  /* valid layer the library does not run */
#define MOE_ERR_WORKSPACE     -3  /* ws_bytes smaller than required        */
#define MOE_ERR_CUDA          -4  /* a CUDA launch or copy failed          */
#define MOE_ERR_TIMEOUT       -5  /* device error word: a bounded wait ran out */
#define MOE_ERR_DEVICE_CHECK  -6  /* device error word: bad index seen    */

/* ---- enumerations (stored as int32 in moe_config_t) ---------------- */
#define MOE_F32   0
#define MOE_BF16  1

/* Selection modes.
 * SOFTMAX_TOPK: p = softmax over all E logits; the k experts with the
 *   largest logits (equivalently largest p) are chosen; w_j = p_j / sum of
 *   the chosen p ("Hands-on build guide", step 2, and its test that the
 *   weights sum to 1).
 * TOPK_SOFTMAX: the k largest raw logits are chosen; w = softmax over those
 *   k logits ("Implementing Mixed Expert (MoE) layers", Core Algorithmic
 *   Steps).
 * SIGMOID_BIAS: s_e = sigmoid(logit_e), evaluated in double and rounded to
 *   fp32; the k largest keys s_e + sel_bias_e (fp32 add) are chosen;
 *   w_j = s_j / sum of the chosen s -- the bias never enters a weight
 *   ("DeepSeek 5.7", section 2).
 * In every mode equal keys go to the lower expert index, and slot j of a
 * token holds its j-th best expert (key descending). */
#define MOE_ROUTE_SOFTMAX_TOPK  0
#define MOE_ROUTE_TOPK_SOFTMAX  1
#define MOE_ROUTE_SIGMOID_BIAS  2

/* Expert kinds.
 * SILU_MLP: y = W2 silu(W1 x + b1) + b2 ("Expert Networks", In[7]).
 * SWIGLU:   y = W2 (silu(W1 x) * (W3 x)) (no bias) ("Implementing Mixed
 *           Expert (MoE) layers", expert forward pass; "DeepSeek 5.7" s.1). */
#define MOE_EXPERT_SILU_MLP  0
#define MOE_EXPERT_SWIGLU    1

/* Limits of the library. */
#define MOE_MAX_EXPERTS  256

/* Layer description.  All fields are read, none is written. */
typedef struct moe_config {
  int64_t n_tokens;        /* N >= 0 (batch * sequence, flattened)            */
  int32_t d_model;         /* d >= 1; multiple of 8 (bf16) or 4 (fp32)        */
  int32_t n_experts;       /* E in [1, MOE_MAX_EXPERTS]                        */
  int32_t top_k;           /* k in [1, E]                                      */
  int32_t d_ff;            /* F >= 1; multiple of 8 (bf16) or 4 (fp32)        */
  int32_t n_shared;        /* number of always-on shared SwiGLU experts (>= 0) */
  int32_t d_ff_shared;     /* their hidden width Fs (multiple of 64 if > 0)    */
  float   capacity_factor; /* <= 0: no limit; else capacity =
                              int(capacity_factor * (N / E)), N / E integer
                              division ("Expert Networks", In[10])            */
  int32_t route;           /* MOE_ROUTE_*                                      */
  int32_t expert;          /* MOE_EXPERT_*                                     */
  int32_t dtype;           /* MOE_F32 or MOE_BF16                              */
  int32_t has_bias;        /* SiLU-MLP only: 1 = b1 and b2 are present         */
  float   balance_coef;    /* coefficient of the balance statistic (0.01 in
                              "Tutorial -- MoE SER Expert Routing")           */
} moe_config_t;

/* Device weights (PyTorch Linear layout [out, in], experts stacked). */
typedef struct moe_weights {
  const void  *w_router;   /* [E, d]                                  required */
  const void  *b_router;   /* [E] router bias / logit offset          nullable */
  const float *sel_bias;   /* [E] fp32 selection-only bias, required in
                              SIGMOID_BIAS mode, ignored otherwise             */
  const void  *w1;         /* [E, F, d] gate (SwiGLU) / first layer  required */
  const void  *b1;         /* [E, F]   SiLU-MLP with has_bias                   */
  const void  *w3;         /* [E, F, d] up projection, SwiGLU only             */
  const void  *w2;         /* [E, d, F] down projection               required */
  const void  *b2;         /* [E, d]   SiLU-MLP with has_bias                   */
  const void  *ws1;        /* [S, Fs, d] shared gate     (n_shared > 0)        */
  const void  *ws3;        /* [S, Fs, d] shared up       (n_shared > 0)        */
  const void  *ws2;        /* [S, d, Fs] shared down     (n_shared > 0)        */
} moe_weights_t;

/* Device statistics outputs; every pointer is nullable. */
typedef struct moe_stats {
  int32_t *counts;   /* [E] selections per expert, before any drop          */
  int32_t *kept;     /* [E] assignments processed (<= capacity)              */
  int32_t *dropped;  /* [E] assignments dropped by the capacity              */
  float   *balance;  /* [1] coef * sum_e (counts_e / N) * mean_t p[t, e]     */
} moe_stats_t;

/* ---- sizes ------------------------------------------------------------ */

/* Bytes of scratch the stage calls below need in `ws` (error word, the
 * running per-expert selection totals of the balance statistic, dispatch
 * per-chunk counts, a logits buffer).  Never fails for a valid config;
 * returns MOE_ERR_INVALID_ARG otherwise. */
MOE_API moe_status_t moe_scratch_size(const moe_config_t *cfg, size_t *bytes);

/* Bytes of workspace moe_forward / moe_forward_host need: the scratch plus
 * every intermediate of the layer sized for the worst case M = N * k
 * (idx, w, offsets, row_of_slot, token_of_row, x_perm, h, y, and for shared
 * experts their hidden activations and fp32 sum; host staging for x, out). */
MOE_API moe_status_t moe_workspace_size(const moe_config_t *cfg, size_t *bytes);

/* ---- stages ----------------------------------------------------------- */

/* Router GEMM plus selection ("Implementing Mixed Expert (MoE) layers", the
 * gate and its top-k routing probabilities; "Hands-on build guide", step 2:
 * the gate is a Linear layer, then softmax and top-k; "DeepSeek 5.7",
 * section 2: sigmoid affinities with a selection-only bias).
 * x [N, d] (device, layer dtype); weights->w_router, ->b_router,
 * ->sel_bias used.  Writes idx [N, k] int32 and w [N, k] fp32 (device), and
 * if non-NULL logits [N, E] fp32 (device).  stats->counts receives the
 * selections per expert and stats->balance the balance statistic (both
 * optional).  ws: scratch of moe_scratch_size bytes. */
MOE_API moe_status_t moe_router_topk(const moe_config_t *cfg, const void *x,
                             const moe_weights_t *weights, float *logits,
                             int32_t *idx, float *w, moe_stats_t *stats,
                             void *ws, size_t ws_bytes, void *stream);

/* Selection alone, from given logits [N, E] fp32 (device): the same
 * selection, weights and statistics as moe_router_topk.  sel_bias [E] fp32
 * (device) is required in SIGMOID_BIAS mode. */
MOE_API moe_status_t moe_route_logits(const moe_config_t *cfg, const float *logits,
                              const float *sel_bias, int32_t *idx, float *w,
                              moe_stats_t *stats, void *ws, size_t ws_bytes,
                              void *stream);

/* Grouping by expert with the capacity drop ("Expert Networks", In[10];
 * "DeepSeek 5.7", section 3).  idx [N, k] int32 (device); x [N, d].
 * Assignments are taken in token order, slot order within a token.  The
 * r-th assignment (r from 0) of expert e is kept iff r < capacity; kept
 * assignments of e occupy rows offsets[e] .. offsets[e+1]-1 in arrival
 * order.  Writes offsets [E+1], row_of_slot [N*k] (-1 = dropped),
 * token_of_row [N*k] (first offsets[E] entries valid) and
 * x_perm [N*k, d] (first offsets[E] rows valid, x_perm[r] = x[token_of_row[r]]),
 * and the stats counts/kept/dropped.  x and x_perm may both be NULL: then
 * the rows are not copied (moe_expert_up_gather reads them from x).  An
 * index outside [0, E) is treated as dropped and sets MOE_ERR_DEVICE_CHECK
 * in the error word. */
MOE_API moe_status_t moe_dispatch_permute(const moe_config_t *cfg, const int32_t *idx,
                                  const void *x, int32_t *offsets,
                                  int32_t *row_of_slot, int32_t *token_of_row,
                                  void *x_perm, moe_stats_t *stats, void *ws,
                                  size_t ws_bytes, void *stream);

/* moe_dispatch_permute with one capacity per expert: room [E] int32
 * (device, 16-byte aligned; negative entries count as 0) replaces the
 * capacity derived from cfg->capacity_factor, which is ignored.  The r-th
 * assignment of expert e (in token order) is kept iff r < room[e].  This is
 * the grouping of one contiguous shard of a larger batch whose capacity is
 * int(cf * (N_batch // E)) over the whole batch ("Expert Networks > Code
 * Implementation", In[10], drops in token order across the batch): with
 * prior[e] the selections of expert e by the tokens before the shard,
 * room[e] = clamp(capacity - prior[e], 0, capacity) keeps exactly the
 * shard's part of the batch's kept set.  Outputs and errors as
 * moe_dispatch_permute. */
MOE_API moe_status_t moe_dispatch_permute_room(const moe_config_t *cfg, const int32_t *idx,
                                  const void *x, const int32_t *room,
                                  int32_t *offsets, int32_t *row_of_slot,
                                  int32_t *token_of_row, void *x_perm,
                                  moe_stats_t *stats, void *ws, size_t ws_bytes,
                                  void *stream);

/* moe_dispatch_permute for callers that cannot give the library any device
 * memory of its own: a serving engine that has already claimed the GPU's
 * memory for its own pool, or a hot loop that must not call cudaMalloc
 * (which can stall the whole device).  The pages have no counterpart; this
 * is a deployment variant of the grouping step above, with the same
 * arguments minus the workspace and bit-identical outputs.
 *   - Its per-chunk histogram lives in a fixed 512 KB array inside the
 *     library (allocated on every GPU that loads it, kept until exit), so
 *     n_tokens is limited to 65536: larger layers get MOE_ERR_UNSUPPORTED.
 *   - The first call on each device looks up that array's device address
 *     (with that device current) and keeps it for the life of the process;
 *     make that first call before any stream capture.  Resetting the device
 *     (cudaDeviceReset) after that first call is not supported: the kept
 *     address would no longer be valid.
 *   - Calls share the array: calls whose GPU work may overlap (other
 *     streams, other host threads) race and must be ordered by the caller.
 *   - With no workspace there is no device error word: an expert index
 *     outside [0, E) is dropped without being flagged.
 * It allocates and frees nothing. */
MOE_API moe_status_t moe_dispatch_permute_noalloc(const moe_config_t *cfg,
                                  const int32_t *idx, const void *x,
                                  int32_t *offsets, int32_t *row_of_slot,
                                  int32_t *token_of_row, void *x_perm,
                                  moe_stats_t *stats, void *stream);

/* Expert up-projection and activation on the expert-sorted rows:
 * for each expert e and row r in [offsets[e], offsets[e+1]):
 *   SwiGLU:   h[r] = silu(W1[e] x_perm[r]) * (W3[e] x_perm[r])
 *   SiLU-MLP: h[r] = silu(W1[e] x_perm[r] + b1[e])
 * x_perm [N*k, d], offsets [E+1] (device, read on the device), h [N*k, F]. */
MOE_API moe_status_t moe_expert_up(const moe_config_t *cfg, const void *x_perm,
                           const int32_t *offsets, const moe_weights_t *weights,
                           void *h, void *ws, size_t ws_bytes, void *stream);

/* moe_expert_up with the grouping gather fused into the GEMM's operand
 * loads: row r of expert e reads token row x[token_of_row[r]] straight from
 * x [N, d] instead of x_perm[r], so the expert-sorted copy of the tokens is
 * never written.  token_of_row [N*k] and offsets [E+1] as written by
 * moe_dispatch_permute (device, read on the device); h [N*k, F].  The
 * result equals moe_expert_up on the materialised x_perm bit for bit.  It
 * saves the N*k*d buffer, not time: the per-row loads (TMA gather4, four
 * rows per copy) feed the tensor cores more slowly than 128-row boxes. */
MOE_API moe_status_t moe_expert_up_gather(const moe_config_t *cfg, const void *x,
                                  const int32_t *token_of_row,
                                  const int32_t *offsets,
                                  const moe_weights_t *weights, void *h,
                                  void *ws, size_t ws_bytes, void *stream);

/* Expert down-projection: y[r] = W2[e] h[r] (+ b2[e]); y [N*k, d] fp32. */
MOE_API moe_status_t moe_expert_down(const moe_config_t *cfg, const void *h,
                             const int32_t *offsets,
                             const moe_weights_t *weights, float *y,
                             void *ws, size_t ws_bytes, void *stream);

/* moe_expert_up followed by moe_expert_down (h is caller memory). */
MOE_API moe_status_t moe_grouped_ffn(const moe_config_t *cfg, const void *x_perm,
                             const int32_t *offsets,
                             const moe_weights_t *weights, void *h, float *y,
                             void *ws, size_t ws_bytes, void *stream);

/* Always-on shared experts ("DeepSeek 5.7", section 4):
 * S[t] = sum_s W2s[s] (silu(W1s[s] x[t]) * (W3s[s] x[t])), each with weight
 * one.  Computed as one SwiGLU of width S*Fs (row-concatenated gate/up,
 * column-concatenated down).  x [N, d]; h_shared [N, S*Fs] layer dtype
 * (device scratch, caller memory); shared_out [N, d] fp32. */
MOE_API moe_status_t moe_shared_ffn(const moe_config_t *cfg, const void *x,
                            const moe_weights_t *weights, void *h_shared,
                            float *shared_out, void *ws, size_t ws_bytes,
                            void *stream);

/* Weighted combine back to token order ("Implementing Mixed Expert (MoE)
 * layers", weighted aggregation; "Hands-on build guide", step 5):
 *   out[t] = sum_{j : row_of_slot[t*k+j] >= 0} w[t,j] * y[row_of_slot[t*k+j]]
 *            (+ shared_out[t])
 * accumulated in fp32 in slot order, one rounding to the layer dtype.
 * y [N*k, d] fp32; row_of_slot [N*k]; w [N, k] fp32; shared_out [N, d] fp32
 * (nullable); out [N, d]. */
MOE_API moe_status_t moe_combine(const moe_config_t *cfg, const float *y,
                         const int32_t *row_of_slot, const float *w,
                         const float *shared_out, void *out, void *ws,
                         size_t ws_bytes, void *stream);

/* ---- the whole layer ---------------------------------------------------- */

/* The sparse-MoE FFN layer ("DeepSeek 5.7: MoE from scratch", sections 1-5:
 * route, group tokens by expert, run each expert on its tokens, combine the
 * weighted outputs, plus the always-on shared experts; "Tutorial -- MoE SER
 * Expert Routing", section 4: the load-balance statistic).  All stages
 * above on one stream, intermediates in `ws` (moe_workspace_size bytes).
 * x [N, d] and out [N, d] are device memory. */
MOE_API moe_status_t moe_forward(const moe_config_t *cfg, const void *x,
                         const moe_weights_t *weights, void *out,
                         moe_stats_t *stats, void *ws, size_t ws_bytes,
                         void *stream);

/* moe_forward that also records caller-created CUDA events (cudaEvent_t
 * handles, passed as void*) on `stream` between its stages, for per-stage
 * timing of exactly the launches moe_forward makes: events[0] before the
 * router, then one after each of router+selection, dispatch, expert up,
 * expert down, shared experts (recorded even without shared experts) and
 * combine.  n_events must be MOE_FORWARD_EVENTS. */
#define MOE_FORWARD_EVENTS 7
MOE_API moe_status_t moe_forward_timed(const moe_config_t *cfg, const void *x,
                               const moe_weights_t *weights, void *out,
                               moe_stats_t *stats, void *ws, size_t ws_bytes,
                               void *stream, void *const *events, int32_t n_events);

/* moe_forward for callers whose activations live in host memory: copies
 * x_host [N, d] into the workspace, runs the layer and copies the result to
 * out_host [N, d] (use page-locked host memory for asynchronous copies).
 * Weights and stats are device memory.  The results equal moe_forward's.
 *   - Without a capacity limit and with N >= 8192, the tokens are split into
 *     up to four chunks (whole 32-token statistics groups; two equal ones,
 *     or 3:5:3 / 3:5:5:3 so that the first and last are short) and the
 *     copies of one chunk overlap the compute of another: the copies run on two
 *     streams that the library creates, with some events, on the first such
 *     call on each device (kept until exit); the compute runs on `stream`;
 *     the statistics are reduced once over all chunks.  When the call
 *     returns, all of it is ordered before later work on `stream`.
 *   - Otherwise everything is enqueued on `stream` in order. */
MOE_API moe_status_t moe_forward_host(const moe_config_t *cfg, const void *x_host,
                              const moe_weights_t *weights, void *out_host,
                              moe_stats_t *stats, void *ws, size_t ws_bytes,
                              void *stream);

/* ---- backward ------------------------------------------------------------ */

/* Gradients of L = <dout, out> + d_balance * B with the routing held fixed
 * ("DeepSeek 5.7: MoE from scratch", Worked example and study lab: the router
 * receives gradients through the contribution weights, the top-k choice is
 * not differentiable, an expert no token chose receives none).  The reading
 * (the pages give no formulas): the selected experts and the kept
 * assignments are those of the forward; the contribution weights (softmax
 * over the selected logits, or s_sel / sum s_sel in the sigmoid mode) and
 * the balance statistic (through p; the counts are constant) are
 * differentiated through the logits; dropped assignments pass nothing to
 * their expert; the shared experts (weight one) take dout itself.  All
 * outputs fp32, device memory, overwritten:
 *   dx [N, d], d_w_router [E, d], d_b_router [E] (nullable; only with a
 *   router bias), d_w1 [E, F, d], d_w3 [E, F, d] (SwiGLU only, else
 *   ignored), d_w2 [E, d, F];
 *   d_b1 [E, F], d_b2 [E, d] (SiLU-MLP with has_bias only, else ignored);
 *   d_ws1 / d_ws3 [S, Fs, d], d_ws2 [S, d, Fs] (n_shared > 0 only, else
 *   ignored). */
typedef struct {
  float *dx;
  float *d_w_router;
  float *d_b_router;
  float *d_w1;
  float *d_w3;
  float *d_w2;
  float *d_b1;
  float *d_b2;
  float *d_ws1;
  float *d_ws3;
  float *d_ws2;
} moe_grads_t;

/* Bytes of workspace moe_backward needs: the forward's routing and grouping
 * (each expert's rows padded to a multiple of 16), the recomputed
 * activations and the gradient intermediates, all in grouped row order. */
MOE_API moe_status_t moe_backward_workspace_size(const moe_config_t *cfg, size_t *bytes);

/* The backward pass: recomputes the forward's routing, grouping and expert
 * activations from x, then runs the gradients back through the combine, the
 * experts and shared experts (data and weight gradients on the tensor
 * cores; the weights and activations are read in place, the weight
 * gradients accumulated per expert over its rows in fp32) and the router.
 * The routing weights' gradient <dout, y> is formed as <dout W2, h> +
 * <dout, b2>, so the expert outputs y are not recomputed.  x [N, d] and
 * dout [N, d] are bf16 device arrays;
 * x, dout and the gradient arrays 16-byte aligned (else
 * MOE_ERR_INVALID_ARG).  Supported: bf16 layers of either expert kind
 * (SwiGLU; SiLU-MLP with or without biases), with or without shared
 * experts, d, F and Fs multiples of 64, E a multiple of 8, N > 0 (else
 * MOE_ERR_UNSUPPORTED, nothing enqueued).  With a capacity the drops are
 * those of the forward.  Enqueued on `stream`; ws as for moe_forward,
 * moe_backward_workspace_size bytes. */
MOE_API moe_status_t moe_backward(const moe_config_t *cfg, const void *x,
                                  const moe_weights_t *weights, const void *dout,
                                  float d_balance, moe_grads_t *grads, void *ws,
                                  size_t ws_bytes, void *stream);

/* ---- between steps ------------------------------------------------------ */

/* Balancing-bias update and load diagnostic ("DeepSeek 5.7", section 2: a
 * non-gradient balancing bias added to the selection keys; its study lab
 * plots expert load before and after bias updates, and its implementation
 * plan asks for a coefficient-of-variation diagnostic).  The pages do not
 * state the update; this is the plainest rule they admit:
 *   sel_bias[e] <- sel_bias[e] + gamma * sign(mean load - counts[e])
 * (one fp32 add per expert; the sign compares E * counts[e] with the total
 * on integers, so an expert exactly at the mean keeps its bias), and
 *   *load_cv = population std(counts) / mean(counts)   (0 if all are 0).
 * counts [E] int32 (device, e.g. stats.counts of a forward); sel_bias [E]
 * fp32 updated in place (device, nullable); load_cv [1] fp32 (device,
 * nullable, not both NULL).  Enqueued on `stream`. */
MOE_API moe_status_t moe_update_selection_bias(const moe_config_t *cfg,
                                       const int32_t *counts, float *sel_bias,
                                       float gamma, float *load_cv, void *stream);

/* ---- diagnostics -------------------------------------------------------- */

/* Failure-path self-check: runs the expert GEMMs' bounded mbarrier wait on
 * barriers nothing completes, with a limit of limit_ns (1 us .. 1 s) instead
 * of the kernels' 2 s.  The wait gives up, records MOE_ERR_TIMEOUT in the
 * device error word of ws (read it with moe_read_device_error) and the
 * kernel returns; the context stays usable.  The error word is sticky:
 * zero the workspace's first 256 bytes before using ws for the layer again.
 * ws: at least 256 bytes, 16-byte aligned.  No counterpart on the pages. */
MOE_API moe_status_t moe_check_wait_timeout(void *ws, size_t ws_bytes, int64_t limit_ns,
                                            void *stream);


/* Consistency check of a grouping on the device ("DeepSeek 5.7", s.3 and
 * Failure modes, where most implementation bugs are indexing bugs): for the
 * selection idx [N, k] and the grouping written by moe_dispatch_permute
 * (offsets [E+1], row_of_slot [N*k], token_of_row [N*k]; device), checks that
 *   - offsets start at 0, never decrease, end at M <= N*k, and no group holds
 *     more rows than the capacity;
 *   - every idx is in [0, E) and a token's k experts are distinct;
 *   - every kept slot s = t*k + j lies in its expert's rows,
 *     offsets[idx[s]] <= row_of_slot[s] < offsets[idx[s]+1], with
 *     token_of_row[row_of_slot[s]] == t, and exactly M slots are kept, so
 *     row_of_slot is a bijection of the kept slots onto [0, M);
 *   - rows of one group hold ascending tokens (arrival order).
 * A failure sets MOE_ERR_DEVICE_CHECK in the device error word of ws (read
 * it with moe_read_device_error); nothing else is written.  ws: scratch of
 * moe_scratch_size bytes (two words of its first 256 bytes are used and left
 * zero).  A debugging aid, not part of moe_forward. */
MOE_API moe_status_t moe_check_grouping(const moe_config_t *cfg, const int32_t *idx,
                                        const int32_t *offsets, const int32_t *row_of_slot,
                                        const int32_t *token_of_row, void *ws,
                                        size_t ws_bytes, void *stream);

/* Waits for `stream`, then reads and clears the device error word at the
 * start of `ws`: *code = MOE_OK, MOE_ERR_DEVICE_CHECK or MOE_ERR_TIMEOUT. */
MOE_API moe_status_t moe_read_device_error(void *ws, int32_t *code, void *stream);

/* Static description of a status code (never NULL). */
MOE_API const char *moe_status_string(moe_status_t status);

/* Library version, major * 10000 + minor * 100 + patch. */
MOE_API int32_t moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H_ */
