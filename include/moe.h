/*
 * moe.h — C ABI of libmoe: forward and backward of one token-choice
 * mixture-of-experts layer on one GB300 (sm_103a).
 *
 * The layer, as the source pages state it:
 *   router     logits = x · W_rᵀ (fp32), scores, top-k, mixing weights
 *              (The Ultimate MoE Training Handbook, §3.1 "Router scoring")
 *   dispatch   per-expert histogram, exclusive scan, stable permutation of
 *              token rows into expert-contiguous order (MoE training cluster:
 *              routing, load balancing — "Read the timeline before blaming the
 *              network")
 *   experts    bias-free SwiGLU FFNs run as one grouped GEMM over the expert
 *              segments, plus an optional shared expert (Handbook §3.4)
 *   combine    y[t] = Σ_j w[t,j]·out[row(t,j)] + y_shared[t] (LeCompute,
 *              "An expert transforms numbers inside the model")
 *   aux loss   Switch load-balancing loss (Handbook §3.3, "Aux loss")
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named x, w_router, logits, ... are DEVICE pointers unless stated.
 *    The caller owns every buffer. Apart from a few bytes of device status
 *    kept for the process, the library allocates nothing: calls that need
 *    scratch take (ws, ws_bytes), sized by moe_workspace_bytes().
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and never synchronises the host. Work whose size depends
 *    on the routing (the per-expert segments) is scheduled on the device from
 *    the offsets array, with no copy back to the host. So every call can be
 *    captured into a CUDA graph: after one call of each kind on the device
 *    (which sets function attributes once), a captured sequence replays to
 *    the same bytes as the same calls issued on a stream. Tensor maps are
 *    encoded at the call, so a captured call stays bound to the buffers it
 *    was captured with. (moe_last_device_status synchronises and is not
 *    capturable.)
 *  - Layouts are row-major and dense. act dtype (cfg->act_dtype) is bf16 or
 *    fp32 for x, expert weights and every activation; the router (W_r,
 *    logits, weights w, their gradients) is always fp32; indices are int32.
 *  - Return value: MOE_OK (0) or a negative MOE_ERR_* code for errors the host
 *    can see (bad arguments, alignment, a failed launch). Errors only the
 *    device can see (an expert index out of range, offsets that do not add
 *    up, a wait that ran out of time) are recorded in a device status word;
 *    read it with moe_last_device_status(). Kernels never trap: on such an
 *    error they skip the offending access and record it.
 *  - Results are deterministic: no floating-point atomics, fixed reduction
 *    orders, so two runs on the same inputs give identical bytes.
 *  - Rows must start on 16-byte boundaries: d and every FFN width must be
 *    multiples of 8 (MOE_ERR_ALIGN otherwise), and every pointer 16-byte
 *    aligned.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

/* ---- status codes ---- */
#define MOE_OK                0
#define MOE_ERR_INVALID_ARG  -1  /* null pointer, bad size, refused configuration  */
#define MOE_ERR_UNSUPPORTED  -2  /* valid but not built (e.g. k > 8, E > 256)      */
#define MOE_ERR_ALIGN        -3  /* a row or pointer not 16-byte aligned           */
#define MOE_ERR_CUDA         -4  /* a CUDA runtime call or launch failed           */
#define MOE_ERR_TIMEOUT      -5  /* (device) a bounded wait ran out of time        */
#define MOE_ERR_DEVICE_INDEX -6  /* (device) index / offsets out of range          */
#define MOE_ERR_WORKSPACE    -7  /* ws_bytes smaller than moe_workspace_bytes()    */
#define MOE_ERR_NO_DEVICE    -8  /* no usable sm_103 device                        */

/* ---- enumerations ---- */
#define MOE_SCORE_SOFTMAX 0 /* top-k on logits, softmax over the k chosen     */
#define MOE_SCORE_SIGMOID 1 /* top-k on sigmoid(l)+bias, renormalised (+1e-20) */
#define MOE_SCORE_SQRT_SOFTPLUS 2 /* top-k on sqrt(softplus(l))+bias, renormalised
                                     (+1e-20) like sigmoid (Handbook §3.1
                                     "Gating function")                      */
#define MOE_SCORE_SOFTMAX_PRE 3 /* softmax over all E first, top-k on those
                                   probabilities, weights = the chosen
                                   probabilities, not renormalised (Megatron's
                                   --moe-router-pre-softmax; Handbook §3.1
                                   "Output scale"); allowed at k = 1          */
#define MOE_F32  0
#define MOE_BF16 1
#define MOE_ACT_SWIGLU       0
#define MOE_ACT_SWIGLU_CLAMP 1
#define MOE_ACT_SITU_GLU     2

/* which workspace moe_workspace_bytes() sizes */
#define MOE_WS_PERMUTE      0
#define MOE_WS_GROUPED      1
#define MOE_WS_GROUPED_BWD  2
#define MOE_WS_AUX          3
#define MOE_WS_ROUTE_BWD    4
#define MOE_WS_ROUTE        5
#define MOE_WS_Z_LOSS       6
#define MOE_WS_SHARED_GATE_BWD 7

/* Layer configuration. Names follow the flags the Handbook uses for the layer
 * (§2.5 and §3.4: --num-experts, --moe-ffn-hidden-size, --moe-router-topk,
 * --moe-shared-expert-intermediate-size, --moe-router-score-function,
 * --moe-aux-loss-coeff; §3.1 "Output scale": the routed scaling factor). */
typedef struct {
  int64_t T;         /* tokens in the micro-batch, >= 0                       */
  int32_t d;         /* hidden size, multiple of 8                            */
  int32_t E;         /* routed experts, 1..256                                */
  int32_t k;         /* experts per token, 1..min(8, E)                       */
  int32_t F;         /* routed expert FFN width, multiple of 8                */
  int32_t F_shared;  /* shared expert FFN width (multiple of 8), 0 = none     */
  int32_t score_fn;  /* MOE_SCORE_SOFTMAX | _SIGMOID | _SQRT_SOFTPLUS | _SOFTMAX_PRE */
  int32_t act_dtype; /* MOE_BF16 | MOE_F32                                    */
  float scaling;     /* routed scaling factor (1.0 = none)                    */
  float aux_coeff;   /* Switch aux-loss coefficient                           */
  /* expert activation on fc1's [gate | linear] halves (routed and shared
   * experts alike; Handbook §3.4 "Experts", part "Activation"):
   *   MOE_ACT_SWIGLU (0):        silu(g) * (u + glu_linear_offset)
   *   MOE_ACT_SWIGLU_CLAMP (1):  silu(min(g, c)) * clamp(u, -c, c),
   *                              c = act_clamp, finite > 0, offset 0
   *   MOE_ACT_SITU_GLU (2):      s tanh(g/s) sigmoid(g) * (lin(u) + offset),
   *                              s = act_gate_scale > 0, lin(u) =
   *                              act_linear_scale * tanh(u / act_linear_scale)
   *                              when act_linear_scale > 0, else u
   * A zero-initialised tail is plain SwiGLU.                                 */
  int32_t act_fn;
  float act_clamp;
  float act_gate_scale;
  float act_linear_scale;
  float glu_linear_offset;
} moe_cfg;

/* Validates cfg the way the Handbook says Megatron does: softmax with top-1
 * and renormalisation is refused (§3.1 "Output scale": the router would get
 * no gradient); k <= E. Returns MOE_OK or an error code. */
int moe_check_cfg(const moe_cfg* cfg);

/* ------------------------------------------------------------------------ *
 * S1 + S2. Router: gate GEMM, scores, sorted top-k, mixing weights.
 * Handbook §3.1 "Router scoring" ("Precision": logits = x·W_rᵀ in fp32 from
 * the [E, d] fp32 router weight; "Gating function": softmax selects on the
 * logits and takes the softmax over the k chosen; sigmoid selects on
 * sigmoid(l) + sel_bias and divides the chosen scores by their sum + 1e-20;
 * "Output scale": times the routed scaling factor) and §3.2 "Who selects"
 * (top-k sorted while training).
 *   x          [T, d] act dtype
 *   w_router   [E, d] fp32
 *   logit_bias [E] fp32 or NULL: added to the logits (moves selection AND
 *              weights; used for a fixed per-expert skew of the logits)
 *   sel_bias   [E] fp32 or NULL: the aux-loss-free expert bias, added to the
 *              sigmoid scores for selection only (Handbook §3.3 "Loss-free
 *              bias"); refused with softmax (MOE_ERR_INVALID_ARG)
 *   logits     [T, E] fp32 out (kept for the backward and the aux loss)
 *   idx        [T, k] int32 out, by descending key; equal keys: lower index
 *   w          [T, k] fp32 out
 *   ws         >= moe_workspace_bytes(cfg, MOE_WS_ROUTE) bytes of scratch
 *              (may be NULL when that size is 0); it holds the router weight
 *              split into three bf16 planes for the tensor-core gate GEMM
 * The logits keep fp32 accuracy either way: on the tensor cores (bf16 x, E a
 * multiple of 64) W_r = W0 + W1 + W2 exactly in bf16 planes, every product
 * with a bf16 x is exact, and the partial sums fold into compensated fp32
 * pairs; on the CUDA cores the fp32 FMA sums fold the same way. Their error
 * is far below the 1e-6 gap that separates a decided top-k from a near tie.
 * MOE_ERR_WORKSPACE when ws_bytes is too small.                            */
int moe_route_topk(const moe_cfg* cfg, const void* x, const float* w_router,
                   const float* logit_bias, const float* sel_bias, float* logits,
                   int32_t* idx, float* w, void* ws, size_t ws_bytes, moe_stream_t stream);

/* S3. Dispatch: counts[e] = #{(t,j): idx[t,j] = e}; offsets = exclusive scan
 * (offsets[E] = T·k); stable permutation row(t,j) = offsets[e] +
 * #{t' < t : t' chose e}; x_perm[row(t,j)] = x[t]. LeCompute, "Four GPUs, with
 * one holding up the group" (counts over the T·k assignments) and "Read the
 * timeline before blaming the network" (grouping rows by expert).
 *   idx      [T, k] int32 (each entry in [0, E); an entry out of range is
 *            skipped and recorded as MOE_ERR_DEVICE_INDEX)
 *   counts   [E] int32 out;  offsets [E+1] int32 out
 *   row_of   [T, k] int32 out;  src_tok [T·k] int32 out
 *   x_perm   [T·k, d] act dtype out, or NULL: counts, offsets, row_of and
 *            src_tok only (for moe_grouped_swiglu_gather, which reads the rows
 *            of x through src_tok itself; x may then be NULL too)
 *   ws       >= moe_workspace_bytes(cfg, MOE_WS_PERMUTE) bytes of scratch  */
int moe_permute(const moe_cfg* cfg, const void* x, const int32_t* idx, int32_t* counts,
                int32_t* offsets, int32_t* row_of, int32_t* src_tok, void* x_perm,
                void* ws, size_t ws_bytes, moe_stream_t stream);

/* S4 + S5. Grouped SwiGLU experts: for group g and its rows r in
 * [offsets[g], offsets[g+1]):  [gate | up] = x_rows[r]·W1_gᵀ,
 * h[r] = silu(gate)·up,  out[r] = h[r]·W2_gᵀ. Handbook §3.4 "Count and size"
 * (fc1 is 2F wide, fc2 maps F back to d) and "Activation" (the first half of
 * fc1's output is the gate). One launch covers all groups; the tile schedule
 * is built on the device from `offsets`. Used for the routed experts
 * (n_groups = E, offsets from moe_permute) and the shared expert (n_groups = 1,
 * offsets = NULL meaning one group of n_rows rows).
 *   n_groups  groups (experts), n_rows total rows (= offsets[n_groups])
 *   F         FFN width of these experts (cfg->F or cfg->F_shared)
 *   offsets   [n_groups+1] int32 device, or NULL when n_groups == 1
 *   x_rows    [n_rows, d] act dtype
 *   w1        [n_groups, 2F, d] act dtype (rows [0,F) gate, [F,2F) up)
 *   w2        [n_groups, d, F] act dtype
 *   pre_gu    [n_rows, 2F] act dtype out (gate | up, kept for the backward),
 *             or NULL (forward only)
 *   h         [n_rows, F] act dtype out
 *   out       [n_rows, d] act dtype out
 * Rows are computed with fp32 accumulation (bf16: tcgen05 tensor cores; fp32:
 * CUDA cores). */
int moe_grouped_swiglu(const moe_cfg* cfg, int32_t n_groups, int64_t n_rows, int32_t F,
                       const int32_t* offsets, const void* x_rows, const void* w1,
                       const void* w2, void* pre_gu, void* h, void* out, void* ws,
                       size_t ws_bytes, moe_stream_t stream);

/* S3's row copy fused into S4's operand load (the pages' "also worth trying":
 * LeCompute, "Read the timeline before blaming the network" groups rows by
 * expert before the expert GEMMs). The same as moe_grouped_swiglu on
 * x_rows = x[src_rows[r]] without x_perm being written or read: fc1's A tile
 * is gathered row by row from x with 16-byte asynchronous copies into the
 * layout the tensor cores read. For a forward without a backward (the
 * backward's weight gradient needs x_perm itself).
 *   x         [x_rows, d] act dtype (the layer's tokens)
 *   src_rows  [n_rows] int32: the token of each permuted row (moe_permute's
 *             src_tok); a row outside [0, x_rows) reads as zeros
 *   the rest as moe_grouped_swiglu. bf16 on the tensor cores only
 *   (MOE_ERR_UNSUPPORTED otherwise). fc1 runs on single CTAs.            */
int moe_grouped_swiglu_gather(const moe_cfg* cfg, int32_t n_groups, int64_t n_rows, int32_t F,
                              const int32_t* offsets, const void* x, int64_t x_rows,
                              const int32_t* src_rows, const void* w1, const void* w2,
                              void* pre_gu, void* h, void* out, moe_stream_t stream);

/* S6. Weighted unpermute-combine: y[t] = Σ_{j<k} w[t,j]·out_perm[row_of[t,j]]
 * (+ g_t · shared_out[t]), accumulated in fp32 in j order, then rounded once.
 * LeCompute, "An expert transforms numbers inside the model"; Handbook §3.4
 * "Shared experts" (shared output added at weight 1, or through the sigmoid
 * shared-expert gate: g_t = shared_gate[t] from moe_shared_gate).
 *   out_perm [T·k, d], shared_out [T, d] or NULL, y [T, d] out: act dtype
 *   shared_gate [T] fp32 or NULL (weight 1); needs shared_out              */
int moe_unpermute_combine(const moe_cfg* cfg, const void* out_perm, const int32_t* row_of,
                          const float* w, const void* shared_out, const float* shared_gate,
                          void* y, moe_stream_t stream);

/* S7. Switch load-balancing loss (Handbook §3.3 "Aux loss"):
 * aux = coeff · E / (k · T²) · Σ_e counts[e] · Σ_t P[t,e], with P the softmax
 * of each token's logits over all E experts (sigmoid scores: s / Σ_e s).
 *   logits [T, E] fp32, counts [E] int32, aux: one fp32 on the device, out.
 *   ws >= moe_workspace_bytes(cfg, MOE_WS_AUX) bytes of scratch            */
int moe_aux_loss(const moe_cfg* cfg, const float* logits, const int32_t* counts,
                 float* aux, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Dispatch for callers that cannot allocate device memory. The source pages
 * have no counterpart: this entry point exists for users of the library, not
 * for the method. Some callers own no device allocator of their own: their
 * device memory belongs to a host framework's pool that the library may not
 * draw from, or they run where a cudaMalloc (with the synchronisation it can
 * imply) is not allowed. Such callers cannot pass moe_permute a workspace.
 * moe_permute_noalloc computes exactly what moe_permute computes (same
 * kernels, same outputs, bit for bit) but keeps its scratch in a fixed device
 * array inside the library (MOE_PERMUTE_NOALLOC_SCRATCH_BYTES = 1 MiB), which
 * every GPU that loads the library holds until the process exits. It calls no
 * allocation routine. The caller still passes every input and output.
 *   Limit: ceil(T / 128) * E * 4 bytes of scratch, i.e. ceil(T/128) * E <=
 *   262144 (T <= 131072 at E = 256); larger sizes return MOE_ERR_UNSUPPORTED
 *   before any device work.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture. The address is kept for the rest of the
 *   process: a cudaDeviceReset between calls is not supported (the module
 *   would be reloaded at another address).
 *   Every call shares the one array and leaves its contents behind; nothing in
 *   it needs to start at zero. Calls that overlap on the GPU (other streams,
 *   other host threads) race on the array: serialise them.               */
#define MOE_PERMUTE_NOALLOC_SCRATCH_BYTES (1u << 20)
int moe_permute_noalloc(const moe_cfg* cfg, const void* x, const int32_t* idx,
                        int32_t* counts, int32_t* offsets, int32_t* row_of,
                        int32_t* src_tok, void* x_perm, moe_stream_t stream);

/* ---------------------------- backward ---------------------------------- */

/* B6. Backward of the combine: d_out_perm[row_of[t,j]] = w[t,j]·dy[t];
 * dw[t,j] = <dy[t], out_perm[row_of[t,j]]> (fp32). The shared expert's
 * upstream gradient is dy itself.
 *   dy [T, d], out_perm [T·k, d], d_out_perm [T·k, d] out: act dtype;
 *   dw [T, k] fp32 out                                                      */
int moe_unpermute_combine_bwd(const moe_cfg* cfg, const void* dy, const void* out_perm,
                              const int32_t* row_of, const float* w, void* d_out_perm,
                              float* dw, moe_stream_t stream);

/* B5 + B4. Backward of moe_grouped_swiglu for the same groups:
 *   dh = d_out·W2_g;  d_pre = [dh·up·σ(g)(1+g(1-σ(g))) | dh·silu(g)];
 *   dx_rows = d_pre·W1_g;  dW2_g = d_outᵀ·h;  dW1_g = d_preᵀ·x_rows.
 * A group with no rows gets dW1_g = dW2_g = 0.
 *   pre_gu [n_rows, 2F] and h [n_rows, F] from the forward; d_out [n_rows, d]
 *   d_pre [n_rows, 2F] act dtype out; dx_rows [n_rows, d] act dtype out;
 *   dw1 [n_groups, 2F, d], dw2 [n_groups, d, F] act dtype out (fp32 sums).
 *   ws >= moe_workspace_bytes(cfg, MOE_WS_GROUPED_BWD)
 * On the tensor cores with d < 4096 and a workspace of at least n_rows·F·2
 * bytes, dh is stored in bf16 and the activation's derivative runs as a
 * separate elementwise pass (a short-K tile cannot hide it); otherwise it
 * runs in the dgrad epilogue on the fp32 accumulators. The last
 * 2·n_groups·128 + 128 bytes of a workspace that has them hold per-group
 * copies of the weight gradients' A tensor maps whose rows end at the
 * group's end (built on the device each call), so that a group's last K
 * block reads the next group's rows as zeros; without them those rows are
 * zeroed in shared memory.                                                 */
int moe_grouped_swiglu_bwd(const moe_cfg* cfg, int32_t n_groups, int64_t n_rows,
                           int32_t F, const int32_t* offsets, const void* x_rows,
                           const void* w1, const void* w2, const void* pre_gu,
                           const void* h, const void* d_out, void* d_pre, void* dx_rows,
                           void* dw1, void* dw2, void* ws, size_t ws_bytes,
                           moe_stream_t stream);

/* B7. Gradient of the aux loss w.r.t. the logits, counts held constant:
 * dP[e] = g_aux·coeff·E·counts[e]/(k·T²); softmax: d_l = P ⊙ (dP − <P,dP>);
 * sigmoid (P = s/S): d_l = (dP − <P,dP>)/S ⊙ s(1−s).
 *   d_logits [T, E] fp32: written (accumulate = 0) or added to (= 1).      */
int moe_aux_loss_bwd(const moe_cfg* cfg, const float* logits, const int32_t* counts,
                     float g_aux, float* d_logits, int32_t accumulate, moe_stream_t stream);

/* B2 + B1/B3. Router backward. From dw (gradient of the mixing weights):
 *   softmax: p = softmax(chosen logits), d_l_chosen = p ⊙ (c·dw − <p, c·dw>);
 *   sigmoid: d_s = c·(dw − <dw,s>/S)/S (k > 1; c·dw for k = 1), d_l = d_s·s(1−s);
 * zero for experts not chosen; the selection bias gets no gradient (c = the
 * routed scaling factor, S = Σ chosen s + 1e-20). Then, with the full
 * d_logits (this part plus whatever d_logits already holds when
 * accumulate = 1, e.g. the aux-loss part):
 *   dx_router = d_logits · W_r   ([T, d] fp32 out), or NULL when
 *               moe_router_dx_in_permute_bwd(cfg) is 1: moe_permute_bwd then
 *               forms this product itself (MOE_ERR_INVALID_ARG otherwise)
 *   dw_router = d_logitsᵀ · x    ([E, d] fp32 out)
 *   ws >= moe_workspace_bytes(cfg, MOE_WS_ROUTE_BWD)                       */
int moe_route_topk_bwd(const moe_cfg* cfg, const void* x, const float* w_router,
                       const float* logits, const int32_t* idx, const float* dw,
                       float* d_logits, int32_t accumulate, float* dx_router,
                       float* dw_router, void* ws, size_t ws_bytes, moe_stream_t stream);

/* B1. Backward of the permutation, fused with the other input gradients:
 * dx[t] = r[t] + Σ_j dx_perm[row_of[t,j]] (+ dx_shared[t])
 *         (+ d_gate_logit[t] · w_gate), summed in fp32 in that order and
 * rounded once to the act dtype, where the router's share r[t] is dx_router[t]
 * when given, d_logits[t] · W_r formed here (fp32, experts in order: the value
 * moe_route_topk_bwd would have written) when d_logits and w_router are
 * given, else 0.
 *   dx_perm [T·k, d] act dtype; dx_router [T, d] fp32 or NULL;
 *   dx_shared [T, d] act dtype or NULL; d_gate_logit [T] and w_gate [d]
 *   fp32, both or neither (the shared-expert gate's path); d_logits [T, E]
 *   and w_router [E, d] fp32, both or neither, not with dx_router, and only
 *   where moe_router_dx_in_permute_bwd(cfg) is 1 (else MOE_ERR_UNSUPPORTED);
 *   dx [T, d] out                                                          */
int moe_permute_bwd(const moe_cfg* cfg, const void* dx_perm, const int32_t* row_of,
                    const float* dx_router, const void* dx_shared, const float* d_gate_logit,
                    const float* w_gate, const float* d_logits, const float* w_router, void* dx,
                    moe_stream_t stream);

/* 1 when moe_permute_bwd forms the router's input gradient d_logits · W_r
 * itself for cfg (few experts: E <= 16, where the product has only E terms
 * per element and writing it out as dx_router costs an fp32 [T, d] round
 * trip through HBM), 0 when moe_route_topk_bwd should write dx_router (many
 * experts: a real GEMM, on the tensor cores for bf16); < 0 on a bad cfg.    */
int moe_router_dx_in_permute_bwd(const moe_cfg* cfg);

/* ---------------------------- utilities --------------------------------- */

/* S1 alone: logits = x·W_rᵀ (+ logit_bias), exactly as moe_route_topk
 * computes them (same kernels, same accuracy, same workspace
 * MOE_WS_ROUTE), for routers that select by other rules (quantile). */
int moe_gate_logits(const moe_cfg* cfg, const void* x, const float* w_router,
                    const float* logit_bias, float* logits, void* ws, size_t ws_bytes,
                    moe_stream_t stream);

/* Near ties of S2 (a diagnostic, not a step of the layer): *count = the
 * number of tokens whose k-th and (k+1)-th selection keys differ by less than
 * `band` (>= 0). The keys are the fp32 values moe_route_topk ranks (the
 * logits for softmax, the probabilities for pre-softmax, sigmoid or
 * sqrt(softplus) scores + sel_bias otherwise); for such a token the choice
 * between the two experts rests on rounding (Handbook §3.1 "Precision": the
 * router runs in fp32 so that these decisions are stable). count is one
 * device int32, overwritten; 0 when k = E. Asynchronous on `stream`.       */
int moe_route_near_ties(const moe_cfg* cfg, const float* logits, const float* sel_bias,
                        float band, int32_t* count, moe_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Quantile balancing (Handbook §3.3 "Load balancing", part "Quantile").
 * moe_quantile_route: per token, rank the experts by key = score - beta[e]
 *   (score: the logit for softmax, sigmoid(l) or sqrt(softplus(l)); fp32
 *   subtraction), keep the first k in idx (descending key, ties to the lower
 *   index) with the mixing weights of cfg's score function over them (beta
 *   only selects), and write the (k+1)-th key to alpha[t]. When beta_local is
 *   not NULL, also solve each expert's quantile: beta_local[e] = the
 *   (T k / E + 1)-th largest of score[t, e] - alpha[t] over the T tokens
 *   (exact: a radix select on the fp32 values; T k must be divisible by E).
 *   Needs k < E. MOE_SCORE_SOFTMAX_PRE is refused (MOE_ERR_UNSUPPORTED).
 *   logits [T, E] fp32; beta [E] fp32; idx [T, k] int32 out; w [T, k] fp32
 *   out; alpha [T] fp32 out; beta_local [E] fp32 out or NULL.
 * moe_quantile_accumulate: accum[e] += beta_local[e]; *count += 1 (the
 *   micro-batches of one global batch).
 * moe_quantile_beta_update: beta = ema * beta + (1 - ema) * accum / max(count,
 *   1), then beta -= mean(beta); accum and count are reset to 0.
 *   0 <= ema <= 1, else MOE_ERR_INVALID_ARG.                              */
int moe_quantile_route(const moe_cfg* cfg, const float* logits, const float* beta,
                       int32_t* idx, float* w, float* alpha, float* beta_local,
                       moe_stream_t stream);
int moe_quantile_accumulate(const moe_cfg* cfg, const float* beta_local, float* accum,
                            int32_t* count, moe_stream_t stream);
int moe_quantile_beta_update(const moe_cfg* cfg, float* beta, float* accum, int32_t* count,
                             float ema, moe_stream_t stream);

/* ------------------------------------------------------------------------ *
 * The shared expert's sigmoid gate (Handbook §3.4 "Shared experts",
 * --moe-shared-expert-gate): the shared output is multiplied per token by
 * g_t = sigmoid(x[t] · w_gate), w_gate a [d] fp32 weight.
 * moe_shared_gate: gate[t] = g_t (fp32 [T] out; fp32 dot over d).
 * moe_shared_gate_bwd, for the loss's gradient dy [T, d] and the ungated
 *   shared output shared_out [T, d] (act dtype):
 *     dy_shared[t]    = g_t · dy[t]            (act dtype out: the shared
 *                                               expert's upstream gradient)
 *     d_gate_logit[t] = <dy[t], shared_out[t]> g_t (1 - g_t)   (fp32 [T] out)
 *     dw_gate         = Σ_t d_gate_logit[t] · x[t]             (fp32 [d] out,
 *                       deterministic slice sums)
 *   ws >= moe_workspace_bytes(cfg, MOE_WS_SHARED_GATE_BWD). The input's share,
 *   d_gate_logit[t] · w_gate, is added by moe_permute_bwd.                  */
int moe_shared_gate(const moe_cfg* cfg, const void* x, const float* w_gate, float* gate,
                    moe_stream_t stream);
int moe_shared_gate_bwd(const moe_cfg* cfg, const void* x, const float* gate, const void* dy,
                        const void* shared_out, void* dy_shared, float* d_gate_logit,
                        float* dw_gate, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Router z-loss (Handbook §3.1 "Router scoring", part "Precision",
 * z_loss_func): z = coeff * mean over the T tokens of logsumexp(l_t)^2.
 * (Megatron logs z / coeff, the mean squared logsumexp.)
 *   logits [T, E] fp32;  z: device fp32 scalar out
 *   ws >= moe_workspace_bytes(cfg, MOE_WS_Z_LOSS)
 * moe_z_loss_bwd: d_logits[t, e] (+)= g_z * coeff * 2 * lse_t * softmax(l_t)_e / T
 * (accumulate != 0 adds to d_logits, else overwrites). Deterministic.       */
int moe_z_loss(const moe_cfg* cfg, const float* logits, float coeff, float* z, void* ws,
               size_t ws_bytes, moe_stream_t stream);
int moe_z_loss_bwd(const moe_cfg* cfg, const float* logits, float coeff, float g_z,
                   float* d_logits, int32_t accumulate, moe_stream_t stream);

/* Sequence-wise Switch loss (Handbook §3.3 "Load balancing", part "Scope",
 * Megatron's seq_aux_loss): the aux loss of each sequence on its own - its
 * counts, its router probabilities, its length S = seq_len - averaged over
 * the B = T / seq_len sequences:
 *   out = (1/B) sum_b coeff * E / (k S^2) * sum_e c[b, e] * sum_{t in b} P[t, e]
 * with P as in moe_aux_loss. Token t of sequence b at position s is
 * t = b * S + s (seq_major = 0) or t = s * B + b (seq_major = 1, the
 * [seq, batch] order of Megatron's activations).
 *   logits [T, E] fp32, idx [T, k] int32 (an index out of range is skipped and
 *   recorded as MOE_ERR_DEVICE_INDEX); out: device fp32 scalar
 *   ws >= moe_seq_aux_workspace_bytes(cfg, seq_len)
 * seq_len must divide T (else MOE_ERR_INVALID_ARG). The backward adds
 * g * d(out)/d(logits) (counts held constant) to d_logits, or overwrites it
 * when accumulate == 0. Deterministic.                                     */
size_t moe_seq_aux_workspace_bytes(const moe_cfg* cfg, int64_t seq_len);
int moe_seq_aux_loss(const moe_cfg* cfg, const float* logits, const int32_t* idx,
                     int64_t seq_len, int32_t seq_major, float coeff, float* out, void* ws,
                     size_t ws_bytes, moe_stream_t stream);
int moe_seq_aux_loss_bwd(const moe_cfg* cfg, const float* logits, const int32_t* idx,
                         int64_t seq_len, int32_t seq_major, float coeff, float g,
                         float* d_logits, int32_t accumulate, void* ws, size_t ws_bytes,
                         moe_stream_t stream);

/* Load-balance bookkeeping (Handbook §3.3 "Load balancing", part "Loss-free
 * bias"; §3.2 "Routing strategy", part "Who selects", for MaxVio).
 * moe_tokens_per_expert_accumulate: tokens_per_expert[e] += counts[e]
 *   (counts [E] int32 from moe_permute; tokens_per_expert [E] int64, the
 *   router's running count, zeroed by the caller when a step starts).
 * moe_expert_bias_update: expert_bias[e] += sign(total - tokens_per_expert[e]
 *   * E) * rate in fp32, total = sum of the counts; the comparison is made on
 *   the int64 values, never on a floating-point mean.
 * moe_max_vio: *max_vio = (max_e count - total / E) / (total / E), computed as
 *   (max * E - total) / total in fp64 and stored as fp32; 0 when total = 0.
 * All three are single small launches on `stream`.                         */
int moe_tokens_per_expert_accumulate(const moe_cfg* cfg, const int32_t* counts,
                                     int64_t* tokens_per_expert, moe_stream_t stream);
int moe_expert_bias_update(const moe_cfg* cfg, const int64_t* tokens_per_expert,
                           float* expert_bias, float rate, moe_stream_t stream);
int moe_max_vio(const moe_cfg* cfg, const int64_t* tokens_per_expert, float* max_vio,
                moe_stream_t stream);

/* Bytes of scratch the call `which` (MOE_WS_*) needs for cfg. For
 * MOE_WS_GROUPED / MOE_WS_GROUPED_BWD the size covers the routed experts
 * (T·k rows, F) and the shared expert (T rows, F_shared). 0 on bad input. */
size_t moe_workspace_bytes(const moe_cfg* cfg, int which);

/* Static English text for a status code. */
const char* moe_status_string(int status);

/* "cudaErrorName: description" of the CUDA runtime error behind the calling
 * thread's most recent MOE_ERR_CUDA, or "" if there was none. The string
 * stays valid until the thread's next call of this function. */
const char* moe_last_cuda_error(void);

/* Synchronises `stream`, returns the first device-detected error recorded
 * on the current device since the previous call (MOE_OK if none) and clears
 * it. `detail` (may be NULL) receives the offending index or a site code. */
int moe_last_device_status(moe_stream_t stream, int32_t* detail);

/* Upper bound, in nanoseconds, of every spin-wait inside the kernels
 * (default 2e9). A wait that runs out records MOE_ERR_TIMEOUT and its kernel
 * returns after releasing what it holds. Returns the previous value. */
uint64_t moe_set_wait_timeout_ns(uint64_t ns);

/* Launches one kernel that waits for a device flag nothing ever sets, with
 * the current timeout; used to test that bounded waits end and report
 * MOE_ERR_TIMEOUT (read it with moe_last_device_status). */
int moe_selftest_wait_timeout(moe_stream_t stream);

/* Which kernels run the grouped expert GEMMs (moe_grouped_swiglu and its
 * backward). MOE_GEMM_AUTO (default): bf16 on the tcgen05 tensor cores, with
 * the forward and data-gradient contractions on CTA pairs (cta_group::2) when
 * the segments average at least 128 rows and on single CTAs otherwise, and
 * the weight gradients on CTA pairs; fp32 on CUDA cores.
 * MOE_GEMM_TC_SINGLE_CTA / MOE_GEMM_TC_PAIRS: bf16 on single-CTA / CTA-pair
 * tcgen05 kernels whatever the segment sizes (the weight gradients too).
 * MOE_GEMM_CUDA_CORES: every dtype on the CUDA-core kernels (fp32
 * accumulation). All but the first are for cross-checking. Process-wide;
 * returns the previous setting, or MOE_ERR_INVALID_ARG. */
#define MOE_GEMM_AUTO          0
#define MOE_GEMM_CUDA_CORES    1
#define MOE_GEMM_TC_SINGLE_CTA 2
#define MOE_GEMM_TC_PAIRS      3
int moe_set_grouped_gemm_impl(int impl);

/* Which kernels compute the router's gate GEMM (moe_route_topk).
 * MOE_ROUTER_AUTO (default): the tcgen05 kernel over three bf16 planes of W_r
 * when x is bf16 and E is a multiple of 64 (E >= 64), the CUDA-core kernels
 * otherwise. MOE_ROUTER_CUDA_CORES: always the CUDA-core kernels (for
 * cross-checking). Process-wide; returns the previous setting, or
 * MOE_ERR_INVALID_ARG. */
#define MOE_ROUTER_AUTO       0
#define MOE_ROUTER_CUDA_CORES 1
int moe_set_router_impl(int impl);

/* K elements per window of the tensor-core gate GEMM's main accumulator
 * before the window's sums fold into the compensated pair (multiple of 16,
 * 16..4096; default 32). Shorter windows bound the fp32 accumulation error
 * more tightly and cost more folding. Returns the previous value, or
 * MOE_ERR_INVALID_ARG. */
int moe_set_router_fold(int fold_k);

/* 1 when moe_route_topk would run its gate GEMM on the tensor cores for cfg
 * under the current setting, else 0. */
int moe_router_uses_tensor_cores(const moe_cfg* cfg);

/* 1 when moe_route_topk_bwd would run dx_router and dW_r on the tensor cores
 * (bf16 activations, E >= 32, E a multiple of 8, tensor-core router setting),
 * else 0. */
int moe_router_bwd_uses_tensor_cores(const moe_cfg* cfg);

/* Per-kernel timing of the tcgen05 grouped GEMM kernels, for measurement.
 * moe_kernel_timing(1) starts recording a CUDA event pair around every such
 * launch on the current device (on the launching stream) and discards earlier
 * records; moe_kernel_timing(0) stops recording. moe_kernel_times() waits for
 * the recorded events and returns, per kernel kind (MOE_KERNEL_*), the summed
 * milliseconds and the number of launches. Arrays hold MOE_KERNEL_KINDS entries. */
#define MOE_KERNEL_FC1_FWD   0  /* fc1 + SwiGLU forward           */
#define MOE_KERNEL_FC2_FWD   1  /* fc2 forward                    */
#define MOE_KERNEL_FC2_DGRAD 2  /* fc2 dgrad + SwiGLU backward    */
#define MOE_KERNEL_FC1_DGRAD 3  /* fc1 dgrad                      */
#define MOE_KERNEL_FC2_WGRAD 4  /* fc2 weight gradient            */
#define MOE_KERNEL_FC1_WGRAD 5  /* fc1 weight gradient            */
#define MOE_KERNEL_KINDS     6
int moe_kernel_timing(int enable);
int moe_kernel_times(float* ms_total, int32_t* launches);

/* Number of CUDA kernels this library has launched in this process (all
 * devices, all streams), counted on the host at launch time. */
uint64_t moe_launch_count(void);

/* Library build identification: "libmoe <version> sm_103a". */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
