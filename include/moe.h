/*
 * moe.h -- C ABI of libmoe.so, the routed-expert path of a Mixture-of-Experts
 * layer on one GB300 (sm_103a).
 *
 * The path, as the FarSkip-Collective and Luffy pages describe the layer:
 *   router (top-k gating) -> Dispatch (expert-contiguous permutation)
 *   -> [optional Luffy token condensation inside each expert bucket]
 *   -> per-expert SwiGLU FFN (+ shared experts on every token)
 *   -> gated Combine, adding the FarSkip-Collective residual base.
 * Sources (page title, section):
 *   "FarSkip-Collective: Unhobbling Blocking Communication in Mixture of
 *    Experts Models" (Pith review of arXiv 2511.11505): "Core claim" (the MoE
 *    sub-block reads the previous layer's full output; the attention input is
 *    the partial activation including the shared expert), ledger axiom Eq. 9
 *    (T_gate, T_Dispatch, T_routed, T_Combine), referee minor comment 1 (Eq. 6
 *    needs the base residual o_0).
 *   "Communication-Efficient Sparsely-Activated Model Training via Sequence
 *    Migration and Token Condensation" (Luffy, Pith review of arXiv
 *    2411.15419): "What carries the argument" (similar tokens routed to the
 *    same expert reuse one representative's expert output; adaptive threshold
 *    h_t = 1/(1+exp(l_norm))), referee major comment 1 (a condensed token's
 *    forward uses the representative's output).
 *
 * Conventions for every entry point below:
 *   - Every data pointer is a DEVICE pointer on the current CUDA device,
 *     allocated and owned by the caller.  The library allocates no device
 *     memory and never frees caller memory.  Scratch comes from the caller's
 *     workspace `ws` of `ws_bytes` bytes (sizes from the *_workspace_size
 *     functions).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  The library never synchronises the stream, except
 *     moe_get_device_status, which says so.
 *   - Tensors are dense, row-major, with no strides.  Every pointer must be
 *     16-byte aligned.  "act" below means the activation/weight dtype of the
 *     config (fp32 or bf16, raw IEEE / bfloat16 bits).
 *   - Errors found on the host are returned before anything is launched:
 *     MOE_ERR_INVALID_ARG (null or misaligned pointer, non-positive size,
 *     k > E, bad enum), MOE_ERR_UNSUPPORTED (a shape the kernels do not
 *     tile), MOE_ERR_WORKSPACE (ws_bytes too small).  A failed launch returns
 *     MOE_ERR_CUDA.  Conditions found on the device (an expert index out of
 *     range, a bounded wait that gave up) are recorded in a per-device status
 *     word that moe_get_device_status reads; the kernels then skip the bad
 *     access and return instead of faulting or hanging.
 *   - Outputs may not alias inputs, except that `out` may alias `residual`.
 *   - Host threads may call concurrently (each with its own outputs and
 *     workspace): the one-time set-up per device is guarded by a lock.
 *   - Sizes: T >= 0 tokens (T == 0 is a no-op), d model dim, E <= 256 routed
 *     experts, 1 <= k <= min(E, 32), H expert hidden, n_shared shared experts
 *     of hidden H_shared (outside these: MOE_ERR_INVALID_ARG).  T * k <= 2^24
 *     routed pairs per call (else MOE_ERR_UNSUPPORTED).
 *     bf16 layers need d % 256 == 0, H % 128 == 0 and H_shared % 128 == 0
 *     (tensor-core tiles); fp32 layers need d % 64 == 0, H % 64 == 0 and
 *     H_shared % 64 == 0.  Otherwise MOE_ERR_UNSUPPORTED.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_WORKSPACE = 3,
  MOE_ERR_CUDA = 4,
  MOE_ERR_TIMEOUT = 5,      /* device: a bounded wait gave up */
  MOE_ERR_DEVICE_INDEX = 6  /* device: an index was out of range and was skipped */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Gating (router page readings; the pages print no router):
 *   SOFTMAX_TOPK        g = softmax over all E logits, at the k selected experts
 *   SOFTMAX_TOPK_RENORM g = softmax over the k selected logits
 *   SIGMOID_TOPK        g = 1/(1+exp(-l_e)) of each selected expert          */
typedef enum {
  MOE_GATE_SOFTMAX_TOPK = 0,
  MOE_GATE_SOFTMAX_TOPK_RENORM = 1,
  MOE_GATE_SIGMOID_TOPK = 2
} moe_gating;

/* Residual base added by the combine (FarSkip-Collective "Core claim": the
 * MoE input x is the previous layer's full output h_{l-1}; the residual base
 * can be a separately given stream such as the attention-partial a_l):
 *   NONE 0; INPUT r = x; EXTERNAL r = residual; INPUT_PLUS_EXTERNAL r = x + residual */
typedef enum {
  MOE_RES_NONE = 0,
  MOE_RES_INPUT = 1,
  MOE_RES_EXTERNAL = 2,
  MOE_RES_INPUT_PLUS_EXTERNAL = 3
} moe_residual;

typedef struct {
  int32_t T, d, E, k, H, n_shared, H_shared;
  int32_t act_dtype; /* moe_dtype */
  int32_t gating;    /* moe_gating */
  int32_t residual;  /* moe_residual */
} moe_config;

typedef struct {
  const float* W_r;         /* [d, E] fp32 router weight                              */
  const float* router_bias; /* [E] fp32, added to the logits before selection; NULL = none */
  const void* W_gu;         /* [E, 2H, d] act: rows 0..H-1 gate proj, rows H..2H-1 up proj */
  const void* W_down;       /* [E, d, H] act                                           */
  const void* Ws_gu;        /* [n_shared, 2H_shared, d] act; NULL when n_shared == 0   */
  const void* Ws_down;      /* [n_shared, d, H_shared] act; NULL when n_shared == 0    */
} moe_weights;

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(moe_status s);

/* Luffy's adaptive condensation threshold h_t = 1/(1+exp(l_norm)), computed
 * on the host in float64 and rounded to float (Luffy review, "What carries the
 * argument", Eq. 2).  l_norm is the normalised loss decrease of the previous
 * iteration; larger l_norm gives a lower threshold (more condensation). */
float moe_adaptive_tau(float l_norm);

/* Reads and clears this device's status word.  SYNCHRONISES `stream` first.
 * Returns MOE_OK, or the first device-side condition recorded since the last
 * read (MOE_ERR_TIMEOUT / MOE_ERR_DEVICE_INDEX), or MOE_ERR_CUDA. */
moe_status moe_get_device_status(moe_stream_t stream);

/* ---------------------------------------------------------------- router
 * T_gate of FarSkip Eq. 9.  logits[t,e] = sum_i x[t,i] W_r[i,e] (+ bias[e]) to
 * fp32 accuracy (no TF32): fp32 layers on the FMA pipe; bf16 layers on tcgen05
 * tensor cores with W_r split exactly into three bf16 terms (x is exactly
 * bf16, so every product is exact and the sums are fp32).  Then the k experts
 * with the largest logits, largest first, a tie going to the lower index (a
 * NaN logit ranks as -inf, -0 as +0); gates per cfg->gating from the fp32
 * logits.
 *   x        [T, d] act           (in)
 *   W_r      [d, E] fp32          (in)
 *   bias     [E] fp32 or NULL     (in)
 *   logits   [T, E] fp32          (out, the caller may read it)
 *   topk_idx [T, k] int32         (out)
 *   topk_gate[T, k] fp32          (out)
 *   ws       moe_route_workspace_size(cfg) bytes (0 for fp32 layers; NULL allowed then) */
size_t moe_route_workspace_size(const moe_config* cfg);
moe_status moe_route(const moe_config* cfg, const void* x, const float* W_r, const float* bias,
                     float* logits, int32_t* topk_idx, float* topk_gate, void* ws,
                     size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- dispatch
 * T_Dispatch of FarSkip Eq. 9, on one GPU: the permutation that the
 * expert-parallel Dispatch all-to-all performs.  Bucket e holds the tokens
 * routed to e in ascending token order; buckets are laid end to end.
 *   topk_idx [T, k] int32   (in)   entries outside [0, E) are skipped and flagged
 *   counts   [E] int32      (out)  tokens per expert
 *   offsets  [E+1] int32    (out)  exclusive prefix of counts; offsets[E] = T*k minus skipped entries
 *   perm     [T*k] int32    (out)  slot -> token
 *   slot_of  [T, k] int32   (out)  (token, j) -> slot; -1 for a skipped entry
 *   x_perm   [T*k, d] act   (out)  x_perm[s] = x[perm[s]]
 *   ws       moe_dispatch_workspace_size(cfg) bytes of scratch              */
size_t moe_dispatch_workspace_size(const moe_config* cfg);
moe_status moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                        int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* slot_of,
                        void* x_perm, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Same as moe_dispatch, with the same outputs, but without a workspace: it
 * allocates nothing.  The paper has no counterpart; this exists for callers
 * that cannot allocate device memory -- for example a host whose device memory
 * is entirely pre-reserved by its own allocator (a cudaMalloc would fail or
 * fragment it), or a serving loop that must not call cudaMalloc because it
 * synchronises the device and stalls its other streams.
 *   - Scratch is a file-scope device array of 1 MiB inside libmoe.so, held by
 *     every GPU that loads the library until the process exits.  The scratch
 *     needed is 8 * E * ceil(T / 128) bytes; larger shapes return
 *     MOE_ERR_WORKSPACE before anything is launched.
 *   - The first call of any entry point on a device looks up the array's
 *     device address (with that device current); make that first call
 *     before any stream capture.
 *   - Every call shares the array and it keeps the last call's contents
 *     (nothing in it has to start at zero: each call writes every entry it
 *     reads).  Calls whose kernels overlap on the GPU -- on two streams, or
 *     from two threads -- race on the array; serialise them.              */
moe_status moe_dispatch_static_scratch(const moe_config* cfg, const void* x,
                                       const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                                       int32_t* perm, int32_t* slot_of, void* x_perm,
                                       moe_stream_t stream);

/* ---------------------------------------------------------------- condensation
 * Luffy token condensation inside each expert bucket (bf16 layers with
 * T <= 65536 when tau <= 1, else MOE_ERR_UNSUPPORTED; a bucket holds each token at most
 * once).  Offsets whose bucket is longer than T (a routing that named one expert twice
 * for a token) are flagged on the device (MOE_ERR_DEVICE_INDEX) and condense nothing.  Walking a
 * bucket in slot order with the set R of representatives, slot j is condensed
 * onto the earliest r in R with cos(x_perm[j], x_perm[r]) >= tau, else j joins
 * R.  Bitwise-identical rows have similarity 1; a zero row is otherwise
 * dissimilar to everything.  tau > 1 or NaN: no slot is condensed.
 *   x_perm      [T*k, d] bf16 (in)   offsets [E+1] int32 (in, from moe_dispatch)
 *   rep_of      [T*k] int32   (out)  representative slot of every slot (itself if a representative)
 *   n_rep       [E] int32     (out)  representatives per bucket
 *   n_condensed [1] int32     (out)  number of condensed slots                 */
size_t moe_condense_workspace_size(const moe_config* cfg);
moe_status moe_condense(const moe_config* cfg, const void* x_perm, const int32_t* offsets, float tau,
                        int32_t* rep_of, int32_t* n_rep, int32_t* n_condensed,
                        void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- condensation with history
 * Luffy's fast similarity measurement (Luffy review, "What carries the argument": expert
 * activation and historical similarity skip most pair-wise comparisons; ledger free
 * parameters S1, S2 classify pairs similar or dissimilar without a cosine; domain
 * assumption that historical similarity persists across consecutive blocks).
 * As moe_condense, except that a pair of slots in one bucket whose two TOKENS were
 * compared at the previous call and got a class there is decided by that class, with no
 * cosine.  Every pair compared at this call goes to hist_out: an inherited class is kept;
 * a pair decided by its cosine gets "similar" if cos >= s1, "dissimilar" if cos <= s2
 * (similar wins if both hold), else no class.  Pairs whose tokens share no bucket at this
 * call are not carried on.  The decisions cos >= tau, >= s1, <= s2 are taken in fp32.
 * Gram tiles (128 x 256 slot pairs) in which every pair has a class get no tensor-core
 * work; n_cos_tiles counts the tiles that did.
 *   perm [T*k], slot_of [T, k] int32 (in, from moe_dispatch of this call)
 *   hist_in   (in) a record written by an earlier call with the same T, k and E, or NULL
 *             (first block).  A record of another shape or never written counts as empty.
 *   hist_out  (out) moe_condense_history_bytes(cfg) bytes; must not overlap hist_in.
 *   n_cos_tiles [1] int32 (out, nullable)
 * Same limits and workspace as moe_condense (tau <= 1 required: MOE_ERR_INVALID_ARG else).
 * History record layout (byte offsets from the record's start; each array starts on a
 * 256-byte boundary after the previous one):
 *   int32 header[5] = {0x48697374, T, k, E, T*k} at 0; int32 offsets[E+1] at 256;
 *   int32 slot_of[T*k]; int64 bits_base[E]; uint32 planes[2 * (T*k) * ceil(min(T, T*k)/32)].
 *   Bucket e's local rows i < n_e (slot offsets[e] + i) are rows of ceil(n_e/32) word pairs
 *   from pair bits_base[e]; word pair q is planes[2q] (known) and planes[2q + 1] (similar);
 *   bit b of pair w of row i is the slot pair (i, 32w + b) for 32w + b < i: known = it has a
 *   class, similar = the class.                                                        */
size_t moe_condense_history_bytes(const moe_config* cfg);
moe_status moe_condense_hist(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                             const int32_t* perm, const int32_t* slot_of, float tau, float s1,
                             float s2, const void* hist_in, void* hist_out, int32_t* rep_of,
                             int32_t* n_rep, int32_t* n_condensed, int32_t* n_cos_tiles,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- expert FFN
 * T_routed of FarSkip Eq. 9: y[s] = W_down,e (SiLU(W_gate,e x_perm[s]) * (W_up,e x_perm[s]))
 * for every slot s of bucket e.  bf16 layers run on tcgen05 tensor cores
 * (bf16 in, fp32 accumulate, the hidden h rounded to bf16, y stored bf16);
 * fp32 layers run fp32 FMA.  With rep_of non-NULL only representative slots
 * are computed and y is written at those slots only (a condensed slot reads
 * its representative's row).  With n_shared > 0 the shared experts run on all
 * T rows of x and shared_out[t] = sum over shared experts.  offsets are as
 * moe_dispatch writes them: non-decreasing from 0 to T*k, each bucket holding
 * a token at most once (at most T rows).  A bf16 batch of at most 128 tokens
 * checks the last on the device: a larger bucket makes the routed GEMM compute
 * nothing and set MOE_ERR_DEVICE_INDEX.
 *   x_perm [T*k, d] act (in)  offsets [E+1] (in)  rep_of [T*k] or NULL (in)
 *   x [T, d] act (in, used when n_shared > 0)
 *   y_perm [T*k, d] act (out)  shared_out [T, d] act (out, NULL when n_shared == 0) */
size_t moe_expert_ffn_workspace_size(const moe_config* cfg, int with_condensation);
moe_status moe_expert_ffn(const moe_config* cfg, const moe_weights* w, const void* x_perm,
                          const int32_t* offsets, const int32_t* rep_of, const void* x,
                          void* y_perm, void* shared_out, void* ws, size_t ws_bytes,
                          moe_stream_t stream);

/* ---------------------------------------------------------------- combine
 * T_Combine of FarSkip Eq. 9 plus the residual add (FarSkip Eq. 6 with its
 * base term): out[t] = r[t] + shared_out[t] + sum_j gate[t,j] * y_perm[rep(slot_of[t,j])],
 * accumulated in fp32 (j in order), one rounding to act.  rep(s) = rep_of[s],
 * or s when rep_of is NULL.  r per cfg->residual.
 *   y_perm [T*k, d] act (in)  shared_out [T, d] act or NULL (in)
 *   slot_of [T, k] (in)  rep_of [T*k] or NULL (in)  topk_gate [T, k] fp32 (in)
 *   x [T, d] act (in, for MOE_RES_INPUT*)  residual [T, d] act (in, for *EXTERNAL)
 *   out [T, d] act (out; may alias residual)                                   */
moe_status moe_combine(const moe_config* cfg, const void* y_perm, const void* shared_out,
                       const int32_t* slot_of, const int32_t* rep_of, const float* topk_gate,
                       const void* x, const void* residual, void* out, moe_stream_t stream);

/* ---------------------------------------------------------------- whole layer
 * route -> dispatch -> [condense if tau <= 1] -> expert FFN -> combine, all on
 * `stream`, no host synchronisation, intermediates in `ws`.
 *   x [T, d] act (in)  residual [T, d] act or NULL (in)  tau: <= 1 condenses (limits as
 *     moe_condense), > 1 or NaN does not
 *   out [T, d] act (out)
 *   topk_idx_out [T, k] int32 or NULL (out)  n_condensed_out [1] int32 or NULL (out)
 *   ws: moe_workspace_size(cfg, tau <= 1) bytes                                 */
size_t moe_workspace_size(const moe_config* cfg, int with_condensation);
moe_status moe_layer_forward(const moe_config* cfg, const moe_weights* w, const void* x,
                             const void* residual, float tau, void* out, int32_t* topk_idx_out,
                             int32_t* n_condensed_out, void* ws, size_t ws_bytes,
                             moe_stream_t stream);

/* ---------------------------------------------------------------- whole layer, FarSkip overlap
 * moe_layer_forward with the two pieces of FarSkip-Collective's single-device
 * execution.  "Core claim": under FarSkip wiring the next attention sub-block
 * reads a partial activation that holds the shared-expert output but not the
 * routed experts.  Section 4 and Eq. 9: the work that does not depend on the
 * routing runs on a second hardware queue beside the dispatch/routed/combine
 * chain.
 *   partial_out [T, d] act or NULL (out): p[t] = r[t] + sum_s shared_s(x)[t], the
 *     combine's fp32 sum before the routed terms, rounded once (r per cfg->residual).
 *     It must not alias an input or out.
 *   aux_stream (may be NULL or equal to `stream`, then everything runs on
 *     `stream`): with n_shared > 0 the shared experts run on aux_stream, after
 *     the router and beside dispatch, condensation and the routed experts; the
 *     combine on `stream` waits for them.  On return, all work of the call is
 *     ordered before later work on `stream` (aux_stream holds none of it
 *     afterwards).  Capturable in a CUDA graph that begins on `stream`.  The
 *     fork/join events are created once per host thread and device.  Measured
 *     on a GB300, an aux_stream of higher priority than `stream` overlaps best.
 * Other arguments, workspace and errors: as moe_layer_forward.                  */
moe_status moe_layer_forward_ex(const moe_config* cfg, const moe_weights* w, const void* x,
                                const void* residual, float tau, void* out, void* partial_out,
                                int32_t* topk_idx_out, int32_t* n_condensed_out, void* ws,
                                size_t ws_bytes, moe_stream_t stream, moe_stream_t aux_stream);

/* ---------------------------------------------------------------- layer backward
 * Gradients of moe_layer_forward's output (with the same tau) for an output gradient
 * d_out, by the chain rule through the residual base, the shared experts, the routed
 * experts' gated SwiGLU and the router's gates (the top-k selection passes no gradient).
 * With condensation (tau <= 1) a condensed pair's expert ran on its representative's
 * input, so that pair's expert gradient reaches the representative's token and none
 * reaches its own (Luffy review, referee major comment 1); its gate still gets
 * <d_out, y_rep>.  The forward pass is recomputed from x (routing, dispatch, the
 * experts' pre-activations), then the expert gradients run on tcgen05 tensor cores
 * (bf16 operands, fp32 accumulation).  Each routing group is padded to a multiple of
 * 64 rows so the weight gradients contract over whole 64-row blocks.  The steps of the
 * path follow FarSkip-Collective's pre-training execution (review page, Figures 11-12):
 * router, Dispatch, routed and shared experts, Combine.
 * bf16 layers only (fp32 layers: MOE_ERR_UNSUPPORTED); condensation needs T <= 65536.
 *   x [T, d] bf16 (in)   d_out [T, d] bf16 (in)   tau: as moe_layer_forward
 *   d_x [T, d] bf16 (out): gradient w.r.t. x (x also feeds the residual base in the
 *       input modes), summed in fp32, rounded once
 *   d_residual [T, d] bf16 or NULL (out): gradient w.r.t. the external residual
 *       (= d_out; zeros when the mode reads none)
 *   dW_r [d, E] fp32 (out)   d_bias [E] fp32 or NULL (out; zeros without a router bias)
 *   dW_gu [E, 2H, d] fp32, dW_down [E, d, H] fp32 (out)
 *   dWs_gu [S, 2Hs, d], dWs_down [S, d, Hs] fp32 (out; NULL when n_shared == 0)
 *   ws: moe_layer_backward_workspace_size(cfg, tau <= 1) bytes
 * Deterministic: no atomics; every sum in a fixed order.                       */
size_t moe_layer_backward_workspace_size(const moe_config* cfg, int with_condensation);
moe_status moe_layer_backward(const moe_config* cfg, const moe_weights* w, const void* x,
                              const void* d_out, float tau, void* d_x, void* d_residual, float* dW_r,
                              float* d_bias, float* dW_gu, float* dW_down, float* dWs_gu,
                              float* dWs_down, void* ws, size_t ws_bytes, moe_stream_t stream);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* MOE_H_ */
