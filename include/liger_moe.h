/*
 * liger_moe.h -- C ABI of the routed Mixture-of-Experts layer on one GPU
 * (forward and backward), hand-written CUDA for sm_103a (GB300).
 *
 * The layer, per token t with router logits l[t, 0..E-1] and input x[t, :]:
 *   route     ids[t, 0..k-1] = the k largest logits (ties -> smaller id),
 *             w[t, j] = softmax of the k selected logits
 *   dispatch  slots s = t*k + j sorted stably by expert -> expert-major rows
 *   experts   per row r of expert e:  g = x W_gu[e, :I]^T,  u = x W_gu[e, I:]^T,
 *             h = bf16(silu(g) * u),   y = bf16(w * (h W_d[e]^T))
 *   combine   Y[t] = bf16(sum_j y[row of slot (t, j)])
 *   backward  dX, dW_gate_up, dW_down and d_logits of L = <dY, Y>.
 * Sources: LightMoE README ("MoE inference": dispatch, gate/up projection,
 * gated activation, down projection, routing-weight application,
 * deterministic combine; "MoE training": MoEDispatch outputs, input-, weight-
 * and router-gradient kernels; "Grouped GEMM": expert-major rows, m_indptr
 * int32 [E+1], empty experts valid; "Limits": K aligned to 64), LigerCute
 * README ("LigerMoE design": forward sorts routed tokens, final local combine
 * applies router weights; backward recomputes activations, computes dX and
 * dW, reduces routed dX to tokens) and the LigerCute PR summary (a flat
 * extern "C" boundary with no torch types; BF16).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers, row-major and contiguous.
 *     bf16 tensors are passed as void* (IEEE bfloat16 bit patterns).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Every call only enqueues work on `stream`: it never synchronises, never
 *     allocates device memory and never frees anything.  The backward entry
 *     points run two of their small kernels on a library-owned stream of the
 *     calling thread, forked from `stream` and joined back into it with
 *     events: to the caller (and to a graph capture of `stream`) all of the
 *     call's work is ordered on `stream`.
 *   - The caller owns every buffer.  Outputs are overwritten, never
 *     accumulated into (one stated exception: liger_moe_router_bwd adds to dx).
 *     Buffers of one call must not overlap unless stated.
 *   - bf16 buffers must be 16-byte aligned; H and I must be multiples of 64.
 *   - Limits: 1 <= E <= 1024; 1 <= k <= min(E, 32); T >= 0;
 *     T*k, E*2I and E*H below 2^31.  T = 0 is valid and launches nothing.
 *   - Entry points that take `workspace` report its size: called with
 *     workspace == NULL they store the required byte count in
 *     *workspace_bytes, validate the other arguments and launch nothing.
 *     Otherwise *workspace_bytes is the size of the caller's buffer (256-byte
 *     aligned device memory) and must be at least the reported size.
 *   - Argument errors are reported before anything is launched.  Errors the
 *     device finds (an expert id outside [0, E), a row index outside [0, R),
 *     an internal pipeline wait that ran past its time limit) set a flag that
 *     liger_moe_device_error() returns; outputs of that call are unspecified.
 *   - Only devices of compute capability 10.3 (sm_103) are supported.
 *   - Launch mode: a call with fewer than 4096 routed rows (T*k) launches its
 *     kernels with programmatic dependent launch: each kernel may start while
 *     the one before it on the stream finishes, and waits for it before
 *     touching memory.  Larger calls run in plain stream order.  The
 *     environment variable LIGER_MOE_PDL (read once per process) overrides
 *     this: "0" never, any other non-empty value always.  Results are
 *     identical in every mode.
 */
#ifndef LIGER_MOE_H_
#define LIGER_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
typedef enum {
  LIGER_MOE_OK = 0,
  LIGER_MOE_ERR_INVALID_ARG = -1,        /* null pointer, k > E, negative size, ... */
  LIGER_MOE_ERR_MISALIGNED = -2,         /* H or I not a multiple of 64, pointer not 16-byte aligned */
  LIGER_MOE_ERR_CAPACITY = -3,           /* workspace too small, or a size above a stated limit */
  LIGER_MOE_ERR_UNSUPPORTED_DEVICE = -4, /* current device is not sm_103 */
  LIGER_MOE_ERR_LAUNCH = -5,             /* a CUDA call failed (see liger_moe_last_cuda_error) */
  LIGER_MOE_ERR_DEVICE = -6              /* returned by liger_moe_device_error when a flag is set */
} liger_moe_status;

/* Activations of the expert MLP, h = act(g, u) with g, u the fp32 gate and up projections.
 * LightMoE README, "Compatibility" and "Highlights" name the variants; their formulas are the
 * plainest published forms.  A clamp passes the gradient on its closed interval and blocks it
 * outside.  LIGER_MOE_ACT_RELU2 is the one non-gated form: its experts hold two weights
 * (LightMoE README, "MoE inference"), the up weight W_up [E, I, H] taking the place of
 * w_gate_up, h = max(a, 0)^2 with a = x W_up^T; its saved factor is dh/da, gu_perm [R, I],
 * and dw_gate_up receives dW_up [E, I, H]. */
enum liger_moe_activation {
  LIGER_MOE_ACT_SWIGLU = 0,         /* silu(g) u                                             */
  LIGER_MOE_ACT_SWIGLU_BOUNDED = 1, /* silu(min(g, c)) clamp(u, -c, c)          (c = clamp)  */
  LIGER_MOE_ACT_SWIGLU_OAI = 2,     /* gc sigmoid(1.702 gc) (clamp(u, -c, c) + 1), gc = min(g, c) */
  LIGER_MOE_ACT_GEGLU = 3,          /* gelu(g) u, gelu(g) = g/2 (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) */
  LIGER_MOE_ACT_REGLU = 4,          /* max(g, 0) u                                           */
  LIGER_MOE_ACT_RELU2 = 5           /* max(a, 0)^2 of one up projection (two-weight experts) */
};

/* Bits of the device error flag. */
#define LIGER_MOE_DEVERR_BAD_EXPERT_ID 0x1 /* topk_ids entry outside [0, E) */
#define LIGER_MOE_DEVERR_BAD_ROW 0x2       /* row / slot index outside [0, T*k) */
#define LIGER_MOE_DEVERR_BAD_INDPTR 0x4    /* m_indptr not 0 = m[0] <= ... <= m[E] = R */
#define LIGER_MOE_DEVERR_WAIT_TIMEOUT 0x8  /* a pipeline wait inside a GEMM kernel gave up */

/*
 * Router: top-k experts and renormalised gate weights per token.
 * LightMoE README, "MoE inference" (top_k_ids int32, distinct per token;
 * top_k_weights float32) and "MoE training" (differentiable_probs).
 *   logits    [T, E] float32, input.
 *   topk_ids  [T, k] int32, output: experts by descending logit; equal logits
 *             -> smaller id first; NaN ranks below every number (by id).
 *             -0.0 and +0.0 are equal.
 *   topk_w    [T, k] float32, output: w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0)
 *             over the selected k (softmax over E, top-k, renormalised).
 * No workspace.  Bit-exact ids for a given logits tensor.
 */
int liger_moe_route_topk(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                         void* stream);

/*
 * Dispatch: deterministic expert-major order of the R = T*k routed slots
 * (slot s = t*k + j).  Rows of expert e are m_indptr[e] .. m_indptr[e+1]-1,
 * in slot order (a stable counting sort: histogram, prefix scan, stable
 * scatter).  LightMoE README, "MoE training" (gather_indices, m_indptr,
 * routing_weights, inverse_slots) and "Grouped GEMM"; LigerCute README,
 * "Forward pass" (routed tokens are sorted and copied before the expert loop).
 *   topk_ids     [T, k] int32, input, entries in [0, E).
 *   topk_w       [T, k] float32, input; may be NULL when w_perm is NULL.
 *   x            [T, H] bf16, input; may be NULL when x_perm is NULL.
 *   counts       [E] int32, output: rows per expert.
 *   m_indptr     [E+1] int32, output: exclusive prefix sum of counts.
 *   row_to_slot  [R] int32, output: slot of each row.
 *   slot_to_row  [R] int32, output: row of each slot (the inverse).
 *   w_perm       [R] float32, output or NULL: topk_w of each row's slot.
 *   x_perm       [R, H] bf16, output or NULL: x[row_to_slot[r] / k].
 * Workspace: per-chunk expert histograms (a few hundred KB at R = 82k, E = 512).
 * Integer outputs are bit-exact and independent of the launch.
 */
int liger_moe_dispatch(const int32_t* topk_ids, const float* topk_w, const void* x, int T, int H, int E,
                       int k, int32_t* counts, int32_t* m_indptr, int32_t* row_to_slot,
                       int32_t* slot_to_row, float* w_perm, void* x_perm, void* workspace,
                       size_t* workspace_bytes, void* stream);

/*
 * liger_moe_dispatch_noalloc: liger_moe_dispatch for callers that cannot
 * allocate device memory (a static memory plan with no room for a workspace,
 * a plug-in limited to the tensors it is handed, host code that must not
 * allocate mid-step).  It has no counterpart in the pages; it exists for such
 * callers.  Same arguments, outputs and results as liger_moe_dispatch, minus
 * the workspace: its scratch is a fixed 1 MiB array inside this library,
 * present in the memory of every GPU that loads the library until the
 * process exits.  It allocates nothing and frees nothing.
 *   Limit: ceil(T*k / 256) * E * 4 <= 1 MiB (T*k <= 131072 at E = 512,
 *   T*k <= 65536 at E = 1024);
 *   larger sizes return LIGER_MOE_ERR_CAPACITY before anything is launched.
 *   The first call on each device looks up the array's device address; make
 *   that first call before any stream capture.
 *   All calls on a device share the array: calls that overlap on the GPU
 *   (e.g. on two streams with no ordering between them) race and give wrong
 *   results.  The array keeps the last call's contents; nothing in it needs
 *   to start at zero.
 */
int liger_moe_dispatch_noalloc(const int32_t* topk_ids, const float* topk_w, const void* x, int T, int H, int E,
                               int k, int32_t* counts, int32_t* m_indptr, int32_t* row_to_slot,
                               int32_t* slot_to_row, float* w_perm, void* x_perm, void* stream);

/*
 * Grouped SwiGLU expert MLP on expert-major rows, with the routing weight
 * applied to the down projection.  LightMoE README, "Grouped GEMM"
 * (out = a[rows_e] @ b[e]^T, b laid out [num_experts, N, K]) and "MoE
 * inference" (gate/up projection, gated activation, down projection,
 * routing-weight application); LigerCute README, "Forward pass".
 *   x_perm     [R, H] bf16, input (rows in expert-major order).
 *   m_indptr   [E+1] int32, input, as produced by liger_moe_dispatch.
 *   w_gate_up  [E, 2I, H] bf16: rows [0, I) gate, rows [I, 2I) up.
 *   w_down     [E, H, I] bf16.
 *   w_perm     [R] float32: routing weight of each row.
 *   h_perm     [R, I] bf16, output: h = bf16(silu(g) * u)  (saved for backward).
 *   gu_perm    [R, 2I] float32, output or NULL: the SwiGLU derivative factors
 *              [dh/dg | dh/du] = [u s (1 + g (1 - s)) | g s], s = sigmoid(g), from
 *              the fp32 accumulators g, u (saved for backward; when NULL the
 *              backward recomputes them).
 *   y_perm     [R, H] bf16, output: bf16(w_perm[r] * (h W_d[e]^T)).
 * fp32 accumulation on the tensor cores.  Workspace: the tile schedule
 * (4*(E+1) bytes, rounded up).
 */
int liger_moe_grouped_swiglu_fwd(const void* x_perm, const int32_t* m_indptr, const void* w_gate_up,
                                 const void* w_down, const float* w_perm, int R, int H, int I, int E,
                                 void* h_perm, float* gu_perm, void* y_perm, void* workspace,
                                 size_t* workspace_bytes, void* stream);

/*
 * The expert MLP with another activation (enum liger_moe_activation) in place of SwiGLU;
 * everything else as liger_moe_grouped_swiglu_fwd.  gu_perm receives that activation's
 * derivative factors [dh/dg | dh/du], so for a gated activation liger_moe_bwd_dx_dw applies
 * to the result unchanged when gu_perm is saved.  LIGER_MOE_ACT_RELU2: w_gate_up is the up
 * weight W_up [E, I, H] and gu_perm [R, I] receives dh/da (its backward is
 * liger_moe_bwd_dx_dw_glu with LIGER_MOE_ACT_RELU2).
 *   activation  LIGER_MOE_ACT_*; anything else is LIGER_MOE_ERR_INVALID_ARG.
 *   clamp       c of the bounded SwiGLU and the limit of SwiGLU-OAI: finite and > 0 for those
 *               two (else LIGER_MOE_ERR_INVALID_ARG); ignored by the others.
 */
int liger_moe_grouped_glu_fwd(const void* x_perm, const int32_t* m_indptr, const void* w_gate_up,
                              const void* w_down, const float* w_perm, int R, int H, int I, int E,
                              int activation, float clamp, void* h_perm, float* gu_perm, void* y_perm,
                              void* workspace, size_t* workspace_bytes, void* stream);

/*
 * The same expert MLP on token-major input: row r's input is x[row_to_slot[r] / k],
 * copied row by row by the gate/up GEMM's loader straight from x, so no
 * expert-major copy of x is written or read (memory-lean; on GB300 the loader's
 * row copies make this GEMM several times slower than the x_perm entry point).
 * LightMoE README, "MoE inference" (the layer is called with token-major x and
 * the routing ids, and copies rows in expert order itself).  Outputs are
 * identical to liger_moe_dispatch's x_perm followed by
 * liger_moe_grouped_swiglu_fwd.
 *   x            [T, H] bf16, input.
 *   row_to_slot  [R] int32, input (R = T*k), as produced by liger_moe_dispatch;
 *                a value outside [0, R) sets LIGER_MOE_DEVERR_BAD_ROW and reads token 0.
 * Other arguments, outputs and the workspace as liger_moe_grouped_swiglu_fwd.
 */
int liger_moe_grouped_swiglu_fwd_gather(const void* x, const int32_t* row_to_slot, int T, int k,
                                        const int32_t* m_indptr, const void* w_gate_up, const void* w_down,
                                        const float* w_perm, int H, int I, int E, void* h_perm, float* gu_perm,
                                        void* y_perm, void* workspace, size_t* workspace_bytes, void* stream);

/*
 * Combine: routed rows back to token order.  LigerCute README, "Forward
 * pass" (final local combine); LightMoE README, "Highlights" (deterministic
 * combine).
 *   y_perm       [R, H] bf16, input (already weighted).
 *   slot_to_row  [R] int32, input.
 *   y            [T, H] bf16, output: bf16( sum_{j=0..k-1} y_perm[slot_to_row[t*k+j]] ),
 *                float sum in j order (deterministic).
 * No workspace.
 */
int liger_moe_combine(const void* y_perm, const int32_t* slot_to_row, int T, int H, int k, void* y,
                      void* stream);

/*
 * Backward of the whole layer for L = <dY, Y>.  LigerCute README, "Backward
 * pass" (expert-output gradients, recomputed activations, input and weight
 * gradients, routed dX reduced back to tokens); LightMoE README, "MoE
 * training" (deterministic input-, weight- and router-gradient kernels).
 * Inputs are the forward's saved state:
 *   dy [T, H] bf16; x_perm [R, H] bf16; h_perm [R, I] bf16;
 *   gu_perm [R, 2I] float32 derivative factors or NULL (then recomputed from x_perm);
 *   topk_ids, topk_w [T, k]; m_indptr [E+1]; row_to_slot, slot_to_row [R];
 *   w_perm [R]; w_gate_up [E, 2I, H]; w_down [E, H, I].
 * Outputs (overwritten):
 *   dx          [T, H] bf16      sum over the token's k rows of dgu W_gu[e]
 *   dw_gate_up  [E, 2I, H] bf16  sum over expert rows of dgu^T x (zero for empty experts)
 *   dw_down     [E, H, I] bf16   sum over expert rows of (w dY)^T h
 *   d_logits    [T, E] float32   w_j (gamma_j - sum_i w_i gamma_i) at the selected
 *                                experts, gamma_j = <dY, expert-j output>; 0 elsewhere
 * Weight gradients are summed in a fixed order (no atomics): results are
 * identical from run to run.  The upstream gradient enters the expert GEMMs
 * unscaled (copied to expert-major order in the workspace); the routing
 * weight is applied in fp32 to the dH accumulator.  The weight-gradient GEMMs
 * take their non-input operand (dgu for dW_gate_up, w * h for dW_down) as two
 * bf16 parts, hi + lo, so that operand carries about 16 significant bits.
 * Experts with at least 384 rows (when R >= 32768 and the experts are gated)
 * take one fp16 pass instead (liger_moe_set_dw_fp16): x and dY rows as
 * fp16(v 2^s) with s set by the tensor's largest magnitude (exact), dgu and
 * w * h as fp16 (11 significant bits) with power-of-two scales derived from
 * it, and the result scaled back exactly.  An expert whose scaled dgu or
 * w * h would leave the fp16 window (overflow, or a largest magnitude too
 * small for full precision) takes the two-part path instead, so every input
 * gets one of the two precisions.
 * Limit: T*k < 2^30.  Workspace: about R*(2H + 6I)*2 bytes, plus R*2I*4 more
 * when gu_perm is NULL, plus R*2H*2 for the fp16 copies when R >= 32768 and
 * the experts are gated.
 */
int liger_moe_bwd_dx_dw(const void* dy, const void* x_perm, const void* h_perm, const float* gu_perm,
                        const int32_t* topk_ids, const float* topk_w, const int32_t* m_indptr,
                        const int32_t* row_to_slot, const int32_t* slot_to_row, const float* w_perm,
                        const void* w_gate_up, const void* w_down, int T, int H, int I, int E, int k,
                        void* dx, void* dw_gate_up, void* dw_down, float* d_logits, void* workspace,
                        size_t* workspace_bytes, void* stream);

/*
 * liger_moe_bwd_dx_dw for a layer whose forward used another activation
 * (liger_moe_grouped_glu_fwd).  For a gated activation, the activation and clamp matter only
 * when gu_perm is NULL, where the derivative factors are recomputed; with saved factors the
 * result equals liger_moe_bwd_dx_dw.  LIGER_MOE_ACT_RELU2 (two-weight experts): w_gate_up is
 * W_up [E, I, H], gu_perm (saved dh/da) [R, I] or NULL, dw_gate_up receives dW_up [E, I, H].
 * Arguments, outputs, limits and workspace otherwise as liger_moe_bwd_dx_dw; activation and
 * clamp are checked as in liger_moe_grouped_glu_fwd.
 */
int liger_moe_bwd_dx_dw_glu(const void* dy, const void* x_perm, const void* h_perm, const float* gu_perm,
                            const int32_t* topk_ids, const float* topk_w, const int32_t* m_indptr,
                            const int32_t* row_to_slot, const int32_t* slot_to_row, const float* w_perm,
                            const void* w_gate_up, const void* w_down, int T, int H, int I, int E, int k,
                            int activation, float clamp, void* dx, void* dw_gate_up, void* dw_down,
                            float* d_logits, void* workspace, size_t* workspace_bytes, void* stream);

/*
 * The same backward on token-major input: x [T, H] bf16 replaces x_perm.  The
 * dH, dW_gate_up and dW_down GEMMs copy the rows of x and dy they need by token
 * (row_to_slot[r] / k) straight from x and dy, so no expert-major copy of
 * either exists (memory-lean, slower, as for the gathered forward).  LightMoE
 * README, "MoE inference" and "MoE training"; LigerCute README, "Backward
 * pass".  Every other argument, output and limit as liger_moe_bwd_dx_dw; the
 * outputs are identical.  Workspace: about R*(H + 6I)*2 bytes, plus R*2I*4
 * more when gu_perm is NULL.
 */
int liger_moe_bwd_dx_dw_gather(const void* dy, const void* x, const void* h_perm, const float* gu_perm,
                               const int32_t* topk_ids, const float* topk_w, const int32_t* m_indptr,
                               const int32_t* row_to_slot, const int32_t* slot_to_row, const float* w_perm,
                               const void* w_gate_up, const void* w_down, int T, int H, int I, int E, int k,
                               void* dx, void* dw_gate_up, void* dw_down, float* d_logits, void* workspace,
                               size_t* workspace_bytes, void* stream);

/*
 * Router projection in front of liger_moe_route_topk: one bias-optional linear layer,
 *   logits[t, e] = sum_h x[t, h] * w_router[e, h] + bias[e]      (fp32 accumulation).
 * The pages leave the router to the host framework (LightMoE README, "MoE training": routing
 * policy is the framework's responsibility); this is its plainest form.  Runs as one dense
 * tcgen05 GEMM (M = T, N = E, K = H); the summation order differs from a sequential sum, so
 * the logits agree with a plain fp32 loop to rounding, not bit for bit.
 *   x         [T, H] bf16, input.
 *   w_router  [E, H] bf16, input.
 *   bias      [E] float32, input, or NULL (no bias); any 4-byte alignment.
 *   logits    [T, E] float32, output (16-byte aligned).
 * No workspace.  Limits: H a multiple of 64; 1 <= E <= 1024.
 */
int liger_moe_router_logits(const void* x, const void* w_router, const float* bias, int T, int H, int E,
                            float* logits, void* stream);

/*
 * Backward of the router projection for the layer's own logit gradient (the d_logits that
 * liger_moe_bwd_dx_dw writes).  Those are zero off each token's top-k selection, so only the
 * selected entries are read:
 *   dx[t, :]         = bf16( dx[t, :] + sum_j d_logits[t, id_j] * w_router[id_j, :] )
 *                      (j = 0..k-1 in slot order, fp32; dx is INPUT AND OUTPUT: the router's
 *                      input gradient is added to the layer's dX in place -- pass zeros for
 *                      the router term alone.  This is the one accumulating output of the ABI.)
 *   dw_router[e, :]  = bf16( sum over expert e's routed rows (token order) of
 *                      d_logits[t, e] * x[t, :] )        (overwritten; zero for an empty expert)
 *   d_bias[e]        = sum over the same rows of d_logits[t, e]   (float32, overwritten), or NULL.
 * Both sums accumulate in fp32 from the exact bf16 inputs, in a fixed order (results are
 * identical from run to run).
 *   d_logits     [T, E] float32, input; entries off the selection are not read (they must be
 *                zero for the result to be the full gradient).
 *   topk_ids     [T, k] int32, input (liger_moe_route_topk); an id outside [0, E) sets
 *                LIGER_MOE_DEVERR_BAD_EXPERT_ID and leaves that token's dx unchanged.
 *   m_indptr     [E+1], row_to_slot [R] int32, inputs: liger_moe_dispatch of the same routing.
 *   x            [T, H] bf16, input (the router's input).
 *   w_router     [E, H] bf16, input.
 * No workspace.  Limits as liger_moe_route_topk and H a multiple of 64.
 */
int liger_moe_router_bwd(const float* d_logits, const int32_t* topk_ids, const int32_t* m_indptr,
                         const int32_t* row_to_slot, const void* x, const void* w_router, int T, int H, int E, int k,
                         void* dx, void* dw_router, float* d_bias, void* stream);

/*
 * Takes the device error flag of the current device after the work already
 * enqueued on `stream`, then synchronises `stream`.  Returns LIGER_MOE_OK and
 * *flags = 0 when no device error was recorded since the last call, or
 * LIGER_MOE_ERR_DEVICE with *flags = the LIGER_MOE_DEVERR_* bits.  The flag is
 * read and cleared in one atomic exchange on the device: a bit that a kernel
 * on another stream sets at the same time is reported now or by the next
 * call, never lost.  Returns LIGER_MOE_ERR_LAUNCH if the launch, the copy or
 * the synchronisation failed.
 */
int liger_moe_device_error(void* stream, int* flags);

/*
 * Precision of the weight-gradient operands of the heavy experts in
 * liger_moe_bwd_dx_dw and liger_moe_bwd_dx_dw_glu (process-wide; default 1):
 *   1  experts with at least 384 rows use the single fp16 pass described there
 *      (half the tensor-core work of the two-part path);
 *   0  every expert uses the bf16 hi + lo parts (about 16 significant bits).
 * The workspace size does not depend on it.  Anything else is LIGER_MOE_ERR_INVALID_ARG.
 */
int liger_moe_set_dw_fp16(int on);

/*
 * Failure-detection self-test (diagnostics).  Launches one kernel in which a thread waits,
 * through the bounded wait that every grouped-GEMM pipeline wait uses, on an mbarrier phase
 * that nothing completes.  After limit_us microseconds the wait gives up and the kernel sets
 * LIGER_MOE_DEVERR_WAIT_TIMEOUT in the device error flag, as a stalled GEMM role would; the
 * context stays usable.  Read the result with liger_moe_device_error().  The GEMMs' own limit
 * is 2 s per wait.
 *   limit_us  1 .. 1000000 (else LIGER_MOE_ERR_INVALID_ARG).
 */
int liger_moe_selftest_wait_timeout(int limit_us, void* stream);

/*
 * Kernel trace (diagnostics; off by default).  While enabled, every kernel
 * this library launches is bracketed by two CUDA events recorded on the
 * launch stream, giving its device-side duration without a profiler.  One
 * logged interval is one kernel, or both launches of a GEMM that runs its
 * heavy and light experts as two launches.
 *   liger_moe_trace_enable(on)       turns tracing on or off and clears the log
 *   liger_moe_trace_count()          number of intervals logged
 *   liger_moe_trace_get(i, ...)      kernel name (static string) and duration in
 *                                    ms of interval i; waits for it to finish
 *   liger_moe_trace_launches(i, n)   number of kernel launches in interval i
 * Host-side cost: two event records per interval while enabled.  The records
 * are "external", so a trace taken while the stream is captured into a CUDA
 * graph times every replay of the captured launches (the last replay wins).
 * Errors: LIGER_MOE_ERR_INVALID_ARG for an index outside the log or a NULL
 * output pointer.
 */
int liger_moe_trace_enable(int on);
int liger_moe_trace_count(void);
int liger_moe_trace_get(int i, const char** name, float* ms);
int liger_moe_trace_launches(int i, int* launches);

/* Text of the last CUDA error seen by this library in this thread ("" if none). */
const char* liger_moe_last_cuda_error(void);

/* Name of a liger_moe_status value. */
const char* liger_moe_status_string(int status);

/* ABI version (major * 100 + minor). */
int liger_moe_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIGER_MOE_H_ */
