/*
 * moe.h - C ABI of libmoe: the forward pass (and, for the BF16 kind, the
 * backward pass) of one DeepSeekMoE layer on one NVIDIA B300 (sm_103a).
 *
 * The layer is the one of the "DeepSeek-V3 Technical Report":
 *   - DeepSeekMoE paragraph: token t's FFN output is the sum of N_s shared
 *     experts plus the gate-weighted outputs of K routed experts; the
 *     affinity of token t to routed expert i is sigmoid(u_t . e_i) and the
 *     gates are the selected affinities normalised among themselves;
 *   - auxiliary-loss-free load balancing paragraph: a per-expert bias b_i is
 *     added to the affinity only to choose the top-K; after each step b_i
 *     goes down by gamma if expert i was overloaded, up by gamma otherwise;
 *     node-limited routing (here: group-limited); no token is dropped;
 *   - fine-grained quantisation and increased-precision accumulation
 *     paragraphs, Appendix B.2: FP8 E4M3 with one scale per 1 x 128
 *     activation tile and per 128 x 128 weight block, FP32 accumulation.
 *
 * One call per step of the layer:
 *     moe_route -> moe_permute -> moe_experts_grouped -> moe_combine
 *               -> moe_bias_update
 * and, for training (BF16 kind), four calls for its backward pass (see
 * "backward pass" below).
 *
 * Conventions shared by every call
 *   - All tensors are dense, row-major, in device memory allocated and owned
 *     by the caller.  The library allocates no memory and keeps no state
 *     between calls except a per-device 32-bit error word.
 *   - Every call enqueues its kernels on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and returns without synchronising.  The
 *     host never learns the per-expert loads: every kernel reads them from
 *     device memory.
 *   - Arguments are checked on the host before anything is launched; a
 *     failed check returns an error status and launches nothing.
 *   - Faults found on the device (a wait that timed out, an index out of
 *     range) never trap: they set bits in the error word, which
 *     moe_get_device_error() reads and clears.
 *   - Pointers must be 16-byte aligned.  For the BF16 and FP8 kinds, d and
 *     I must be multiples of 128.
 *   - Results are deterministic: the same inputs give bitwise-identical
 *     outputs (no atomics decide any output order or floating-point sum).
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Arithmetic kind of the expert path. */
typedef enum {
  MOE_DTYPE_FP32 = 0,     /* x, weights, intermediates and output in fp32 */
  MOE_DTYPE_BF16 = 1,     /* x, weights, h, y in bf16; fp32 accumulation  */
  MOE_DTYPE_FP8_E4M3 = 2  /* x in bf16, quantised to E4M3 per 1x128 tile;
                             weights E4M3 + fp32 128x128 block scales;
                             fp32 accumulation; bf16 output              */
} moe_dtype_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer or inconsistent configuration */
  MOE_ERR_SHAPE = 2,        /* size outside what a kernel supports          */
  MOE_ERR_ALIGN = 3,        /* pointer not 16-byte aligned                  */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call failed                   */
  MOE_ERR_TIMEOUT = 5,      /* a device wait gave up (error word)           */
  MOE_ERR_DEVICE = 6,       /* another device-side check failed             */
  MOE_ERR_WORKSPACE = 7     /* workspace smaller than moe_workspace_bytes   */
} moe_status_t;

/* Shape of one layer.  Symbols of the DeepSeekMoE paragraph: N_r = E routed
 * experts, K_r = K active per token, N_s = n_shared; node-limited routing
 * reads as n_groups contiguous groups of E / n_groups experts of which a
 * token may use topk_groups. */
typedef struct {
  int32_t T;                /* tokens in the batch                          */
  int32_t d;                /* hidden size (FFN input/output width)         */
  int32_t E;                /* routed experts                               */
  int32_t n_groups;         /* expert groups (E % n_groups == 0)            */
  int32_t topk_groups;      /* groups a token may use                       */
  int32_t K;                /* routed experts per token                     */
  int32_t n_shared;         /* shared experts (0 allowed)                   */
  int32_t inter;            /* intermediate size I of every expert          */
  int32_t group_score_topn; /* a group's score: sum of its top-n biased
                               affinities (2 in the DeepSeek-V3 reading)    */
  float route_scale;        /* rho: gates sum to rho for every token        */
  float gamma;              /* bias update speed                            */
  int32_t dtype;            /* moe_dtype_t                                  */
} moe_cfg_t;

/* Human-readable name of a status. */
const char* moe_status_str(moe_status_t status);

/* Library version as 10000*major + 100*minor + patch. */
int32_t moe_version(void);

/* Checks a configuration: MOE_OK, MOE_ERR_INVALID_ARG or MOE_ERR_SHAPE.
 * Limits: 1 <= T <= 2^22; 1 <= E <= 1024; 1 <= K <= min(32, E);
 * n_groups divides E; 1 <= topk_groups <= n_groups <= 32; the kept groups
 * hold at least K experts; 1 <= group_score_topn; d, inter >= 1. */
moe_status_t moe_check_cfg(const moe_cfg_t* cfg);

/* Bytes of scratch memory that moe_route and moe_experts_grouped need for
 * this configuration (one buffer serves both; contents need not survive
 * between calls).  0 for an invalid configuration. */
size_t moe_workspace_bytes(const moe_cfg_t* cfg);

/*
 * moe_route - affinities, group-limited top-K, gates, per-expert segments.
 *
 * DeepSeekMoE paragraph (sigmoid affinity, gates normalised among the
 * selected affinities) and auxiliary-loss-free paragraph (bias for the
 * choice only; no token dropped).
 *
 *   x            [T, d]   fp32 (FP32 kind) or bf16 (BF16 / FP8 kinds)
 *   router_w     [E, d]   fp32 centroids e_i (routing stays in fp32)
 *   bias         [E]      fp32 b_i
 *   affinity_in  [T, E]   fp32, nullable: when given, these affinities are
 *                         used as s and the router product is skipped
 *   affinity_out [T, E]   fp32, nullable: receives s = sigmoid(x e^T)
 *   topk_idx     [T, K]   int32 out: chosen experts by descending biased
 *                         score fl32(s + b), ties to the lower index
 *   topk_w       [T, K]   fp32 out: rho * s / sum of the chosen s
 *   counts       [E]      int32 out: tokens routed to each expert
 *   offsets      [E + 1]  int32 out: exclusive prefix sum of counts
 *   row_of_slot  [T, K]   int32 out: permuted row of token t's k-th copy
 *   token_of_row [T * K]  int32 out: token copied into each permuted row;
 *                         inside an expert's segment rows follow ascending
 *                         token index
 *   ws, ws_bytes          scratch, at least moe_workspace_bytes(cfg)
 *
 * Group score: the fp32 sum, in descending order, of the group's top
 * group_score_topn biased scores; groups are kept by descending score,
 * ties to the lower group index.  Bit-exact given the same fp32 s.
 */
moe_status_t moe_route(const moe_cfg_t* cfg, const void* x, const float* router_w,
                       const float* bias, const float* affinity_in,
                       float* affinity_out, int32_t* topk_idx, float* topk_w,
                       int32_t* counts, int32_t* offsets, int32_t* row_of_slot,
                       int32_t* token_of_row, void* ws, size_t ws_bytes,
                       void* stream);

/*
 * moe_permute - copy every token row into its experts' segments
 * (the single-device form of the dispatch of the cross-node all-to-all
 * paragraph).
 *
 *   x             [T, d]      fp32 / bf16 input rows
 *   token_of_row  [T * K]     from moe_route
 *   x_perm        [T * K, d]  out: FP32 kind fp32, BF16 kind bf16, FP8 kind
 *                             E4M3 bytes (row r = x[token_of_row[r]])
 *   x_perm_scales [T * K, d/128] fp32 out, FP8 kind only (else NULL): the
 *                 1 x 128 tile scales fl32(amax / 448), 1 for a zero tile
 *   x_q, x_q_scales  FP8 kind only (else NULL): [T, d] E4M3 and
 *                 [T, d/128] fp32 - each token quantised once, before the
 *                 copies ("dispatch activations in FP8"); the shared expert
 *                 reads them too
 */
moe_status_t moe_permute(const moe_cfg_t* cfg, const void* x,
                         const int32_t* token_of_row, void* x_perm,
                         float* x_perm_scales, void* x_q, float* x_q_scales,
                         void* stream);

/*
 * moe_experts_grouped - every routed expert's SwiGLU FFN on its segment,
 * plus the shared experts on all T tokens.
 *
 * DeepSeekMoE paragraph (fine-grained routed experts and shared experts;
 * every expert is W2 (silu(W1 u) * (W3 u))).
 *
 *   x_perm, x_perm_scales  from moe_permute (scales: FP8 kind only)
 *   x, x_scales   [T, d] shared-expert input rows: the layer input (FP32 /
 *                 BF16 kinds; x_scales NULL) or moe_permute's x_q and
 *                 x_q_scales (FP8 kind)
 *   offsets       [E + 1] from moe_route
 *   w13           [E, 2I, d] rows [0, I) = W1 (gate), [I, 2I) = W3 (up)
 *   w2            [E, d, I]
 *   ws13, ws2     [N_s, 2I, d], [N_s, d, I] shared experts (NULL if N_s = 0)
 *   *_scales      FP8 kind: fp32 block scales of the weight above it,
 *                 [E, 2I/128, d/128], [E, d/128, I/128], [N_s, ...]
 *                 (see moe_quantize_weights_fp8); NULL otherwise
 *   y_perm        [T * K, d] out: expert output of every permuted row
 *                 (fp32 for the FP32 kind, else bf16)
 *   y_shared      [T, d] out: sum of the shared experts' outputs (NULL
 *                 if N_s = 0)
 *
 * The N_s shared experts are evaluated as one expert of intermediate size
 * N_s * I (the same sum, in one fp32 accumulator).
 */
moe_status_t moe_experts_grouped(const moe_cfg_t* cfg, const void* x_perm,
                                 const float* x_perm_scales, const void* x,
                                 const float* x_scales, const int32_t* offsets,
                                 const void* w13, const float* w13_scales,
                                 const void* w2, const float* w2_scales,
                                 const void* ws13, const float* ws13_scales,
                                 const void* ws2, const float* ws2_scales,
                                 void* y_perm, void* y_shared, void* ws,
                                 size_t ws_bytes, void* stream);

/*
 * moe_experts_grouped_gather - moe_experts_grouped with the permute folded
 * into the gate/up GEMM: the routed A rows are read straight from x by
 * token_of_row instead of from a permuted copy (the single-device dispatch
 * of the cross-node all-to-all paragraph, done while the expert GEMM loads
 * its operands; x_perm is never written).
 *
 *   x             [T, d] bf16: the layer input (routed and shared rows)
 *   token_of_row  [T * K] from moe_route
 *   everything else as in moe_experts_grouped (x_perm is not an argument)
 *
 * BF16 kind only (MOE_ERR_SHAPE otherwise).  Results are bitwise equal to
 * moe_permute followed by moe_experts_grouped.  A token index outside
 * [0, T) sets the error word (MOE_ERR_DEVICE) and its row is skipped.
 */
moe_status_t moe_experts_grouped_gather(const moe_cfg_t* cfg, const void* x,
                                        const float* x_scales, const int32_t* token_of_row,
                                        const int32_t* offsets, const void* w13,
                                        const float* w13_scales, const void* w2,
                                        const float* w2_scales, const void* ws13,
                                        const float* ws13_scales, const void* ws2,
                                        const float* ws2_scales, void* y_perm, void* y_shared,
                                        void* ws, size_t ws_bytes, void* stream);

/*
 * moe_experts_grouped_gated - moe_experts_grouped with the gate multiply of
 * the DeepSeekMoE paragraph's weighted sum folded into the down projection:
 *   y_perm[r] = g_{t,k} * FFN_e(u_t)   for the copy (t, k) that row r holds,
 * the gate applied to the fp32 sum before the one rounding to the output
 * type.  moe_combine(..., topk_w = NULL, ...) then only adds the rows.
 *
 *   row_of_slot, topk_w  [T, K] from moe_route (required)
 *   everything else as in moe_experts_grouped; y_shared is not gated
 *
 * All kinds.  The gates of the permuted rows are scattered into the
 * workspace first (one small kernel): moe_workspace_bytes covers them.  A
 * row index outside [0, T*K) sets the error word (MOE_ERR_DEVICE) and is
 * skipped.  The backward pass needs the ungated y_perm (dL/dg = dL/dy . y):
 * train with moe_experts_grouped_train and the gated moe_combine.
 */
moe_status_t moe_experts_grouped_gated(const moe_cfg_t* cfg, const void* x_perm,
                                       const float* x_perm_scales, const void* x,
                                       const float* x_scales, const int32_t* offsets,
                                       const void* w13, const float* w13_scales,
                                       const void* w2, const float* w2_scales,
                                       const void* ws13, const float* ws13_scales,
                                       const void* ws2, const float* ws2_scales,
                                       const int32_t* row_of_slot, const float* topk_w,
                                       void* y_perm, void* y_shared, void* ws,
                                       size_t ws_bytes, void* stream);

/*
 * moe_combine - gate-weighted un-permute:
 *   out[t] = y_shared[t] + sum_{k < K} topk_w[t, k] * y_perm[row_of_slot[t, k]]
 * summed in fp32 in exactly that order (DeepSeekMoE paragraph).
 *
 *   y_perm [T*K, d], y_shared [T, d] (nullable): fp32 (FP32 kind) or bf16
 *   topk_w [T, K] fp32, or NULL when y_perm already holds the gated rows
 *          of moe_experts_grouped_gated (then out[t] = y_shared[t] +
 *          sum_k y_perm[row_of_slot[t, k]], same order)
 *   out    [T, d] fp32 (FP32 kind) or bf16
 */
moe_status_t moe_combine(const moe_cfg_t* cfg, const void* y_perm,
                         const void* y_shared, const int32_t* row_of_slot,
                         const float* topk_w, void* out, void* stream);

/*
 * moe_bias_update - the sign rule of the auxiliary-loss-free paragraph:
 *   b_i <- fl32(b_i - gamma) if counts_i * E > T * K   (overloaded)
 *   b_i <- fl32(b_i + gamma) otherwise
 *   counts [E] int32 (from moe_route), bias [E] fp32 in/out.
 * Only E, K, T and gamma are read, and only these are checked: 1 <= E <=
 * 1024, 1 <= K <= min(32, E), T >= 1, gamma not NaN (MOE_ERR_INVALID_ARG /
 * MOE_ERR_SHAPE otherwise; pointers are checked after the shape).  T may
 * exceed moe_route's limit of 2^22 tokens: data-parallel replicas pass the
 * whole batch, world size x T, with counts summed over the replicas.
 */
moe_status_t moe_bias_update(const moe_cfg_t* cfg, const int32_t* counts,
                             float* bias, void* stream);

/*
 * moe_balance_stat - the sequence-wise balance statistic
 *     L_Bal = alpha * sum_i f_i P_i
 * of every sequence of seq_len consecutive tokens (auxiliary-loss-free
 * paragraph: the complementary sequence-wise balance loss, with a small
 * factor alpha, 0.0001 in the training hyper-parameters).  The pages do not
 * define f_i and P_i; here
 *     f_i = E / (K * seq_len) * (selections of expert i in the sequence)
 *     P_i = mean over the sequence's tokens of s_i / sum_j s_j
 * so an even split gives f_i = 1.  Forward statistic only (no gradient).
 *
 *   affinity  [T, E]  fp32 unbiased s (moe_route's affinity_out)
 *   topk_idx  [T, K]  int32 from moe_route
 *   seq_len   divides T; T / seq_len <= 65535 sequences
 *   f_out, p_out [T / seq_len, E] fp32 out; loss_out [T / seq_len] fp32 out
 *   ws, ws_bytes  scratch for per-chunk partial sums: 2 * align256(4 *
 *                 (T / seq_len) * ceil(seq_len / 256) * E) bytes, which
 *                 moe_workspace_bytes(cfg) covers for seq_len >= 2
 *                 (MOE_ERR_WORKSPACE if too small)
 * Sums are fp32 in a fixed order (deterministic).
 */
moe_status_t moe_balance_stat(const moe_cfg_t* cfg, const float* affinity,
                              const int32_t* topk_idx, int32_t seq_len, float alpha,
                              float* f_out, float* p_out, float* loss_out, void* ws,
                              size_t ws_bytes, void* stream);

/*
 * ------------------------------------------------------------ backward pass
 * BF16 kind only (MOE_ERR_SHAPE otherwise; also for n_shared > 64).
 *
 * The chain rule of the layer above with the top-K selection held fixed (a
 * choice has no gradient) and no gradient for the selection bias (it only
 * steers the choice, auxiliary-loss-free paragraph).  Mixed precision
 * framework paragraph: each linear has a Dgrad and a Wgrad GEMM next to
 * its Fprop; DualPipe paragraph: the MLP backward splits into backward for
 * input and backward for weights.  One step, given dL/dy (`dout`) and the
 * forward's routing outputs:
 *     moe_combine_backward -> moe_experts_backward_input
 *         -> moe_route_backward        (dx and dL/de: input side complete)
 *         -> moe_experts_backward_weights
 * (with moe_experts_grouped_train in place of moe_experts_grouped in the
 * forward, the input call skips recomputing the gate/up products).
 * The weights call may run any time after the input call, on the same
 * workspace (it reads the intermediates the input call left there).
 *
 * With a = x W1^T, b = x W3^T, h = silu(a) b, g = rho s / S:
 *   dy_perm[row(t,k)] = g_{t,k} dout_t          dgate_{t,k} = dout_t . y_perm[row(t,k)]
 *   dh = dy W2,  da = dh b silu'(a),  db = dh silu(a),  dx_e = [da | db] W13
 *   dW2 = dy^T h,  dW13 = [da | db]^T x  (per expert, over its segment)
 *   ds_k = rho / S (dgate_k - sum_j dgate_j s_j / S),  dlogit_k = ds_k s_k (1 - s_k)
 *   dx_t = dx_shared_t + sum_k (dx_perm[row(t,k)] + dlogit_{t,k} e_{idx(t,k)})
 *   drouter_w_i = sum over the tokens t that chose i of dlogit_{t,k} x_t
 * All GEMMs accumulate in fp32; every stored intermediate and gradient is
 * bf16 except dgate, dlogit and drouter_w (fp32).  Sums run in a fixed
 * order: results are deterministic.
 */

/* Scratch of the backward calls: the expert part, then align256(T*K*4)
 * bytes for moe_route_backward.  BF16 kind: align256((T*K + T*N_s) * 3I * 2)
 * bytes of expert intermediates ([a | b] then [da | db], and h; they must
 * survive from moe_experts_backward_input to moe_experts_backward_weights).
 * FP8 kind (N_s <= 1): the buffers of moe_experts_backward_input_fp8 for
 * T*K + T rows (q(dy) codes and scales, [a | b] and dh in bf16, q([da | db])
 * codes and scales), then those of moe_experts_backward_weights_fp8 (the
 * segments' padded starts and the four transposed 128 x 1-tile operands).  0 for a configuration the backward does not support.
 * moe_combine_backward and moe_route_backward take both kinds (their data
 * are bf16 in both); the other backward calls name their kind. */
size_t moe_backward_workspace_bytes(const moe_cfg_t* cfg);

/*
 * moe_combine_backward - gradient of moe_combine.
 *   dout        [T, d]    bf16 dL/dy of the layer output
 *   y_perm      [T*K, d]  bf16 routed expert outputs of the forward
 *   row_of_slot [T, K], topk_w [T, K]  from moe_route
 *   dy_perm     [T*K, d]  bf16 out: g_{t,k} dout_t at row(t,k)
 *   dgate       [T, K]    fp32 out: dout_t . y_perm[row(t,k)]
 * A row index outside [0, T*K) sets the error word; that slot is skipped.
 */
moe_status_t moe_combine_backward(const moe_cfg_t* cfg, const void* dout, const void* y_perm,
                                  const int32_t* row_of_slot, const float* topk_w,
                                  void* dy_perm, float* dgate, void* stream);

/*
 * moe_experts_grouped_train - moe_experts_grouped (BF16 kind) for a
 * training step: the same outputs, and the gate/up epilogue also keeps
 * a = x W1^T and b = x W3^T of every routed row and shared expert (bf16)
 * in the backward workspace `bws`, so that moe_experts_backward_input with
 * ab_kept = 1 does not recompute them (0.5 GB written at the DeepSeek-V3
 * shape instead of 4.3 TFLOP recomputed).
 *   arguments as in moe_experts_grouped (no scales), plus
 *   bws, bws_bytes   at least moe_backward_workspace_bytes(cfg); pass the
 *                    same buffer to the backward calls of this step
 */
moe_status_t moe_experts_grouped_train(const moe_cfg_t* cfg, const void* x_perm, const void* x,
                                       const int32_t* offsets, const void* w13, const void* w2,
                                       const void* ws13, const void* ws2, void* y_perm,
                                       void* y_shared, void* ws, size_t ws_bytes, void* bws,
                                       size_t bws_bytes, void* stream);

/*
 * moe_experts_backward_input - Dgrad of every expert FFN: [a | b] (kept by
 * moe_experts_grouped_train, or recomputed with the forward's grouped
 * GEMM), then dh, the SwiGLU backward and dx, leaving [da | db] (over
 * [a | b]) and h in `ws` for moe_experts_backward_weights.
 *   x_perm [T*K, d], x [T, d]       bf16 forward inputs (routed / shared)
 *   offsets [E + 1]                 from moe_route
 *   w13, w2, ws13, ws2              as in moe_experts_grouped
 *   dy_perm [T*K, d]                from moe_combine_backward
 *   dout    [T, d]                  dL/dy (the shared experts' dy)
 *   dx_perm [T*K, d]   bf16 out: routed experts' input gradient per row
 *   dx_shared [T, d]   bf16 out: sum of the shared experts' input
 *                      gradients (NULL if N_s = 0)
 *   ab_kept            nonzero: `ws` holds [a | b] from this step's
 *                      moe_experts_grouped_train (consumed: the call
 *                      overwrites it with [da | db]); 0: recompute it
 *   ws, ws_bytes       at least moe_backward_workspace_bytes(cfg)
 */
moe_status_t moe_experts_backward_input(const moe_cfg_t* cfg, const void* x_perm,
                                        const void* x, const int32_t* offsets, const void* w13,
                                        const void* w2, const void* ws13, const void* ws2,
                                        const void* dy_perm, const void* dout, void* dx_perm,
                                        void* dx_shared, int32_t ab_kept, void* ws,
                                        size_t ws_bytes, void* stream);

/*
 * moe_experts_backward_weights - Wgrad of every expert FFN from the
 * intermediates moe_experts_backward_input left in `ws` (same cfg, same
 * offsets, workspace untouched in between except by moe_route_backward).
 *   x_perm, x, offsets, dy_perm, dout   as for the input call
 *   dw13 [E, 2I, d], dw2 [E, d, I]      bf16 out (an expert with no rows
 *                                       gets zeros)
 *   dws13 [N_s, 2I, d], dws2 [N_s, d, I] bf16 out (NULL if N_s = 0)
 */
moe_status_t moe_experts_backward_weights(const moe_cfg_t* cfg, const void* x_perm,
                                          const void* x, const int32_t* offsets,
                                          const void* dy_perm, const void* dout, void* dw13,
                                          void* dw2, void* dws13, void* dws2, void* ws,
                                          size_t ws_bytes, void* stream);

/*
 * moe_route_backward - gradient through the gates and the sigmoid router,
 * and the layer's input gradient.
 *   x [T, d] bf16, router_w [E, d] fp32     forward inputs
 *   affinity [T, E] fp32                    the s the gates were made from
 *                                           (moe_route's affinity_out)
 *   topk_idx, row_of_slot, token_of_row, offsets   from moe_route
 *   dgate [T, K] fp32                       from moe_combine_backward
 *   dx_perm, dx_shared                      from moe_experts_backward_input
 *   dlogit [T, K] fp32 out: dL/d(x . e) of every selected expert
 *   dx [T, d] bf16 out: dL/dx of the layer input
 *   drouter_w [E, d] fp32 out: dL/de (zero rows for unchosen experts)
 *   ws, ws_bytes  the backward workspace (its last T*K*4 bytes)
 */
moe_status_t moe_route_backward(const moe_cfg_t* cfg, const void* x, const float* router_w,
                                const float* affinity, const int32_t* topk_idx,
                                const float* dgate, const int32_t* row_of_slot,
                                const int32_t* token_of_row, const int32_t* offsets,
                                const void* dx_perm, const void* dx_shared, float* dlogit,
                                void* dx, float* drouter_w, void* ws, size_t ws_bytes,
                                void* stream);

/*
 * moe_transpose_weights_fp8 - offline utility for the FP8 backward:
 * transposes `n_mats` E4M3 matrices [rows, cols] (rows, cols % 128 == 0) to
 * [cols, rows], and their 128 x 128 block scales [n, rows/128, cols/128] to
 * [n, cols/128, rows/128].  The blocks are the same blocks, so a transposed
 * copy quantises nothing again: W2 [E, d, I] gives W2^T [E, I, d] and W13
 * [E, 2I, d] gives W13^T [E, d, 2I] for moe_experts_backward_input_fp8.
 */
moe_status_t moe_transpose_weights_fp8(const void* w_q, const float* w_scales,
                                       int32_t n_mats, int32_t rows, int32_t cols,
                                       void* wt_q, float* wt_scales, void* stream);

/*
 * moe_quantize_act_fp8_128x1 - E4M3 quantisation of bf16 x [rows, cols] in
 * 128 x 1 tiles (128 consecutive rows of one column), the tiles Wgrad's
 * operands use (moe_experts_backward_weights_fp8 quantises dy, u, h and
 * [da | db] this way, per segment):
 *   scale[t][c] = fl32(amax / 448) over rows 128t .. 128t + 127 of column c
 *                 (1 for an all-zero tile; a ragged last tile over the rows
 *                 it has)
 *   q[r][c]     = E4M3(fl32(x[r][c] / scale)), nearest even, saturating
 *   x       [rows, cols] bf16, cols % 128 == 0
 *   q       [ceil(rows/128) * 128, cols] E4M3 out (the rows past `rows` of the
 *           last tile are written as zero codes)
 *   scales  [ceil(rows/128), cols] fp32 out
 * MOE_ERR_SHAPE when cols is not a multiple of 128.
 */
moe_status_t moe_quantize_act_fp8_128x1(const void* x, int32_t rows, int32_t cols, void* q,
                                        float* scales, void* stream);

/*
 * moe_experts_backward_input_fp8 - Dgrad of every expert FFN in FP8 E4M3
 * (mixed precision framework paragraph, Figure 6: Dgrad in FP8 with fp32
 * accumulation; fine-grained quantisation paragraph: 1 x 128 activation
 * tiles, 128 x 128 weight blocks).  The gradients are tiled along the
 * contraction of their GEMM, so that each tile's scale factors out:
 *   [a | b] = u W13^T   recomputed from the forward's E4M3 codes of u
 *                       (unless moe_experts_grouped_train_fp8 kept it)
 *   dh = q(dy) W2       dy (bf16) in 1 x 128 tiles along d
 *   da = dh b silu'(a), db = dh silu(a)   in fp32
 *   du = q([da | db]) W13   [da | db] in 1 x 128 tiles along 2I
 * with scale fl32(amax / 448) per tile and fp32 promotion of every
 * 128-deep partial sum, as in the FP8 forward.
 *   x_perm, x_perm_scales    the forward's E4M3 rows and scales (moe_permute)
 *   x_q, x_q_scales          the forward's E4M3 token rows (shared expert)
 *   offsets [E + 1]          from moe_route
 *   w13, w13_scales          [E, 2I, d] forward codes and block scales
 *   w13t, w13t_scales        [E, d, 2I] their transpose (moe_transpose_weights_fp8)
 *   w2t, w2t_scales          [E, I, d]  the transpose of the forward's W2
 *   ws13.., ws13t.., ws2t..  the same for the shared expert (NULL if N_s = 0)
 *   dy_perm [T*K, d] bf16    from moe_combine_backward
 *   dout    [T, d] bf16      dL/dy of the layer (the shared expert's dy)
 *   dx_perm [T*K, d] bf16 out, dx_shared [T, d] bf16 out (NULL if N_s = 0)
 *   ab_kept                  nonzero: `ws` holds [a | b] from this step's
 *                            moe_experts_grouped_train_fp8 (not recomputed)
 *   ws, ws_bytes             at least moe_backward_workspace_bytes(cfg)
 * FP8 kind with at most one shared expert (MOE_ERR_SHAPE otherwise).  It
 * leaves [a | b] and dh in `ws` for moe_experts_backward_weights_fp8.
 */
moe_status_t moe_experts_backward_input_fp8(
    const moe_cfg_t* cfg, const void* x_perm, const float* x_perm_scales, const void* x_q,
    const float* x_q_scales, const int32_t* offsets, const void* w13, const float* w13_scales,
    const void* w13t, const float* w13t_scales, const void* w2t, const float* w2t_scales,
    const void* ws13, const float* ws13_scales, const void* ws13t, const float* ws13t_scales,
    const void* ws2t, const float* ws2t_scales, const void* dy_perm, const void* dout,
    void* dx_perm, void* dx_shared, int32_t ab_kept, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_experts_grouped_train_fp8 - moe_experts_grouped (FP8 kind, at most one
 * shared expert) for a training step: the same outputs, and the gate/up
 * epilogue also keeps a = x W1^T and b = x W3^T (the promoted fp32 sums,
 * rounded to bf16) of every routed row and of the shared expert in the
 * backward workspace `bws`, so that moe_experts_backward_input_fp8 with
 * ab_kept = 1 does not recompute them (0.5 GB written at the DeepSeek-V3
 * shape instead of 4.3 TFLOP of FP8 GEMM).
 *   arguments as in moe_experts_grouped, plus
 *   bws, bws_bytes   at least moe_backward_workspace_bytes(cfg); pass the
 *                    same buffer to this step's backward calls
 * MOE_ERR_SHAPE for another kind or more than one shared expert.
 */
moe_status_t moe_experts_grouped_train_fp8(
    const moe_cfg_t* cfg, const void* x_perm, const float* x_perm_scales, const void* x,
    const float* x_scales, const int32_t* offsets, const void* w13, const float* w13_scales,
    const void* w2, const float* w2_scales, const void* ws13, const float* ws13_scales,
    const void* ws2, const float* ws2_scales, void* y_perm, void* y_shared, void* ws,
    size_t ws_bytes, void* bws, size_t bws_bytes, void* stream);

/*
 * moe_experts_backward_weights_fp8 - Wgrad of every expert FFN in FP8 E4M3
 * (mixed precision framework paragraph: Wgrad in FP8 with fp32
 * accumulation).  The contraction runs over the token rows of each segment,
 * so both operands are quantised in 128 x 1 tiles (128 consecutive rows of
 * one column, scale fl32(amax / 448); a segment's last tile holds the rows
 * it has):
 *   dW2 = q(dy)^T q(h),   dW13 = q([da | db])^T q(u)
 * with u the dequantised forward codes and h, [da | db] formed (fp32) from
 * the [a | b] and dh that moe_experts_backward_input_fp8 left in `ws`; every
 * 128-row partial is promoted to fp32 with both tiles' scales.
 *   x_perm, x_perm_scales, x_q, x_q_scales, offsets  as for the input call
 *   dy_perm [T*K, d], dout [T, d]  bf16, as for the input call
 *   dw13 [E, 2I, d], dw2 [E, d, I]  bf16 out (zeros for an expert with no rows)
 *   dws13 [1, 2I, d], dws2 [1, d, I] bf16 out (NULL if N_s = 0)
 *   ws, ws_bytes  the workspace of this step's input call (untouched in
 *                 between except by moe_route_backward)
 * Each operand is first written transposed, every segment padded to whole
 * 128-row tiles, so that each K block of the GEMM starts on an aligned
 * boundary; moe_backward_workspace_bytes covers those copies.
 */
moe_status_t moe_experts_backward_weights_fp8(
    const moe_cfg_t* cfg, const void* x_perm, const float* x_perm_scales, const void* x_q,
    const float* x_q_scales, const int32_t* offsets, const void* dy_perm, const void* dout,
    void* dw13, void* dw2, void* dws13, void* dws2, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_quantize_weights_fp8 - offline utility: quantise `n_mats` bf16
 * matrices [rows, cols] (contiguous, cols % 128 == 0) to E4M3 in 128 x 128
 * blocks (fine-grained quantisation paragraph): scale = fl32(amax / 448)
 * (1 for a zero block), code = E4M3(fl32(w / scale)), round to nearest
 * even, saturating.  q [n_mats, rows, cols] bytes; scales
 * [n_mats, ceil(rows/128), cols/128] fp32.
 */
moe_status_t moe_quantize_weights_fp8(const void* w_bf16, int32_t n_mats,
                                      int32_t rows, int32_t cols, void* q,
                                      float* scales, void* stream);

/*
 * moe_route_static_scratch - moe_route without a workspace argument.
 *
 * The paper has no counterpart: this entry point exists for callers that
 * cannot call cudaMalloc - for example a plugin running inside a serving
 * engine that has already reserved all device memory for its own pool and
 * exposes no allocator, or a latency-critical caller that must not pay the
 * device-wide synchronisation an allocation can cause.  Arguments, outputs
 * and results are those of moe_route; the caller still passes every input
 * and output buffer.
 *
 * Scratch: a 32 MiB array inside the library, reserved on every GPU that
 * loads the library until the process exits.  A call needs the routing part
 * of moe_workspace_bytes: align256(ceil(T/32) * E * 4) for the per-tile
 * loads; align256(T * E * 4) for the affinities when both affinity_in and
 * affinity_out are NULL; and, for the BF16 and FP8 kinds, align256(E * 3d * 2)
 * for the centroids split into bf16 terms plus, when T is small, at most
 * 9.7 MB of split-K partial sums.  (DeepSeek-V3 shape E=256, d=7168, T=8192,
 * no affinity buffer: 19.7 MiB.)  A larger need is rejected with
 * MOE_ERR_WORKSPACE before anything is launched.  The call allocates nothing.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture.  Every call shares the one array and it keeps the last
 * call's contents (no call needs it cleared): calls that overlap on the GPU
 * (on different streams, or from several host threads) race on it.
 */
moe_status_t moe_route_static_scratch(const moe_cfg_t* cfg, const void* x,
                                      const float* router_w, const float* bias,
                                      const float* affinity_in, float* affinity_out,
                                      int32_t* topk_idx, float* topk_w, int32_t* counts,
                                      int32_t* offsets, int32_t* row_of_slot,
                                      int32_t* token_of_row, void* stream);

/*
 * moe_selftest_wait - failure-detection self test.  One thread waits, with
 * the same bounded mbarrier wait the GEMM kernels use, on a barrier that
 * nothing arrives on; after limit_ns nanoseconds (1 .. 10^10) it gives up
 * and sets the timeout bit of the error word, so that the next
 * moe_get_device_error() returns MOE_ERR_TIMEOUT.  Nothing traps and the
 * device stays usable.  MOE_ERR_INVALID_ARG for a limit outside the range.
 */
moe_status_t moe_selftest_wait(int64_t limit_ns, void* stream);

/* Synchronises `stream`, returns the device error word (MOE_OK if clear,
 * MOE_ERR_TIMEOUT if a wait gave up, MOE_ERR_DEVICE for any other device
 * check) and clears it. */
moe_status_t moe_get_device_error(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
