/* moe_backward.h -- the backward pass of the top-k routed MoE FFN layer (libmoe, C ABI).
 *
 * Definition (the pages on mixture of experts): selecting the top-k experts is not
 * differentiable, so the gradient reaches the router only through the weights of the chosen
 * experts, and for Switch top-1 through the router probability p_i (llm.curionode.com "Mixture of
 * Experts.", opening text; lensaml.com "Mixture of Experts", Step 3 "Top-k Routing"); of the
 * auxiliary term E sum_i f_i P_i only P_i is differentiable (lensaml.com Step 4 "Load
 * Balancing"); the router is trained jointly by ordinary backpropagation (arjunjaggi.com "Mixture
 * of Experts in LLMs", "How Routing Works"). So the expert choice idx, the routed counts (f_i)
 * and the capacity drops of the forward are held fixed, and moe_backward returns the exact
 * chain-rule gradients of
 *
 *     L = sum_{t,o} dy[t,o] y[t,o] + aux_weight * (E sum_e f_e P_e) + zloss_weight * zloss
 *
 * with respect to h, W_r, b_r, W1, W3, W2, b1 and b2, where y, the auxiliary value and the
 * z-loss are those of moe_forward (include/moe.h). The selection-only routing bias changes only
 * idx, which is taken from the forward.
 *
 * Precision: bf16 layers run their matrix products on the tensor cores with f32 accumulation;
 * the pre-activations, dHu = dy W2 and the intermediate gradients are stored as bf16; the
 * activation derivative, the gate and router gradients and the bias sums are f32; the router's
 * two contractions use hi + lo bf16 pieces of dz and W_r (f32 quality). f32 layers run every
 * product on the CUDA cores in f32 and always recompute the pre-activations.
 */
#ifndef MOE_BACKWARD_H
#define MOE_BACKWARD_H

#include <stddef.h>
#include <stdint.h>

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of backward workspace `bws` for cfg: the pre-activations, the per-slot intermediate
 * gradients (padded row layout) and the router's partial sums. MOE_ERR_INVALID_ARG for an
 * invalid cfg. */
moe_status_t moe_backward_workspace_size(const moe_config_t *cfg, size_t *bytes);

/* Number of kernels one moe_backward call with cfg and saved_preact launches (0 for T = 0;
 * device memsets not counted). Host-only. */
moe_status_t moe_backward_launch_count(const moe_config_t *cfg, int32_t saved_preact,
                                       int32_t *kernels);

/* moe_forward (include/moe.h; same arguments, results and errors) for a training step: the first
 * expert GEMM also stores its pre-activations -- x . W1_e (+ b1_e), and x . W3_e for SwiGLU,
 * [T k, f] bf16 each, the values its epilogue activates -- into the backward workspace bws
 * (moe_backward_workspace_size bytes, 16-byte aligned), so that moe_backward with
 * saved_preact = 1 need not recompute them. bf16 only (MOE_ERR_UNSUPPORTED for f32);
 * MOE_ERR_WORKSPACE if bws is too small or misaligned, MOE_ERR_INVALID_ARG if it is NULL. */
moe_status_t moe_forward_train(const moe_config_t *cfg, const void *h, const float *W_r,
                               const float *b_r, const float *sel_bias, const void *W1,
                               const float *b1, const void *W3, const void *W2, const float *b2,
                               void *y, float *aux_out, float *zloss_out, int32_t *topk_idx_out,
                               int32_t *counts_out, void *ws, size_t ws_bytes, void *bws,
                               size_t bws_bytes, void *stream);

/* Gradients of the layer for the upstream gradient dy, after a moe_forward call with the same
 * cfg, inputs and workspace `ws` (the backward reads the routing the forward left there:
 * gates, offsets, sorted_token, slot_of, the permuted rows unless cfg->fuse_gather, and, for a
 * bf16 layer whose router ran on the tensor cores, the router logits in the router's scratch;
 * ws must not be used for another forward in between).
 *   h, W_r, b_r, W1, b1, W3, W2, b2   the forward's inputs, same layouts (include/moe.h)
 *   topk_idx [T, k] int32 or NULL     the forward's topk_idx_out if it was given one, else NULL
 *                                     (the copy in ws)
 *   counts   [E] int32 or NULL        likewise for counts_out
 *   dy       [T, d] (layer's type)    upstream gradient of y
 *   aux_weight, zloss_weight          the weights of the auxiliary value and of the z-loss in L
 *   saved_preact                      1: the forward was moe_forward_train with this bws, whose
 *                                     pre-activations are used (bf16 layers); 0: they are
 *                                     recomputed (two grouped GEMMs for SwiGLU, one for GELU)
 * Outputs (device, caller-owned, fully overwritten):
 *   dW_r [d, E] f32;  db_r [E] f32 (given exactly when b_r is given)
 *   dW1  [E, f, d];  dW3 [E, f, d] (SwiGLU only, else ignored);  dW2 [E, d, f] -- in the
 *        layer's type (bf16 or f32); dh [T, d] likewise
 *   db1  [E, f] f32, db2 [E, d] f32 (when cfg->has_bias, else ignored)
 * An expert that received no slot gets zero weight gradients. Alignment: h, dy, dh and the
 * weight tensors 16 bytes, the f32 tensors 4 bytes, ws and bws 16 bytes.
 * Errors: MOE_ERR_INVALID_ARG (pointers, alignment, a non-finite aux_weight or zloss_weight, b_r
 * given without db_r or the reverse, saved_preact not 0 or 1), MOE_ERR_UNSUPPORTED
 * (saved_preact = 1 for an f32 layer, or an f32 layer past 4M padded rows), MOE_ERR_WORKSPACE
 * (ws or bws too small), MOE_ERR_CUDA (a launch failed); out-of-range indices in the forward's
 * routing set MOE_ERR_DEVICE_INDEX in the device status word (moe_device_status). Asynchronous
 * on `stream`; allocates nothing. */
moe_status_t moe_backward(const moe_config_t *cfg, const void *h, const float *W_r,
                          const float *b_r, const void *W1, const float *b1, const void *W3,
                          const void *W2, const float *b2, const int32_t *topk_idx,
                          const int32_t *counts, const void *dy, float aux_weight,
                          float zloss_weight, void *dh, float *dW_r, float *db_r, void *dW1,
                          float *db1, void *dW3, void *dW2, float *db2, void *ws, size_t ws_bytes,
                          void *bws, size_t bws_bytes, int32_t saved_preact, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_BACKWARD_H */
