/*
 * moe_backward.h -- backward pass of the MoE layer of moe.h.
 *
 * The pages train the layer end to end ("Mixture of Experts: Scaling
 * Parameters Without Scaling Compute", section "The MoE layer"; the
 * load-balancing loss of section "The central problem: load balancing"):
 * this call gives the gradients of
 *     L = <dy, y> + aux_grad * aux + z_grad * z_loss
 * for the forward pass moe_forward computes on the same inputs, where dy is
 * the caller's upstream gradient of the layer output and aux_grad, z_grad
 * the weights of the two router losses.  The routing decisions (top-k and
 * the capacity drop) are held fixed, as automatic differentiation treats
 * them; the gate weights carry gradient to the router logits through the
 * softmax (and the renormalisation over the k choices), the auxiliary loss
 * through the mean probabilities P (the counts f are constants) and the
 * z-loss through the log-sum-exp.  Per kept assignment (token t, expert e,
 * weight w; u = W1_e x + b1_e, h = GELU(u), o = W2_e h + b2_e):
 *     dW2_e += (w dy_t) h^T, db2_e += w dy_t,
 *     du = (W2_e^T (w dy_t)) * GELU'(u), dW1_e += du x_t^T, db1_e += du,
 *     dx_t += W1_e^T du,
 * and with s = <dy_t, w o> per routed slot the logit gradient dg (renormalised:
 * s_e - w_e sum_j s_j on the choices; raw probabilities: s_e [e chosen] -
 * p_e sum_j s_j) plus the two loss terms gives dW_r = dg^T x and
 * dx += dg W_r.  The layer variants of moe.h follow the same rule:
 *   shared experts   the n_shared always-on slots (weight 1) feed the expert
 *                    gradients and dx but no logit; the router covers the
 *                    E - n_shared routed experts;
 *   rerouting        a slot moved to another expert has that expert's
 *                    probability as its weight (over the same normaliser as
 *                    the token's k choices), so its s goes to the new
 *                    expert's logit;
 *   expert choice    each selected (expert, token) pair has weight p_e(t);
 *                    dg_e = s_e - p_e sum_j s_j over the token's pairs, and
 *                    there is no balancing loss (aux_grad is ignored).
 *
 * The call recomputes the forward intermediates it needs (routing, dispatch,
 * the expert pre-activations, the expert outputs) from x and the weights:
 * it does not read a previous moe_forward's workspace.
 *
 * Supported: every configuration moe_forward accepts.  bf16 layers keep the
 * pre-activations, activations and scaled upstream rows in bf16 and run the
 * products on the tcgen05 tensor cores (the router terms dg W_r and dg^T x,
 * with 16-64 routed experts, as tf32 mma.sync); fp32 layers keep them in fp32 and
 * run every product with fp32 FMA on the CUDA cores (GELU' from erff).
 *
 * Arguments (device pointers, caller-owned, layouts as in moe.h):
 *   x [T][d] (layer dtype); W_r [E - n_shared][d] fp32;
 *   logit_bias [E - n_shared] fp32 or NULL;
 *   W1 [E][d_ff][d], b1 [E][d_ff], W2 [E][d][d_ff], b2 [E][d] (layer dtype);
 *   dy [T][d] (layer dtype)              upstream gradient of y
 *   aux_grad, z_grad                     weights of the two losses in L
 *   dx [T][d] (layer dtype)              written (not accumulated)
 *   dW_r [E - n_shared][d], dW1 [E][d_ff][d], db1 [E][d_ff], dW2 [E][d][d_ff],
 *   db2 [E][d]                           fp32, written (not accumulated)
 *   ws, ws_bytes                         at least
 *                                        moe_backward_workspace_size(cfg)
 *                                        bytes, 256-byte aligned, whose first
 *                                        256 bytes hold the device error
 *                                        record (moe_get_device_error)
 * Alignment: x, dy, dx, W1, W2 16-byte aligned; d and d_ff multiples of 8.
 * Asynchronous on `stream`; invalid arguments return a status before
 * anything is enqueued.  T = 0 writes zero gradients.
 */
#ifndef MOE_BACKWARD_H
#define MOE_BACKWARD_H

#include <stddef.h>
#include <stdint.h>

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of workspace moe_backward needs for this configuration (0 if the
 * configuration is invalid or unsupported). */
size_t moe_backward_workspace_size(const moe_config* cfg);

moe_status moe_backward(const moe_config* cfg, const void* x, const float* W_r,
                        const float* logit_bias, const void* W1, const void* b1, const void* W2,
                        const void* b2, const void* dy, float aux_grad, float z_grad, void* dx,
                        float* dW_r, float* dW1, float* db1, float* dW2, float* db2, void* ws,
                        size_t ws_bytes, void* stream);

/*
 * Diagnostics: the weight-gradient products of moe_backward read each expert
 * segment through its own TMA tensor map, made on the device by editing a
 * copy of a whole-buffer map (base address and row extent, PTX
 * tensormap.replace).  This call makes such maps for three test segments (a
 * ragged, an empty and a long one) in both views the products use (3-D and
 * 2-D boxes), copies them back and compares them byte for byte with the
 * driver's own encoding of the same segments (cuTensorMapEncodeTiled).  No
 * tensor copy runs.  ws: at least 3 MiB of device memory, 256-byte aligned
 * (MOE_ERR_WORKSPACE otherwise); its first 2 KB are overwritten.  Returns
 * MOE_OK when every map matches, MOE_ERR_UNSUPPORTED on a mismatch,
 * MOE_ERR_CUDA when a CUDA call fails.  Synchronises `stream`.  No
 * counterpart on the pages.
 */
moe_status moe_check_segment_maps(void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_BACKWARD_H */
