/*
 * moe.h -- C ABI of the B300 (sm_103a) sparsely-gated Mixture-of-Experts FFN
 * layer forward pass.
 *
 * The operation is the MoE layer of "Mixture of Experts: Scaling Parameters
 * Without Scaling Compute", section "The MoE layer": router logits
 * g = W_r x, probabilities p = softmax(g), the top-k experts per token, and
 * the output y = sum over the selected experts i of w_i * f_i(x), where each
 * expert f_i is Linear(d, d_ff) + bias, exact GELU, Linear(d_ff, d) + bias and
 * w_i is the selected probability, renormalised over the k choices or not.
 * Section "The central problem: load balancing" of the same page adds the
 * expert capacity (overflow assignments are dropped) and the Switch-style
 * auxiliary loss E * sum_i f_i P_i.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every pointer argument is a DEVICE pointer owned by the caller, except
 *    `cfg` (host).  The library allocates no memory.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL means the
 *    legacy default stream) and returns after enqueueing its kernels; none
 *    synchronises, except moe_get_device_error.
 *  - Layouts are row-major.  Weights use the nn.Linear (out, in) layout:
 *      W_r [E][d] fp32, W1 [E][d_ff][d], b1 [E][d_ff], W2 [E][d][d_ff],
 *      b2 [E][d].
 *    x, W1, b1, W2, b2 and y have the element type cfg->dtype (fp32 or bf16).
 *  - Alignment: x, W1, W2, x_perm, y_perm and y must be 16-byte aligned; d
 *    and d_ff must be multiples of 8.
 *  - Routing: experts are ranked by their fp32 router logit, larger first;
 *    equal logits rank the lower expert index first (softmax is monotone, so
 *    this is the top-k of p).
 *  - Capacity: when cfg->capacity >= 0 each expert keeps at most that many
 *    assignments, the first ones in (token, slot) order; the others are
 *    dropped and contribute zero to y.  cfg->capacity < 0 means no cap.
 *  - Dispatch order: the kept assignments of expert e occupy rows
 *    offsets[e] .. offsets[e+1]-1 of the permuted buffers, in ascending token
 *    order (the per-expert row lists of the page's dispatch loop).
 *  - Errors: arguments are validated on the host before any launch; an
 *    invalid call returns a status and enqueues nothing.  A problem found on
 *    the device (an expert index outside [0, E) handed to moe_dispatch, a
 *    pipeline wait that gave up) is recorded in the workspace and reported by
 *    moe_get_device_error; the offending element is skipped, never written
 *    out of bounds.
 *  - Workspace: `ws` is scratch device memory of at least
 *    moe_workspace_size(cfg) bytes, 256-byte aligned.  Calls that run
 *    concurrently must not share a workspace.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad size or shape */
    MOE_ERR_ALIGNMENT = 2,    /* a pointer or a row length breaks the alignment rule */
    MOE_ERR_WORKSPACE = 3,    /* ws_bytes < moe_workspace_size(cfg) or ws misaligned */
    MOE_ERR_UNSUPPORTED = 4,  /* shape outside what the kernels implement (E > 256 ...) */
    MOE_ERR_CUDA = 5,         /* a CUDA runtime call failed (launch, memset ...) */
    MOE_ERR_DEVICE = 6        /* the device recorded an error (see moe_get_device_error) */
} moe_status;

typedef enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Shape and options of one layer call. */
typedef struct moe_config {
    int32_t T;           /* tokens in the batch (>= 0) */
    int32_t d;           /* model width (multiple of 8) */
    int32_t d_ff;        /* expert hidden width (multiple of 8) */
    int32_t E;           /* experts, 1 .. 256 */
    int32_t k;           /* experts per token, 1 .. min(E, 8) */
    int32_t dtype;       /* moe_dtype of x, W1, b1, W2, b2, y */
    int32_t capacity;    /* < 0: no cap; >= 0: kept assignments per expert at most */
    int32_t renormalize; /* 1: w = p_sel / sum(p_sel); 0: w = p_sel */
    int32_t n_shared;    /* shared experts, 0 .. E-1 (see below); 0 for a plain layer */
    int32_t routing;     /* moe_routing: MOE_TOKEN_CHOICE (0) or MOE_EXPERT_CHOICE (1) */
    int32_t overflow;    /* moe_overflow: MOE_DROP (0) or MOE_REROUTE (1); see below */
} moe_config;

typedef enum moe_routing { MOE_TOKEN_CHOICE = 0, MOE_EXPERT_CHOICE = 1 } moe_routing;
typedef enum moe_overflow { MOE_DROP = 0, MOE_REROUTE = 1 } moe_overflow;

/*
 * Rerouting on overflow ("The central problem: load balancing" and the
 * inferensys glossary's expert capacity: an overflowing token may go to its
 * next-ranked expert instead of being dropped), cfg->overflow = MOE_REROUTE, token choice only, n_shared = 0: after the
 * capacity drop (as above), the r-th dropped slot of a token (r = 0, 1, ...)
 * is offered once to the token's (k + r)-th ranked expert, the best one it
 * does not use; offers are taken in (token, slot) order and an expert
 * accepts them while its kept assignments plus accepted offers stay below
 * the capacity; a refused offer is dropped.  An accepted slot's weight is
 * the new expert's probability with the normalisation of the token's other
 * weights (divided by the sum over its k choices when renormalising).
 * Expert e's rows are its kept slots in token order, then the offers it
 * accepted in token order.  The router then ranks K2 = min(2k, E) experts
 * per token: moe_route writes topk_idx / topk_w with K2 columns (the k
 * choices, then the next K2 - k, weights normalised as the choices'), and
 * moe_dispatch reads them so; expert_counts and the auxiliary loss count the
 * k choices only.  slot_of, perm_* and the other per-assignment arrays keep
 * their k columns (slot_of[t][j]: the row slot j ended in).  K2 <= 8.
 */

/*
 * Shared experts ("Design variations": experts that every token uses):
 * with n_shared > 0, experts 0 .. n_shared-1 of the E in W1, b1, W2, b2 are
 * applied to every token with weight 1 and are never capped; the router
 * covers the other E - n_shared experts (W_r, logit_bias, logit_noise,
 * logits_in and logits_out have E - n_shared rows / columns; softmax, top-k,
 * the auxiliary loss and the z-loss are over them) and picks k of them.
 * Every per-assignment array below then has K = k + n_shared columns per
 * token ([T][K]: topk_idx, topk_w, slot_of; T*K: perm_token, perm_w, x_perm,
 * y_perm): the k routed choices (expert ids n_shared .. E-1, best first),
 * then the shared experts 0 .. n_shared-1.  k + n_shared <= 8.  With
 * n_shared = 0, K = k and everything below reads as written.
 */

/*
 * Expert-choice routing ("Design variations": the experts select the tokens,
 * which balances the load by construction), cfg->routing = MOE_EXPERT_CHOICE:
 * the
 * router computes p = softmax(g) as for token choice, then every expert e
 * takes the C tokens with the largest p[t][e] - larger first, the lower
 * token index first among equal p - where
 *   C = min(T, cfg->capacity)          if cfg->capacity >= 0,
 *   C = min(T, ceil(T * cfg->k / E))   otherwise (k: experts per token on
 *                                      average, as top-k token choice);
 * see moe_expert_choice_capacity.  Expert e's rows are e*C .. e*C + C - 1,
 * its chosen tokens in ascending token order; a token's output is the sum,
 * over the experts that chose it (any number, 0 .. E), of p[t][e] times the
 * expert's output, unnormalised; a token no expert chose gets 0.  There is
 * no balancing loss: aux_out receives 0; expert_counts receives C for every
 * expert; the z-loss and logits_out are as for token choice.  The
 * per-assignment arrays have the expert-choice shapes:
 *   offsets [E+1] (= e*C), perm_token / perm_w / x_perm / y_perm [E*C],
 *   slot_of [T][E] (row of (t, e), -1 if e did not choose t).
 * Calls: moe_route_expert_choice (route + dispatch), then moe_expert_ffn and
 * moe_combine with the same cfg, or moe_forward.  moe_route, moe_dispatch
 * and moe_dispatch_noalloc are token-choice steps and return
 * MOE_ERR_UNSUPPORTED for it; so does n_shared > 0.
 */

/* Bytes of workspace any call below needs for this configuration. */
size_t moe_workspace_size(const moe_config* cfg);

/* Static text for a status code. */
const char* moe_status_string(moe_status s);

/*
 * Router: logits, softmax, top-k and gate weights, per-expert counts, the
 * auxiliary loss and the router z-loss ("The MoE layer", steps 1-2; "The
 * central problem: load balancing", auxiliary loss and router z-loss).
 *   x           [T][d] dtype          token batch
 *   W_r         [E][d] fp32           router weight
 *   logit_bias  [E] fp32 or NULL      added to every token's logits
 *   logit_noise [T][E] fp32 or NULL   noisy gating: added to the logits
 *                                     before the softmax and the top-k (the
 *                                     caller draws it; "The central problem:
 *                                     load balancing", noisy gating)
 *   logits_in   [T][E] fp32 or NULL   if given, used as the logits (x, W_r,
 *                                     logit_bias and logit_noise are then
 *                                     not read)
 *   logits_out  [T][E] fp32 or NULL   receives the logits used for routing
 *   topk_idx    [T][k] int32          selected experts, best first ([T][K2]
 *                                     with MOE_REROUTE, see above)
 *   topk_w      [T][k] fp32           gate weights of the selected experts
 *   expert_counts [E] int32 or NULL   assignments per expert, all k slots,
 *                                     before any capacity drop
 *   aux_out     [1] fp32 or NULL      E * sum_i f_i P_i, f_i from the first
 *                                     slot; 0 when T == 0
 *   z_loss_out  [1] fp32 or NULL      router z-loss: the mean over tokens of
 *                                     (log sum_e exp g[t][e])^2 over the
 *                                     logits used for routing; 0 when T == 0
 */
moe_status moe_route(const moe_config* cfg, const void* x, const float* W_r,
                     const float* logit_bias, const float* logit_noise,
                     const float* logits_in, float* logits_out,
                     int32_t* topk_idx, float* topk_w, int32_t* expert_counts, float* aux_out,
                     float* z_loss_out, void* ws, size_t ws_bytes, void* stream);

/*
 * Dispatch: expert offsets, the capacity drop and the gather of token rows
 * into expert-contiguous order ("The MoE layer", dispatch of each expert's
 * tokens; "The central problem: load balancing", capacity).
 *   x           [T][d] dtype
 *   topk_idx    [T][k] int32          from moe_route (values outside [0, E)
 *                                     are skipped and flagged; [T][K2] with
 *                                     MOE_REROUTE, and so topk_w)
 *   topk_w      [T][k] fp32 or NULL   gate weights; if given, copied to perm_w
 *   offsets     [E+1] int32           segment starts; offsets[E] = kept total
 *   slot_of     [T][k] int32          row of each assignment, -1 if dropped
 *   perm_token  [T*k] int32           token of each kept row (first
 *                                     offsets[E] entries are written)
 *   perm_w      [T*k] fp32 or NULL    gate weight of each kept row
 *   x_perm      [T*k][d] dtype        gathered rows (first offsets[E] rows)
 */
moe_status moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                        const float* topk_w, int32_t* offsets, int32_t* slot_of,
                        int32_t* perm_token, float* perm_w, void* x_perm,
                        void* ws, size_t ws_bytes, void* stream);

/*
 * Expert-choice route and dispatch (cfg->routing = MOE_EXPERT_CHOICE; see
 * above): router logits and p as in moe_route, each expert's top-C tokens,
 * the row layout and, when x_perm is not NULL, the gather of the rows.
 *   x, W_r, logit_bias, logit_noise, logits_in, logits_out   as moe_route
 *   offsets     [E+1] int32           e*C
 *   perm_token  [E*C] int32           chosen tokens, ascending per expert
 *   perm_w      [E*C] fp32            p[token][e] of each row
 *   slot_of     [T][E] int32          row of (t, e), -1 if e did not choose t
 *   x_perm      [E*C][d] dtype or NULL   x rows of perm_token
 *   expert_counts [E] int32 or NULL   C for every expert
 *   z_loss_out  [1] fp32 or NULL      router z-loss as in moe_route
 */
moe_status moe_route_expert_choice(const moe_config* cfg, const void* x, const float* W_r,
                                   const float* logit_bias, const float* logit_noise,
                                   const float* logits_in, float* logits_out, int32_t* offsets,
                                   int32_t* perm_token, float* perm_w, int32_t* slot_of,
                                   void* x_perm, int32_t* expert_counts, float* z_loss_out,
                                   void* ws, size_t ws_bytes, void* stream);

/* C, the tokens each expert takes under expert-choice routing (formula
 * above); -1 for an invalid cfg. */
int32_t moe_expert_choice_capacity(const moe_config* cfg);

/*
 * Experts: for every expert segment, y_perm = w * (GELU(x_perm W1^T + b1)
 * W2^T + b2) ("The MoE layer", expert = Linear, GELU, Linear).
 *   x_perm      [T*k][d] dtype        rows grouped by expert (moe_dispatch)
 *   offsets     [E+1] int32           segment starts (device; not read on the host)
 *   W1, b1, W2, b2                    expert bank, dtype
 *   perm_w      [T*k] fp32 or NULL    per-row weight; NULL means 1
 *   y_perm      [T*k][d] fp32         expert outputs (first offsets[E] rows)
 * The hidden activations live in the workspace (bf16 for bf16 layers).
 * Expert choice: E*C rows instead of T*k.
 */
moe_status moe_expert_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                          const void* W1, const void* b1, const void* W2, const void* b2,
                          const float* perm_w, float* y_perm,
                          void* ws, size_t ws_bytes, void* stream);

/*
 * Combine: y[t] = sum over j = 0..k-1 with slot_of[t][j] >= 0 of
 * y_perm[slot_of[t][j]], summed in slot order in fp32, stored as dtype; a
 * token with every assignment dropped gets 0 ("The MoE layer", weighted
 * combination; the weights were applied by moe_expert_ffn).
 *   y_perm [T*k][d] fp32, slot_of [T][k] int32, y [T][d] dtype.
 * Expert choice: k reads E (slot_of [T][E], slots in expert order) and
 * y_perm has E*C rows.
 */
moe_status moe_combine(const moe_config* cfg, const float* y_perm, const int32_t* slot_of,
                       void* y, void* stream);

/*
 * The whole layer: route, dispatch, experts, combine.  Intermediates live in
 * the workspace.  logit_noise, aux_out, expert_counts, logits_out and
 * z_loss_out (as in moe_route) may be NULL.
 */
moe_status moe_forward(const moe_config* cfg, const void* x, const float* W_r,
                       const float* logit_bias, const float* logit_noise,
                       const void* W1, const void* b1,
                       const void* W2, const void* b2, void* y, float* aux_out,
                       int32_t* expert_counts, float* logits_out, float* z_loss_out,
                       void* ws, size_t ws_bytes, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device error record of
 * workspace `ws`.  Returns MOE_OK, or MOE_ERR_DEVICE with *code (if not
 * NULL) set to the first recorded error code (1: expert index out of range;
 * 2: pipeline wait timed out) and *info to a detail value.
 */
moe_status moe_get_device_error(void* ws, void* stream, int32_t* code, int32_t* info);

/*
 * moe_dispatch without a workspace, for callers that cannot provide one: a
 * host whose GPU memory is handed out once, up front, by another component
 * (a serving engine's fixed pool, a plugin host that owns every allocation)
 * has no allocator to call for scratch space.  The pages have no counterpart
 * of this call; it is a deployment convenience of this library.
 *   Arguments and results are those of moe_dispatch, minus ws / ws_bytes.
 *   Scratch lives in a fixed array inside the library (768.25 KB, held on
 *   every GPU that loads the library until the process exits), so the call
 *   allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   Limits: T * k <= 65536 and E <= 256; larger problems return
 *   MOE_ERR_UNSUPPORTED without enqueueing anything.
 *   The first call in a CUDA context, made while that context is current,
 *   looks up the array's device address (cudaGetSymbolAddress); make that
 *   first call before any stream capture.  Any context works: the primary
 *   context the runtime uses, contexts the host creates with the driver
 *   API, several contexts on one device, and the new primary context after
 *   a device reset each get their own lookup (keyed on the context's unique
 *   ID, the last 16 contexts remembered).
 *   All calls on a device share the one array: calls whose work overlaps on
 *   the GPU (different streams without ordering) race and give wrong results.
 *   Each call clears the part that must start at zero.  An expert index
 *   outside [0, E) is skipped (slot -1) as in moe_dispatch, but the record of
 *   it cannot be read back (there is no workspace to pass to
 *   moe_get_device_error).
 */
moe_status moe_dispatch_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                                const float* topk_w, int32_t* offsets, int32_t* slot_of,
                                int32_t* perm_token, float* perm_w, void* x_perm, void* stream);

/*
 * Auxiliary-loss-free balancing ("The central problem: load balancing":
 * per-expert bias terms that follow the observed load): after a batch,
 * moves each expert's router logit bias by `step` toward balanced load -
 *   logit_bias[e] -= step  if expert_counts[e] > mean count,
 *   logit_bias[e] += step  if expert_counts[e] < mean count,
 * unchanged at the mean (mean = sum of the E counts / E, compared exactly in
 * integers).  expert_counts [E] int32 as written by moe_route/moe_forward;
 * logit_bias [E] fp32, updated in place, for the next call's logit_bias.
 * cfg supplies E.  No workspace.
 */
moe_status moe_update_balance_bias(const moe_config* cfg, const int32_t* expert_counts,
                                   float* logit_bias, float step, void* stream);

/*
 * Diagnostics: number of CUDA kernels libmoe has enqueued in this process
 * since it was loaded (memsets excluded).  No counterpart on the pages.
 */
uint64_t moe_launch_count(void);

/*
 * Diagnostics: runs the bounded pipeline wait of the tensor-core GEMMs (the
 * mbarrier wait their producer, MMA and epilogue warps use) on a barrier that
 * nothing completes, with a limit of timeout_ns (clamped to 1 s), in one
 * single-thread kernel on `stream`.  The wait gives up and records the
 * time-out in the error record of workspace `ws` exactly as a stalled
 * pipeline would, so moe_get_device_error then reports MOE_ERR_DEVICE with
 * code 2 (info 900) and the context stays usable.  `ws`: at least 256 bytes
 * of device memory (only the error record is touched).  No counterpart on
 * the pages.
 */
moe_status moe_check_wait_timeout(void* ws, uint64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
