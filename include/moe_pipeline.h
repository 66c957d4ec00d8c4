/*
 * moe_pipeline.h -- host-buffer executor of the MoE layer forward pass.
 *
 * The layer is the one of moe.h ("Mixture of Experts: Scaling Parameters
 * Without Scaling Compute", section "The MoE layer"); moe_forward computes
 * it from device buffers.  This executor takes token batches in HOST memory
 * and returns y and the auxiliary loss to HOST memory, overlapping the three
 * stages of consecutive batches: while batch s runs moe_forward on the
 * compute stream, the input copy of batch s+1 runs on one copy stream and
 * the output copy of batch s-1 on another.  The pages have no counterpart;
 * it is the serving loop around the layer (each batch is an independent
 * forward pass: results equal moe_forward's on the same batch, bit for bit).
 *
 * Ownership and memory
 *  - The executor is an opaque host object made by moe_pipeline_create and
 *    freed by moe_pipeline_destroy.  It holds two CUDA streams and a few
 *    events of its own; it allocates no device memory.
 *  - Device memory: the caller's workspace `ws` (256-byte aligned, at least
 *    moe_pipeline_workspace_size(cfg, depth) bytes, zero-filled before
 *    create, used by nothing else until destroy) holds moe_forward's
 *    workspace and `depth` staging slots (x, y and the loss of one batch
 *    each).  The weights (device pointers, layouts as in moe.h) are bound at
 *    create and read by every batch; the caller keeps them alive and may
 *    update them in place with work enqueued on `stream` between submits.
 *  - Host buffers: x_host [T][d] and y_host [T][d] of cfg->dtype, aux_host
 *    one float (or NULL).  They must stay valid, and x_host unchanged, until
 *    moe_pipeline_join has been called and `stream` has completed the work
 *    enqueued before the join.  For the copies to overlap with compute the
 *    host buffers must be page-locked (cudaHostAlloc, cudaHostRegister or a
 *    pinned torch tensor); pageable buffers give the same results with the
 *    copies serialised by the CUDA runtime.
 *
 * Ordering
 *  - Every call returns after enqueueing its work; none synchronises except
 *    moe_pipeline_destroy.  Batches run in submission order.
 *  - moe_forward of each batch runs on `stream` (the caller's stream given
 *    at create), so work the caller enqueues on `stream` between submits
 *    runs between the batches' forward passes.
 *  - The input copies wait for the point of `stream` at the last
 *    moe_pipeline_create or moe_pipeline_join call, and a slot is refilled
 *    only after the batch that last used it has been read out.
 *  - moe_pipeline_join makes `stream` wait until every batch submitted so
 *    far has its outputs in host memory.
 *
 * Errors: arguments are checked on the host before anything is enqueued
 * (status codes of moe.h; a rejected call changes nothing).  After a CUDA
 * runtime failure (MOE_ERR_CUDA) the executor's state is undefined: destroy
 * it.  Device-side errors of the forward passes are recorded in the forward
 * workspace at the start of `ws` and read with
 * moe_get_device_error(ws, stream, ...) after a join.
 */
#ifndef MOE_PIPELINE_H
#define MOE_PIPELINE_H

#include <stddef.h>
#include <stdint.h>

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_pipeline moe_pipeline;

/* Bytes of device workspace for `depth` (1 .. 4) batches in flight; 0 if
 * cfg or depth is invalid. */
size_t moe_pipeline_workspace_size(const moe_config* cfg, int32_t depth);

/*
 * Creates an executor for batches of cfg->T tokens (T >= 1) on the current
 * device.  W_r, logit_bias (may be NULL), W1, b1, W2, b2: device weights as
 * for moe_forward.  depth: staging slots, 2 for full overlap of the input
 * copy, the forward pass and the output copy of consecutive batches.
 * *out receives the executor (NULL on failure).
 */
moe_status moe_pipeline_create(const moe_config* cfg, int32_t depth, const float* W_r,
                               const float* logit_bias, const void* W1, const void* b1,
                               const void* W2, const void* b2, void* ws, size_t ws_bytes,
                               void* stream, moe_pipeline** out);

/* Enqueues one batch: copy x_host in, moe_forward, copy y (and the auxiliary
 * loss, when aux_host is not NULL) out. */
moe_status moe_pipeline_submit(moe_pipeline* p, const void* x_host, void* y_host,
                               float* aux_host);

/* Makes the executor's stream wait for the outputs of every submitted batch
 * (see Ordering). */
moe_status moe_pipeline_join(moe_pipeline* p);

/* Waits for the executor's copies to finish and frees its host objects
 * (streams, events).  The workspace stays the caller's.  NULL is a no-op. */
moe_status moe_pipeline_destroy(moe_pipeline* p);

#ifdef __cplusplus
}
#endif
#endif /* MOE_PIPELINE_H */
