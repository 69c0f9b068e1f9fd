/*
 * moe_pipeline.h -- the layer forward over a stream of batches that live in HOST memory.
 *
 * A serving loop hands the layer one batch of activations after another from host memory and
 * wants each batch's output back in host memory. Run one after another, every batch pays its
 * host->device copy, the layer, and its device->host copy in sequence. A pipeline object runs the
 * three on three CUDA streams instead: the copy-in of batch i+1 and the copy-out of batch i-1
 * overlap the layer computation of batch i (PCIe/C2C copies in both directions run alongside the
 * kernels). Every batch's layer computation is exactly moe_forward (include/moe.h) on a device
 * copy of its h, so the outputs are bit-identical to moe_forward's.
 *
 * This is the one part of libmoe that allocates device memory and keeps state: at create time
 * it allocates a workspace and two device slots for h, y and aux (2 (T d s + T d s) + ws bytes,
 * s = dtype size); it creates two streams and a few events. Nothing is allocated per batch.
 *
 * Ordering. The layer runs on the caller's `stream` given at create time. Work the caller
 * enqueued on that stream before the first submit (after create or after a join) completes
 * before that submit's copy-in starts. moe_pipeline_join(p, s) makes stream s wait until every
 * batch submitted so far has been copied out. Host buffers passed to submit must stay valid and
 * unchanged (h) / unread (y, aux) until a join has been reached; page-locked (pinned) host memory
 * is needed for the copies to overlap the computation (pageable memory works, synchronously).
 *
 * Errors follow include/moe.h: host-side checks return a status before anything is enqueued;
 * device-side failures are read with moe_pipeline_device_status. The calling thread's current
 * CUDA device must be the one the pipeline was created on. A pipeline is not thread-safe.
 */
#ifndef MOE_PIPELINE_H_
#define MOE_PIPELINE_H_

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_pipeline moe_pipeline_t;

/* Create a pipeline for layers of shape `cfg` with the given DEVICE weights (same meaning,
 * layout and alignment as moe_forward's; caller-owned, they must outlive the pipeline).
 * `stream` (cudaStream_t as void*, it must outlive the pipeline) is where the layer computation
 * runs. On success *out holds the new pipeline. MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for a bad cfg or weight pointer
 * (checked before any CUDA call), MOE_ERR_CUDA when an allocation or stream creation fails
 * (nothing is leaked). */
moe_status_t moe_pipeline_create(const moe_config_t *cfg, const float *W_r, const float *b_r,
                                 const float *sel_bias, const void *W1, const float *b1,
                                 const void *W3, const void *W2, const float *b2, void *stream,
                                 moe_pipeline_t **out);

/* Enqueue one batch and return without waiting:
 *   h_host   [T, d] dtype, host memory (read by the copy-in)
 *   y_host   [T, d] dtype, host memory (written by the copy-out)
 *   aux_host one float, host memory (written by the copy-out), the batch's auxiliary value.
 * MOE_ERR_INVALID_ARG for a NULL pipeline or buffer. */
moe_status_t moe_pipeline_submit(moe_pipeline_t *p, const void *h_host, void *y_host,
                                 float *aux_host);

/* Make `stream` wait for every batch submitted so far, copy-out included (no host wait). */
moe_status_t moe_pipeline_join(moe_pipeline_t *p, void *stream);

/* Wait for everything submitted, then read and clear the device status word of the pipeline's
 * workspace (as moe_device_status). */
moe_status_t moe_pipeline_device_status(moe_pipeline_t *p);

/* Wait for everything submitted and free the pipeline. NULL is a no-op. */
moe_status_t moe_pipeline_destroy(moe_pipeline_t *p);

#ifdef __cplusplus
}
#endif
#endif /* MOE_PIPELINE_H_ */
