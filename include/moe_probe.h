/*
 * moe_probe.h -- a measurement probe of libmoe: the GPU's FP32 fused multiply-add rate.
 *
 * The f32 layer's expert MLPs run as FFMA chains on the CUDA cores, so their roofline is the FP32
 * FFMA rate, which the tensor-core and copy peaks do not give. This probe measures it: a kernel
 * of independent FFMA chains with no memory traffic but one conditional store. The caller times
 * the launch on `stream` (for instance with CUDA events) and divides the returned flop count by
 * that time. The pages have no counterpart of this call; it only serves the library's benchmark.
 */
#ifndef MOE_PROBE_H_
#define MOE_PROBE_H_

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Launch `blocks` x `threads` threads on `stream`, each running 8 independent chains of
 * 16 * iters dependent fmaf steps. out: one float of device memory, written only in the
 * (never taken) case that the chains end on a value the caller cannot predict, so the work is
 * not optimised away. *flops (host) receives the launch's flop count,
 * 2 * 8 * 16 * iters * blocks * threads. Limits: 1 <= blocks <= 65535, threads a multiple of 32
 * in [32, 1024], 1 <= iters <= 2^20; else MOE_ERR_INVALID_ARG. A failed launch returns
 * MOE_ERR_CUDA. */
moe_status_t moe_fp32_ffma_probe(int32_t blocks, int32_t threads, int32_t iters, float *out,
                                 void *stream, double *flops);

#ifdef __cplusplus
}
#endif
#endif /* MOE_PROBE_H_ */
