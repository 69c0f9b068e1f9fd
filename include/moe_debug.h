/*
 * moe_debug.h -- test hooks of libmoe: failure detection without a GPU fault.
 *
 * Every spin-wait in libmoe's kernels (the dispatch look-back and done flag, every mbarrier wait
 * of the tensor-core GEMM) is bounded by the device clock; when the bound runs out, the kernel
 * records MOE_ERR_TIMEOUT in the workspace status word, stops issuing work, waits (bounded) for
 * its own copies and MMAs, frees its tensor memory and returns. These hooks run one step with a
 * short bound and one signal withheld -- a flag that nothing sets -- so that the bounded wait runs
 * out on purpose. Nothing faults, traps or hangs; the CUDA context stays usable and
 * moe_device_status() then returns MOE_ERR_TIMEOUT (and clears it). Outputs of a hooked call are
 * meaningless. The pages describe no such mechanism; it exists for the library's own tests.
 *
 * spin_limit_ns must lie in [1e6, 2e9] (1 ms .. 2 s); arguments are otherwise those of the
 * ordinary call of the same step (include/moe.h).
 */
#ifndef MOE_DEBUG_H_
#define MOE_DEBUG_H_

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* moe_build_dispatch (without the gather) in which chunk 0 never publishes its look-back word,
 * so every later chunk's look-back runs out. Needs at least two chunks: T * k > 1024, else
 * MOE_ERR_INVALID_ARG. */
moe_status_t moe_debug_dispatch_timeout(const moe_config_t *cfg, const int32_t *topk_idx,
                                        int32_t *counts, int32_t *offsets,
                                        int32_t *sorted_token, int32_t *slot_of, void *ws,
                                        size_t ws_bytes, uint64_t spin_limit_ns, void *stream);

/* moe_expert_ffn (bf16, tensor cores) in which the TMA producer issues no loads, so the MMA
 * warp's wait for the first stage runs out and the whole CTA aborts. MOE_ERR_UNSUPPORTED for
 * f32 configurations. */
moe_status_t moe_debug_expert_ffn_timeout(const moe_config_t *cfg, const void *x_perm,
                                          const int32_t *offsets, const void *W1, const float *b1,
                                          const void *W3, const void *W2, const float *b2,
                                          void *y_perm, void *ws, size_t ws_bytes,
                                          uint64_t spin_limit_ns, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_DEBUG_H_ */
