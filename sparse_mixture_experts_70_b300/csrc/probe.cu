// probe.cu -- FP32 FFMA rate probe (include/moe_probe.h): the compute roof of the f32 expert MLPs.
#include "internal.cuh"
#include "moe_probe.h"

namespace moe {
namespace {

// Eight independent dependency chains per thread keep every FP32 lane busy despite the FMA
// latency; 16 unrolled steps per loop trip keep the loop overhead out of the issue slots.
__global__ void __launch_bounds__(1024) ffma_probe_kernel(float *out, int iters, float a, float b) {
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = (float)(threadIdx.x & 31) * 1e-3f + (float)i;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < 16; ++u) {
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = fmaf(x[i], a, b);
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += x[i];
    if (s == a * 1e30f) out[0] = s;  // a * 1e30 is unreachable for |a| < 1: never stores
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_fp32_ffma_probe(int32_t blocks, int32_t threads, int32_t iters,
                                            float *out, void *stream, double *flops) {
    if (blocks < 1 || blocks > 65535 || threads < 32 || threads > 1024 || threads % 32 != 0 ||
        iters < 1 || iters > (1 << 20) || !out || !flops || ((uintptr_t)out & 3u) != 0)
        return MOE_ERR_INVALID_ARG;
    moe::ffma_probe_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        out, iters, 0.999f, 1e-3f);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    *flops = 2.0 * 8.0 * 16.0 * (double)iters * (double)blocks * (double)threads;
    return MOE_OK;
}
