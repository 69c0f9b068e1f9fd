// pipeline.cu -- moe_pipeline_* (include/moe_pipeline.h): batches in host memory through
// moe_forward, with the copy-in, the layer and the copy-out of neighbouring batches overlapped on
// three streams. Built on the public entry points only.
//
// Batch n uses slot s = n mod 2 of the device buffers (h, y, aux). Its three steps:
//   in      : [wait fwd_done[s] of batch n-2: h[s] is free]  h_host -> h[s]     record h_ready[s]
//   compute : wait h_ready[s]; [wait y_copied[s] of batch n-2: y[s], aux[s] are free]
//             moe_forward(h[s] -> y[s], aux[s])                                   record fwd_done[s]
//   out     : wait fwd_done[s]; y[s] -> y_host, aux[s] -> aux_host               record y_copied[s]
// so batch n+1's copy-in and batch n-1's copy-out run while batch n computes. The workspace is
// shared by all batches; their forwards are ordered on the compute stream.
#include <cuda_runtime.h>
#include <stdint.h>

#include <new>

#include "moe_pipeline.h"

struct moe_pipeline {
    moe_config_t cfg;
    const float *W_r, *b_r, *sel_bias, *b1, *b2;
    const void *W1, *W3, *W2;
    cudaStream_t compute;   // the caller's stream
    cudaStream_t in, out;   // owned
    void *h[2], *y[2];
    float *aux[2];
    void *ws;
    size_t ws_bytes, act_bytes;
    cudaEvent_t h_ready[2], fwd_done[2], y_copied[2], fence;
    int64_t n;              // batches submitted
    bool need_fence;        // the next submit orders its copies after the caller's stream
};

namespace {

bool aligned16(const void *p) { return p && ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void *p) { return p && ((uintptr_t)p & 3u) == 0; }

void release(moe_pipeline *p) {
    if (p->in) cudaStreamSynchronize(p->in);
    if (p->out) cudaStreamSynchronize(p->out);
    cudaStreamSynchronize(p->compute);
    for (int s = 0; s < 2; ++s) {
        if (p->h[s]) cudaFree(p->h[s]);
        if (p->y[s]) cudaFree(p->y[s]);
        if (p->aux[s]) cudaFree(p->aux[s]);
        if (p->h_ready[s]) cudaEventDestroy(p->h_ready[s]);
        if (p->fwd_done[s]) cudaEventDestroy(p->fwd_done[s]);
        if (p->y_copied[s]) cudaEventDestroy(p->y_copied[s]);
    }
    if (p->fence) cudaEventDestroy(p->fence);
    if (p->ws) cudaFree(p->ws);
    if (p->in) cudaStreamDestroy(p->in);
    if (p->out) cudaStreamDestroy(p->out);
    delete p;
}

}  // namespace

extern "C" {

moe_status_t moe_pipeline_create(const moe_config_t *cfg, const float *W_r, const float *b_r,
                                 const float *sel_bias, const void *W1, const float *b1,
                                 const void *W3, const void *W2, const float *b2, void *stream,
                                 moe_pipeline_t **out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    size_t ws_bytes = 0;
    const moe_status_t st = moe_workspace_size(cfg, &ws_bytes);
    if (st != MOE_OK) return st;
    if (!aligned4(W_r) || (b_r && !aligned4(b_r)) || (sel_bias && !aligned4(sel_bias)) ||
        !aligned16(W1) || !aligned16(W2))
        return MOE_ERR_INVALID_ARG;
    if (cfg->act == MOE_ACT_SWIGLU && !aligned16(W3)) return MOE_ERR_INVALID_ARG;
    if (cfg->has_bias && (!aligned4(b1) || !aligned4(b2))) return MOE_ERR_INVALID_ARG;

    moe_pipeline *p = new (std::nothrow) moe_pipeline();
    if (!p) return MOE_ERR_CUDA;
    p->cfg = *cfg;
    p->W_r = W_r;
    p->b_r = b_r;
    p->sel_bias = sel_bias;
    p->W1 = W1;
    p->b1 = b1;
    p->W3 = W3;
    p->W2 = W2;
    p->b2 = b2;
    p->compute = static_cast<cudaStream_t>(stream);
    p->ws_bytes = ws_bytes;
    p->act_bytes = (size_t)cfg->T * cfg->d * (cfg->dtype == MOE_BF16 ? 2 : 4);
    p->need_fence = true;
    const size_t slot = p->act_bytes > 0 ? p->act_bytes : 16;
    bool ok = cudaStreamCreateWithFlags(&p->in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p->fence, cudaEventDisableTiming) == cudaSuccess &&
              cudaMalloc(&p->ws, ws_bytes) == cudaSuccess &&
              cudaMemsetAsync(p->ws, 0, ws_bytes, p->compute) == cudaSuccess;
    for (int s = 0; s < 2 && ok; ++s) {
        ok = cudaMalloc(&p->h[s], slot) == cudaSuccess && cudaMalloc(&p->y[s], slot) == cudaSuccess &&
             cudaMalloc((void **)&p->aux[s], 16) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->h_ready[s], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->fwd_done[s], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->y_copied[s], cudaEventDisableTiming) == cudaSuccess;
    }
    if (!ok) {
        release(p);
        return MOE_ERR_CUDA;
    }
    *out = p;
    return MOE_OK;
}

moe_status_t moe_pipeline_submit(moe_pipeline_t *p, const void *h_host, void *y_host,
                                 float *aux_host) {
    if (!p || !h_host || !y_host || !aux_host) return MOE_ERR_INVALID_ARG;
    const int s = (int)(p->n & 1);
    const bool reuse = p->n >= 2;  // slot s was used by batch n-2
    if (p->need_fence) {
        if (cudaEventRecord(p->fence, p->compute) != cudaSuccess ||
            cudaStreamWaitEvent(p->in, p->fence, 0) != cudaSuccess ||
            cudaStreamWaitEvent(p->out, p->fence, 0) != cudaSuccess)
            return MOE_ERR_CUDA;
        p->need_fence = false;
    }
    if (reuse && cudaStreamWaitEvent(p->in, p->fwd_done[s], 0) != cudaSuccess) return MOE_ERR_CUDA;
    if (p->act_bytes > 0 &&
        cudaMemcpyAsync(p->h[s], h_host, p->act_bytes, cudaMemcpyHostToDevice, p->in) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaEventRecord(p->h_ready[s], p->in) != cudaSuccess ||
        cudaStreamWaitEvent(p->compute, p->h_ready[s], 0) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (reuse && cudaStreamWaitEvent(p->compute, p->y_copied[s], 0) != cudaSuccess)
        return MOE_ERR_CUDA;
    const moe_status_t st = moe_forward(&p->cfg, p->h[s], p->W_r, p->b_r, p->sel_bias, p->W1,
                                        p->b1, p->W3, p->W2, p->b2, p->y[s], p->aux[s], nullptr,
                                        nullptr, nullptr, p->ws, p->ws_bytes, p->compute);
    if (st != MOE_OK) return st;
    if (cudaEventRecord(p->fwd_done[s], p->compute) != cudaSuccess ||
        cudaStreamWaitEvent(p->out, p->fwd_done[s], 0) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (p->act_bytes > 0 &&
        cudaMemcpyAsync(y_host, p->y[s], p->act_bytes, cudaMemcpyDeviceToHost, p->out) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaMemcpyAsync(aux_host, p->aux[s], sizeof(float), cudaMemcpyDeviceToHost, p->out) !=
            cudaSuccess ||
        cudaEventRecord(p->y_copied[s], p->out) != cudaSuccess)
        return MOE_ERR_CUDA;
    ++p->n;
    return MOE_OK;
}

moe_status_t moe_pipeline_join(moe_pipeline_t *p, void *stream) {
    if (!p) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the copy-out stream runs in order and each copy-out waited for its forward: its last event
    // covers every batch
    if (p->n > 0 && cudaStreamWaitEvent(s, p->y_copied[(p->n - 1) & 1], 0) != cudaSuccess)
        return MOE_ERR_CUDA;
    p->need_fence = true;
    return MOE_OK;
}

moe_status_t moe_pipeline_device_status(moe_pipeline_t *p) {
    if (!p) return MOE_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(p->in) != cudaSuccess || cudaStreamSynchronize(p->out) != cudaSuccess)
        return MOE_ERR_CUDA;
    p->need_fence = true;
    return moe_device_status(p->ws, p->compute);
}

moe_status_t moe_pipeline_destroy(moe_pipeline_t *p) {
    if (!p) return MOE_OK;
    release(p);
    return MOE_OK;
}

}  // extern "C"
