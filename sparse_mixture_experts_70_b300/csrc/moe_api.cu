// moe_api.cu -- the extern "C" entry points declared in include/moe.h: argument checks, the
// workspace layout, and the launch sequence of the layer forward. No allocation, no global state
// beyond a per-device cache of the SM count.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "internal.cuh"
#include "moe_debug.h"

namespace moe {

int num_sms() {
    // per-device cache; several host threads may fill it at once (they store the same value)
    static std::atomic<int> cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t set_max_dynamic_smem(const void *kernel, size_t bytes) {
    struct Entry {
        const void *kernel;
        int dev;
        size_t bytes;
    };
    static Entry table[64];
    static int used = 0;
    static std::mutex mu;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (table[i].kernel == kernel && table[i].dev == dev && table[i].bytes >= bytes)
            return cudaSuccess;
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (err != cudaSuccess) return err;
    for (int i = 0; i < used; ++i)
        if (table[i].kernel == kernel && table[i].dev == dev) {
            table[i].bytes = bytes;
            return cudaSuccess;
        }
    if (used < 64) table[used++] = Entry{kernel, dev, bytes};
    return cudaSuccess;
}

static size_t align_up(size_t x) { return (x + 1023) & ~(size_t)1023; }

WsLayout ws_layout(const moe_config_t &c) {
    WsLayout L;
    const size_t P = (size_t)(c.T * c.k);
    const size_t es = c.dtype == MOE_BF16 ? 2 : 4;
    const size_t E = (size_t)c.E;
    const size_t nch = (size_t)dispatch_chunks(c);
    size_t off = 0;
    L.status = off;                       off = align_up(off + WS_HEADER_BYTES);
    L.disp_flags = off;
    L.disp_flags_bytes = 256 + nch * E * 8;
    off = align_up(off + L.disp_flags_bytes);
    L.disp_excl = off;                    off = align_up(off + nch * E * 4);
    L.psum = off;                         off = align_up(off + (size_t)router_partial_rows(c) * (E + 1) * 4);
    L.router = off;                       off = align_up(off + router_scratch_bytes(c));
    L.topk_idx = off;                     off = align_up(off + P * 4);
    L.gates = off;                        off = align_up(off + P * 4);
    L.counts = off;                       off = align_up(off + E * 4);
    L.offsets = off;                      off = align_up(off + (E + 1) * 4);
    L.sorted_token = off;                 off = align_up(off + P * 4);
    L.slot_of = off;                      off = align_up(off + P * 4);
    L.aux = off;                          off = align_up(off + 4);
    L.x_perm = off;
    if (!(c.fuse_gather && c.dtype == MOE_BF16)) off = align_up(off + P * (size_t)c.d * es);
    L.H = off;                            off = align_up(off + P * (size_t)c.f * es);
    L.y_perm = off;                       off = align_up(off + P * (size_t)c.d * es);
    L.total = off;
    return L;
}

}  // namespace moe

using namespace moe;

namespace {

moe_status_t check_cfg(const moe_config_t *c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->T < 0 || c->E < 1 || c->E > 256 || c->k < 1 || c->k > c->E) return MOE_ERR_INVALID_ARG;
    if (c->d < 64 || c->f < 64 || c->d % 64 != 0 || c->f % 64 != 0) return MOE_ERR_INVALID_ARG;
    if (c->T * (int64_t)c->k >= ((int64_t)1 << 31)) return MOE_ERR_INVALID_ARG;
    if ((int64_t)c->E * c->d >= ((int64_t)1 << 31) || (int64_t)c->E * c->f >= ((int64_t)1 << 31))
        return MOE_ERR_INVALID_ARG;
    if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (c->act != MOE_ACT_GELU_TANH && c->act != MOE_ACT_SWIGLU) return MOE_ERR_UNSUPPORTED;
    if (c->gate != MOE_GATE_RENORM && c->gate != MOE_GATE_RAW_PROB) return MOE_ERR_UNSUPPORTED;
    if (c->k > 32) return MOE_ERR_UNSUPPORTED;
    if (c->has_bias && c->act == MOE_ACT_SWIGLU) return MOE_ERR_UNSUPPORTED;
    if (!(c->capacity_factor >= 0.f) || !isfinite(c->capacity_factor)) return MOE_ERR_INVALID_ARG;
    if (c->fuse_gather != 0 && c->fuse_gather != 1) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace

moe_status_t moe::validate_config(const moe_config_t *c) { return check_cfg(c); }

namespace {

bool aligned16(const void *p) { return p && ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void *p) { return p && ((uintptr_t)p & 3u) == 0; }

moe_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

extern "C" {

moe_status_t moe_workspace_size(const moe_config_t *cfg, size_t *bytes) {
    const moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = ws_layout(*cfg).total;
    return MOE_OK;
}

moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, void *stream) {
    if (!aligned16(ws) || ws_bytes < WS_HEADER_BYTES) return MOE_ERR_INVALID_ARG;
    return from_cuda(
        cudaMemsetAsync(ws, 0, WS_HEADER_BYTES, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_router_partials(const moe_config_t *cfg, int64_t *rows) {
    const moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if (!rows) return MOE_ERR_INVALID_ARG;
    *rows = router_partial_rows(*cfg);
    return MOE_OK;
}

moe_status_t moe_router_topk(const moe_config_t *cfg, const void *h, const float *W_r,
                             const float *b_r, const float *sel_bias, int32_t *topk_idx,
                             float *gates, float *psum_part, void *ws, size_t ws_bytes,
                             void *stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    if (cfg->T == 0) return MOE_OK;
    if (!aligned16(h) || !aligned4(W_r) || (b_r && !aligned4(b_r)) ||
        (sel_bias && !aligned4(sel_bias)) || !aligned4(topk_idx) || !aligned4(gates) ||
        !aligned4(psum_part))
        return MOE_ERR_INVALID_ARG;
    char *w = static_cast<char *>(ws);
    return from_cuda(launch_router_topk(*cfg, h, W_r, b_r, sel_bias, topk_idx, gates, psum_part,
                                        w + L.router, reinterpret_cast<uint32_t *>(w + L.status),
                                        static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_build_dispatch(const moe_config_t *cfg, const int32_t *topk_idx, const void *h,
                                int32_t *counts, int32_t *offsets, int32_t *sorted_token,
                                int32_t *slot_of, void *x_perm, void *ws, size_t ws_bytes,
                                void *stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if (!aligned4(counts) || !aligned4(offsets) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cfg->T > 0) {
        if (!aligned4(topk_idx) || !aligned4(sorted_token) || !aligned4(slot_of))
            return MOE_ERR_INVALID_ARG;
        if (x_perm && (!aligned16(x_perm) || !aligned16(h))) return MOE_ERR_INVALID_ARG;
    }
    char *w = static_cast<char *>(ws);
    DispatchBufs b{counts, offsets, sorted_token, slot_of, w + L.disp_flags, L.disp_flags_bytes,
                   reinterpret_cast<int32_t *>(w + L.disp_excl),
                   reinterpret_cast<uint32_t *>(w + L.status)};
    st = from_cuda(launch_dispatch(*cfg, topk_idx, b, s));
    if (st != MOE_OK || !x_perm || cfg->T == 0) return st;
    return from_cuda(launch_permute(*cfg, h, slot_of, x_perm, b.dev_status, s));
}

moe_status_t moe_build_dispatch_static(const moe_config_t *cfg, const int32_t *topk_idx,
                                       const void *h, int32_t *counts, int32_t *offsets,
                                       int32_t *sorted_token, int32_t *slot_of, void *x_perm,
                                       uint32_t *status, void *stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if (dispatch_chunks(*cfg) * (int64_t)cfg->E > STATIC_LOOKBACK_CELLS) return MOE_ERR_WORKSPACE;
    if (!aligned4(counts) || !aligned4(offsets) || (status && !aligned4(status)))
        return MOE_ERR_INVALID_ARG;
    if (cfg->T > 0) {
        if (!aligned4(topk_idx) || !aligned4(sorted_token) || !aligned4(slot_of))
            return MOE_ERR_INVALID_ARG;
        if (x_perm && (!aligned16(x_perm) || !aligned16(h))) return MOE_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = from_cuda(launch_dispatch_static(*cfg, topk_idx, counts, offsets, sorted_token, slot_of,
                                          status, s));
    if (st != MOE_OK || !x_perm || cfg->T == 0) return st;
    return from_cuda(launch_permute(*cfg, h, slot_of, x_perm, status, s));
}

moe_status_t moe_expert_ffn(const moe_config_t *cfg, const void *x_perm, const int32_t *offsets,
                            const void *W1, const float *b1, const void *W3, const void *W2,
                            const float *b2, void *y_perm, void *ws, size_t ws_bytes,
                            void *stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    if (cfg->T == 0) return MOE_OK;
    if (!aligned16(x_perm) || !aligned4(offsets) || !aligned16(W1) || !aligned16(W2) ||
        !aligned16(y_perm))
        return MOE_ERR_INVALID_ARG;
    if (cfg->act == MOE_ACT_SWIGLU && !aligned16(W3)) return MOE_ERR_INVALID_ARG;
    if (cfg->has_bias && (!aligned4(b1) || !aligned4(b2))) return MOE_ERR_INVALID_ARG;
    char *w = static_cast<char *>(ws);
    FfnBufs b{x_perm, offsets, W1, W3, W2, b1, b2, w + L.H, y_perm,
              reinterpret_cast<uint32_t *>(w + L.status)};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return from_cuda(cfg->dtype == MOE_BF16 ? launch_ffn_tc(*cfg, b, s) : launch_ffn_f32(*cfg, b, s));
}

moe_status_t moe_combine(const moe_config_t *cfg, const void *y_perm, const int32_t *slot_of,
                         const float *gates, void *y, void *stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if (cfg->T == 0) return MOE_OK;
    if (!aligned16(y_perm) || !aligned4(slot_of) || !aligned4(gates) || !aligned16(y))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_combine(*cfg, y_perm, slot_of, gates, y, nullptr,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_aux_loss(const moe_config_t *cfg, const int32_t *counts, const float *psum_part,
                          float *aux_out, float *zloss_out, void *stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if (!aligned4(aux_out) || (zloss_out && !aligned4(zloss_out))) return MOE_ERR_INVALID_ARG;
    if (cfg->T > 0 && (!aligned4(counts) || !aligned4(psum_part))) return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_aux(*cfg, counts, psum_part, aux_out, zloss_out,
                                static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_update_sel_bias(const moe_config_t *cfg, const int32_t *counts, float *sel_bias,
                                 float gamma, void *stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if (!aligned4(counts) || !aligned4(sel_bias) || !isfinite(gamma)) return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_update_sel_bias(*cfg, counts, sel_bias, gamma,
                                            static_cast<cudaStream_t>(stream)));
}

// The fused variants moe_forward takes. The first expert launch gathers its rows of h itself (no
// permuted copy): always for f32 (a 16-byte cp.async per piece, from any row), with fuse_gather
// on the tensor-core path. A dropless top-1 bf16 layer's second GEMM scatters g * output straight
// into y (no combine kernel). A layer whose slots fit one dispatch chunk reduces its auxiliary
// value in the dispatch's block (dispatch_aux). A small f32 layer's second expert launch also
// forms y (f32_combine). Every variant gives the step calls' bits except the top-1 scatter (one
// bf16 rounding fewer).
struct ForwardPlan {
    bool gather, scatter, dispatch_aux, f32_combine;
};

// NVTX range over the launches of one step of the layer (host side: it marks where the step's
// kernels are issued; profilers can filter kernels by it). Costs nothing without a tool attached.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

static ForwardPlan plan_of(const moe_config_t &c) {
    const bool tc = c.dtype == MOE_BF16;
    return {!tc || c.fuse_gather != 0, tc && c.k == 1 && capacity_of(c) < 0,
            c.T > 0 && dispatch_chunks(c) == 1, !tc && ffn_f32_combine_ok(c)};
}

static moe_status_t forward_impl(const moe_config_t *cfg, const void *h, const float *W_r,
                                 const float *b_r, const float *sel_bias, const void *W1,
                                 const float *b1, const void *W3, const void *W2,
                                 const float *b2, void *y, float *aux_out, float *zloss_out,
                                 int32_t *topk_idx_out, int32_t *counts_out, void *ws,
                                 size_t ws_bytes, void *stream, cudaEvent_t ev_ffn0,
                                 cudaEvent_t ev_ffn1, void *bws = nullptr,
                                 size_t bws_bytes = 0) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    const moe_config_t &c = *cfg;
    if (!aligned16(ws) || !aligned4(aux_out) || (zloss_out && !aligned4(zloss_out)))
        return MOE_ERR_INVALID_ARG;
    if (c.T > 0) {
        if (!aligned16(h) || !aligned4(W_r) || (b_r && !aligned4(b_r)) ||
            (sel_bias && !aligned4(sel_bias)) || !aligned16(W1) || !aligned16(W2) ||
            !aligned16(y))
            return MOE_ERR_INVALID_ARG;
        if (c.act == MOE_ACT_SWIGLU && !aligned16(W3)) return MOE_ERR_INVALID_ARG;
        if (c.has_bias && (!aligned4(b1) || !aligned4(b2))) return MOE_ERR_INVALID_ARG;
        if ((topk_idx_out && !aligned4(topk_idx_out)) || (counts_out && !aligned4(counts_out)))
            return MOE_ERR_INVALID_ARG;
    }
    const WsLayout L = ws_layout(c);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    if (bws && (c.dtype != MOE_BF16)) return MOE_ERR_UNSUPPORTED;
    if (bws && (!aligned16(bws) || bws_bytes < backward_ws_bytes(c))) return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *w = static_cast<char *>(ws);
    uint32_t *dev_status = reinterpret_cast<uint32_t *>(w + L.status);
    int32_t *topk = topk_idx_out ? topk_idx_out : reinterpret_cast<int32_t *>(w + L.topk_idx);
    int32_t *counts = counts_out ? counts_out : reinterpret_cast<int32_t *>(w + L.counts);
    float *gates = reinterpret_cast<float *>(w + L.gates);
    float *psum = reinterpret_cast<float *>(w + L.psum);
    int32_t *offsets = reinterpret_cast<int32_t *>(w + L.offsets);
    int32_t *sorted_token = reinterpret_cast<int32_t *>(w + L.sorted_token);
    int32_t *slot_of = reinterpret_cast<int32_t *>(w + L.slot_of);
    void *x_perm = w + L.x_perm;
    void *y_perm = w + L.y_perm;

    if (c.T == 0) {
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.E, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(aux_out, 0, sizeof(float), s);
        if (e == cudaSuccess && zloss_out) e = cudaMemsetAsync(zloss_out, 0, sizeof(float), s);
        return from_cuda(e);
    }
    const ForwardPlan plan = plan_of(c);
    const bool scatter = plan.scatter;
    DispatchBufs db{counts, offsets, sorted_token, slot_of, w + L.disp_flags, L.disp_flags_bytes,
                    reinterpret_cast<int32_t *>(w + L.disp_excl), dev_status};
    NvtxRange layer_range("moe_forward");
    cudaError_t e;
    {
        NvtxRange r("moe router + top-k");
        e = launch_router_topk(c, h, W_r, b_r, sel_bias, topk, gates, psum, w + L.router,
                               dev_status, s);
    }
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    // the auxiliary value and z-loss need only the counts and the router's partial sums: reduce
    // them right after the dispatch, while both are still in L2, not after the expert GEMMs have
    // streamed the weights through it (for a single-chunk layer, in the dispatch's own block)
    {
        NvtxRange r("moe dispatch + aux + permute");
        if (plan.dispatch_aux) {
            if ((e = launch_dispatch_aux(c, topk, db, psum, aux_out, zloss_out, s)) != cudaSuccess)
                return MOE_ERR_CUDA;
        } else {
            if ((e = launch_dispatch(c, topk, db, s)) != cudaSuccess) return MOE_ERR_CUDA;
            if ((e = launch_aux(c, counts, psum, aux_out, zloss_out, s)) != cudaSuccess)
                return MOE_ERR_CUDA;
        }
        if (!plan.gather &&
            (e = launch_permute(c, h, slot_of, x_perm, dev_status, s)) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    FfnBufs fb{x_perm, offsets, W1, W3, W2, b1, b2, w + L.H, y_perm, dev_status};
    fb.sorted_token = sorted_token;
    if (plan.gather) fb.gather_h = h;
    if (scatter) {
        fb.scatter_y = y;
        fb.gates = gates;
    }
    if (bws) {
        fb.pre1 = static_cast<char *>(bws) + backward_pre_offset(c, 0);
        fb.pre3 = static_cast<char *>(bws) + backward_pre_offset(c, 1);
    }
    if (plan.f32_combine) {
        fb.combine_y = y;
        fb.slot_of = slot_of;
        fb.gates = gates;
        fb.arrive = reinterpret_cast<uint32_t *>(w + L.status + WS_ARRIVE_OFFSET);
    }
    if (ev_ffn0 && cudaEventRecord(ev_ffn0, s) != cudaSuccess) return MOE_ERR_CUDA;
    {
        NvtxRange r("moe expert ffn");
        e = c.dtype == MOE_BF16 ? launch_ffn_tc(c, fb, s) : launch_ffn_f32(c, fb, s);
    }
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (ev_ffn1 && cudaEventRecord(ev_ffn1, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (!scatter && !plan.f32_combine) {
        NvtxRange r("moe combine");
        if ((e = launch_combine(c, y_perm, slot_of, gates, y, dev_status, s)) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status_t moe_debug_dispatch_timeout(const moe_config_t *cfg, const int32_t *topk_idx,
                                        int32_t *counts, int32_t *offsets,
                                        int32_t *sorted_token, int32_t *slot_of, void *ws,
                                        size_t ws_bytes, uint64_t spin_limit_ns, void *stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if (spin_limit_ns < 1000000ull || spin_limit_ns > 2000000000ull) return MOE_ERR_INVALID_ARG;
    if (dispatch_chunks(*cfg) < 2) return MOE_ERR_INVALID_ARG;
    if (!aligned4(topk_idx) || !aligned4(counts) || !aligned4(offsets) || !aligned4(sorted_token) ||
        !aligned4(slot_of) || !aligned16(ws))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    char *w = static_cast<char *>(ws);
    DispatchBufs b{counts, offsets, sorted_token, slot_of, w + L.disp_flags, L.disp_flags_bytes,
                   reinterpret_cast<int32_t *>(w + L.disp_excl),
                   reinterpret_cast<uint32_t *>(w + L.status)};
    FaultHook hook;
    hook.spin_limit_ns = spin_limit_ns;
    hook.withhold = 1;
    return from_cuda(launch_dispatch(*cfg, topk_idx, b, static_cast<cudaStream_t>(stream), hook));
}

moe_status_t moe_debug_expert_ffn_timeout(const moe_config_t *cfg, const void *x_perm,
                                          const int32_t *offsets, const void *W1, const float *b1,
                                          const void *W3, const void *W2, const float *b2,
                                          void *y_perm, void *ws, size_t ws_bytes,
                                          uint64_t spin_limit_ns, void *stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if (cfg->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (spin_limit_ns < 1000000ull || spin_limit_ns > 2000000000ull) return MOE_ERR_INVALID_ARG;
    if (!aligned16(ws) || !aligned16(x_perm) || !aligned4(offsets) || !aligned16(W1) ||
        !aligned16(W2) || !aligned16(y_perm) || (cfg->act == MOE_ACT_SWIGLU && !aligned16(W3)))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    if (cfg->T == 0) return MOE_OK;
    char *w = static_cast<char *>(ws);
    FfnBufs b{x_perm, offsets, W1, W3, W2, b1, b2, w + L.H, y_perm,
              reinterpret_cast<uint32_t *>(w + L.status)};
    FaultHook hook;
    hook.spin_limit_ns = spin_limit_ns;
    hook.withhold = 1;
    return from_cuda(launch_ffn_tc(*cfg, b, static_cast<cudaStream_t>(stream), hook));
}

}  // extern "C"

extern "C" {

moe_status_t moe_forward_launch_count(const moe_config_t *cfg, int32_t *kernels) {
    const moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if (!kernels) return MOE_ERR_INVALID_ARG;
    if (cfg->T == 0) {
        *kernels = 0;
        return MOE_OK;
    }
    const ForwardPlan plan = plan_of(*cfg);
    // router (+ split), dispatch and aux (one kernel for a single chunk), permute, two FFN
    // launches, combine
    *kernels = router_launches(*cfg) + (plan.dispatch_aux ? 1 : 2) + (plan.gather ? 0 : 1) + 2 +
               ((plan.scatter || plan.f32_combine) ? 0 : 1);
    return MOE_OK;
}

moe_status_t moe_forward(const moe_config_t *cfg, const void *h, const float *W_r,
                         const float *b_r, const float *sel_bias, const void *W1,
                         const float *b1, const void *W3, const void *W2, const float *b2,
                         void *y, float *aux_out, float *zloss_out, int32_t *topk_idx_out,
                         int32_t *counts_out, void *ws, size_t ws_bytes, void *stream) {
    return forward_impl(cfg, h, W_r, b_r, sel_bias, W1, b1, W3, W2, b2, y, aux_out, zloss_out,
                        topk_idx_out, counts_out, ws, ws_bytes, stream, nullptr, nullptr);
}

moe_status_t moe_forward_train(const moe_config_t *cfg, const void *h, const float *W_r,
                               const float *b_r, const float *sel_bias, const void *W1,
                               const float *b1, const void *W3, const void *W2, const float *b2,
                               void *y, float *aux_out, float *zloss_out, int32_t *topk_idx_out,
                               int32_t *counts_out, void *ws, size_t ws_bytes, void *bws,
                               size_t bws_bytes, void *stream) {
    if (!bws) return MOE_ERR_INVALID_ARG;
    return forward_impl(cfg, h, W_r, b_r, sel_bias, W1, b1, W3, W2, b2, y, aux_out, zloss_out,
                        topk_idx_out, counts_out, ws, ws_bytes, stream, nullptr, nullptr, bws,
                        bws_bytes);
}

moe_status_t moe_forward_events(const moe_config_t *cfg, const void *h, const float *W_r,
                                const float *b_r, const float *sel_bias, const void *W1,
                                const float *b1, const void *W3, const void *W2,
                                const float *b2, void *y, float *aux_out, float *zloss_out,
                                int32_t *topk_idx_out, int32_t *counts_out, void *ws,
                                size_t ws_bytes, void *stream, void *ffn_begin, void *ffn_end) {
    if (!ffn_begin || !ffn_end) return MOE_ERR_INVALID_ARG;
    return forward_impl(cfg, h, W_r, b_r, sel_bias, W1, b1, W3, W2, b2, y, aux_out, zloss_out,
                        topk_idx_out, counts_out, ws, ws_bytes, stream,
                        static_cast<cudaEvent_t>(ffn_begin), static_cast<cudaEvent_t>(ffn_end));
}

moe_status_t moe_device_status(void *ws, void *stream) {
    if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (word != 0) {
        if (cudaMemsetAsync(ws, 0, sizeof(word), s) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (word & DEV_ERR_TIMEOUT) return MOE_ERR_TIMEOUT;
    if (word & DEV_ERR_INDEX) return MOE_ERR_DEVICE_INDEX;
    return MOE_OK;
}

const char *moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_DEVICE_INDEX: return "MOE_ERR_DEVICE_INDEX";
        default: return "MOE_ERR_UNKNOWN";
    }
}

}  // extern "C"
