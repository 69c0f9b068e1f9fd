// dispatch.cu -- step 3 of the MoE layer: group the token copies by expert.
//
// lensaml.com "Mixture of Experts", Step 4 "Load Balancing" shows the histogram of routing slots
// per expert; Step 5 "Capacity & Dropped Tokens" names dropless block-sparse kernels (MegaBlocks)
// that accept any number of tokens per expert. Here every slot s = t*k + j is kept and the slots
// are stably sorted by expert, so that each expert's rows are contiguous:
//   sorted position of slot s (expert e) = offsets[e] + #{slots s' < s routed to e}.
//
// One cooperative kernel, 1024 slots per chunk, one chunk per block iteration:
//   1. Histogram without atomics: __match_any_sync groups the lanes of a warp by expert; the
//      group's lowest lane writes the group size into a per-warp row of shared memory; thread e
//      then scans the 32 warp rows of expert e in warp order. This gives the chunk aggregate and,
//      per slot, its rank inside the chunk (warp base + rank among equal lanes below it).
//   2. Decoupled look-back over chunks (Merrill & Garland, single-pass prefix scan): thread e
//      publishes (AGGREGATE, count) for its expert, then walks back over earlier chunks adding
//      aggregates until it meets an INCLUSIVE prefix, and publishes (INCLUSIVE, prefix). Each
//      flag/value pair is one 64-bit release store; readers load eight earlier words per round
//      trip (relaxed loads: the word itself is all they need).
//   3. The last chunk knows the totals: it writes counts and offsets (an exclusive scan over
//      experts by warp scans) and raises a done flag; every block waits for it and scatters
//      sorted_token and slot_of.
// The launch is cooperative, so all blocks are co-resident and every wait can be satisfied;
// each wait is still bounded by %globaltimer and reports DEV_ERR_TIMEOUT instead of hanging.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "internal.cuh"
#include "layer_dev.cuh"

namespace moe {
namespace {

using namespace dev;

__global__ void __launch_bounds__(DISPATCH_THREADS, 1) dispatch_single_kernel(DispatchArgs a) {
    __shared__ int32_t cnt[32 * 256];
    __shared__ int32_t s_tot[256], s_off[257], s_wsum[8];
    pdl_wait();
    dispatch_single_block(a, cnt, s_tot, s_off, s_wsum);
    pdl_trigger();
}

// A single-chunk layer's dispatch and its auxiliary value and z-loss in one block: the counts the
// dispatch publishes and the router's partial sums are reduced right after, in the same fixed
// order as aux_kernel (both call aux_block).
__global__ void __launch_bounds__(DISPATCH_THREADS, 1)
    dispatch_aux_kernel(DispatchArgs a, const float *psum, int64_t rows, int64_t T,
                        float *aux_out, float *zloss_out) {
    __shared__ int32_t cnt[32 * 256];
    __shared__ int32_t s_tot[256], s_off[257], s_wsum[8];
    __shared__ float part[1024];
    __shared__ float colsum[257];
    __shared__ int32_t s_counts[256];
    pdl_wait();
    dispatch_single_block(a, cnt, s_tot, s_off, s_wsum);
    __syncthreads();  // the counts written by the dispatch are visible to the whole block
    aux_block(a.counts, psum, rows, a.E, T, a.k, aux_out, zloss_out, part, colsum, s_counts);
    pdl_trigger();
}

__global__ void __launch_bounds__(DISPATCH_THREADS, 1) dispatch_kernel(DispatchArgs a) {
    __shared__ int32_t cnt[32 * 256];
    __shared__ int32_t s_tot[257], s_pub[257], s_wsum[8];
    __shared__ int s_abort;
    const int tid = threadIdx.x, E = a.E;
    if (tid == 0) s_abort = 0;
    __syncthreads();
    // a block that owns exactly one chunk keeps its ranks for the scatter
    const bool one_chunk = a.nchunks <= (int)gridDim.x;
    int keep_e = -1, keep_rank = 0;

    for (int c = blockIdx.x; c < a.nchunks; c += gridDim.x) {
        int lrank, agg;
        keep_e = chunk_ranks(a, c, cnt, &lrank, &agg);
        keep_rank = lrank;
        if (tid < E) {
            unsigned long long *mine = a.words + (size_t)c * E + tid;
            int excl = 0;
            if (c == 0) {
                if (!a.withhold) st_release(mine, FLAG_INC | (uint32_t)agg);
            } else {
                st_release(mine, FLAG_AGG | (uint32_t)agg);
                unsigned long long t_start = 0;
                int q = c - 1;
                uint32_t spins = 0;
                // walk back LB_WINDOW chunks per round trip: read their words together, then
                // add them in order up to the first INCLUSIVE one; an unpublished word ends the
                // round and is read again
                while (q >= 0) {
                    unsigned long long v[LB_WINDOW];
#pragma unroll
                    for (int i = 0; i < LB_WINDOW; ++i)
                        v[i] = q - i >= 0 ? ld_relaxed(a.words + (size_t)(q - i) * E + tid) : 0ull;
                    int used = 0;
                    bool inclusive = false;
#pragma unroll
                    for (int i = 0; i < LB_WINDOW; ++i) {
                        if (q - i < 0) break;
                        const unsigned long long flag = v[i] & 0xffffffff00000000ull;
                        if (flag == 0) break;
                        excl += (int)(uint32_t)v[i];
                        ++used;
                        if (flag == FLAG_INC) {
                            inclusive = true;
                            break;
                        }
                    }
                    if (inclusive) break;
                    q -= used;
                    if (used == 0 && (++spins & 255u) == 0) {
                        const unsigned long long now = globaltimer_ns();
                        if (t_start == 0) t_start = now;
                        else if (now - t_start > a.spin_limit_ns) {
                            report(a.dev_status, DEV_ERR_TIMEOUT);
                            s_abort = 1;
                            break;
                        }
                    }
                }
                st_release(mine, FLAG_INC | (uint32_t)(excl + agg));
            }
            a.excl[(size_t)c * E + tid] = excl;
            if (c == a.nchunks - 1) s_tot[tid] = excl + agg;
        }
        if (c == a.nchunks - 1) {
            __syncthreads();
            publish_offsets(a, s_tot, s_pub, s_wsum);
            if (tid == 0) {
                __threadfence();
                st_release_u32(a.done, 1u);
            }
        }
    }

    // Wait until the last chunk has published the offsets.
    __syncthreads();
    __shared__ int32_t s_off[257];
    if (tid == 0) {
        unsigned long long t_start = 0;
        uint32_t spins = 0;
        while (ld_acquire_u32(a.done) == 0u) {
            if ((++spins & 255u) == 0) {
                const unsigned long long now = globaltimer_ns();
                if (t_start == 0) t_start = now;
                else if (now - t_start > a.spin_limit_ns) {
                    report(a.dev_status, DEV_ERR_TIMEOUT);
                    s_abort = 1;
                    break;
                }
            }
        }
    }
    __syncthreads();
    if (s_abort) return;
    for (int e = tid; e <= E; e += DISPATCH_THREADS) s_off[e] = __ldcg(a.offsets + e);
    __syncthreads();

    for (int c = blockIdx.x; c < a.nchunks; c += gridDim.x) {
        int lrank = keep_rank, agg;
        const int e = one_chunk ? keep_e : chunk_ranks(a, c, cnt, &lrank, &agg);
        if (e >= 0) {
            const int64_t s = (int64_t)c * DISPATCH_THREADS + tid;
            const int64_t rank = (int64_t)a.excl[(size_t)c * E + e] + lrank;  // within expert e
            const int64_t pos = (int64_t)s_off[e] + rank;
            if (a.cap >= 0 && rank >= a.cap) {
                a.slot_of[s] = -1;  // over capacity: dropped
            } else if (pos >= 0 && pos < a.P) {
                a.sorted_token[pos] = (int32_t)(s / a.k);
                a.slot_of[s] = (int32_t)pos;
            } else {
                report(a.dev_status, DEV_ERR_INDEX);
            }
        }
    }
    pdl_trigger();  // (this kernel is launched cooperatively, without a dependent wait of its own)
}

// x_perm[slot_of[t k + j], :] = h[t, :] for every kept slot (slot_of >= 0; -1 marks a slot the
// capacity dropped): one thread per (token, 16-byte vector), two units in flight per thread. Each
// row of h is read once and stored to its token's k places, which is x_perm[r] =
// h[sorted_token[r]] for every kept row r.
__global__ void __launch_bounds__(256) permute_kernel(const uint4 *__restrict__ h,
                                                      const int32_t *__restrict__ slot_of,
                                                      uint4 *__restrict__ x_perm, int64_t P,
                                                      int64_t T, int k, int vecs,
                                                      uint32_t *dev_status) {
    pdl_wait();
    const int64_t units = T * vecs;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t u0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u0 < units;
         u0 += 2 * stride) {
        uint4 v[2];
        int64_t t[2];
        int iv[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int64_t u = u0 + q * stride;
            t[q] = -1;
            if (u < units) {
                t[q] = u / vecs;
                iv[q] = (int)(u - t[q] * vecs);
                v[q] = __ldg(h + u);
            }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            if (t[q] < 0) continue;
            for (int j = 0; j < k; ++j) {
                const int32_t r = __ldg(slot_of + t[q] * k + j);
                if (r == -1) continue;
                if (r < 0 || r >= P) {
                    report(dev_status, DEV_ERR_INDEX);
                    continue;
                }
                x_perm[(int64_t)r * vecs + iv[q]] = v[q];
            }
        }
    }
    pdl_trigger();
}

}  // namespace

int dispatch_blocks_per_sm() {
    // per-device cache; several host threads may fill it at once (they store the same value)
    static std::atomic<int> cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int per_sm = cache[dev].load(std::memory_order_relaxed);
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_kernel,
                                                          DISPATCH_THREADS, 0) != cudaSuccess)
            return 0;
        cache[dev].store(per_sm, std::memory_order_relaxed);
    }
    return per_sm;
}

cudaError_t launch_dispatch(const moe_config_t &c, const int32_t *topk_idx, const DispatchBufs &b,
                            cudaStream_t s, const FaultHook &hook) {
    const int64_t P = c.T * c.k;
    if (P == 0) {
        cudaError_t err = cudaMemsetAsync(b.counts, 0, sizeof(int32_t) * c.E, s);
        if (err != cudaSuccess) return err;
        return cudaMemsetAsync(b.offsets, 0, sizeof(int32_t) * (c.E + 1), s);
    }
    DispatchArgs a;
    a.idx = topk_idx;
    a.counts = b.counts;
    a.offsets = b.offsets;
    a.sorted_token = b.sorted_token;
    a.slot_of = b.slot_of;
    a.excl = b.excl;
    a.done = reinterpret_cast<uint32_t *>(b.flags);
    a.words = reinterpret_cast<unsigned long long *>(static_cast<char *>(b.flags) + 256);
    a.dev_status = b.dev_status;
    a.P = P;
    a.k = c.k;
    a.E = c.E;
    a.nchunks = (int)dispatch_chunks(c);
    a.cap = capacity_of(c);
    a.spin_limit_ns = hook.spin_limit_ns;
    a.withhold = hook.withhold;
    if (a.nchunks == 1 && !hook.withhold) {
        return launch_pdl(dispatch_single_kernel, dim3(1), dim3(DISPATCH_THREADS), 0, s, 1, a);
    }
    cudaError_t err = cudaMemsetAsync(b.flags, 0, b.flags_bytes, s);
    if (err != cudaSuccess) return err;
    const int per_sm = dispatch_blocks_per_sm();
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int64_t grid = (int64_t)per_sm * num_sms();
    if (grid > a.nchunks) grid = a.nchunks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(DISPATCH_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dispatch_kernel, a);
}

// ---------------------------------------------------------------------------------------------
// Dispatch without a caller workspace. Its scratch is this file-scope device array: the look-back
// header (done flag), up to STATIC_LOOKBACK_CELLS look-back words and as many per-chunk counts.
// Every GPU that loads the library holds it until the process exits; all calls share it.
constexpr size_t STATIC_HDR = 256;
constexpr size_t STATIC_SCRATCH_BYTES =
    STATIC_HDR + (size_t)STATIC_LOOKBACK_CELLS * 8 + (size_t)STATIC_LOOKBACK_CELLS * 4;
static __device__ __align__(256) unsigned char g_dispatch_scratch[STATIC_SCRATCH_BYTES];

// Device address of g_dispatch_scratch in the current device's context. Host code only sees a
// stand-in symbol, which must never reach a kernel. The address is looked up once per (device,
// context) -- the first call on a device, and again after cudaDeviceReset gave the device a new
// primary context (the module, and with it the array, is then loaded anew) -- under a mutex, so
// concurrent first calls from several host threads are safe.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);

static CtxGetCurrentFn ctx_get_current_fn() {
    static const CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<CtxGetCurrentFn>(p);
        return nullptr;
    }();
    return fn;
}

static cudaError_t static_scratch(unsigned char **out) {
    struct Entry {
        CUcontext ctx;
        unsigned char *ptr;
    };
    static Entry cache[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    CUcontext ctx = nullptr;
    if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS) return cudaErrorInitializationError;
    if (!ctx) {  // no context on this thread yet: cudaSetDevice binds the primary context
        err = cudaSetDevice(dev);
        if (err != cudaSuccess) return err;
        if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorInitializationError;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].ctx != ctx || !cache[dev].ptr) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_dispatch_scratch);
        if (err != cudaSuccess) return err;
        cache[dev].ctx = ctx;
        cache[dev].ptr = static_cast<unsigned char *>(p);
    }
    *out = cache[dev].ptr;
    return cudaSuccess;
}

cudaError_t launch_dispatch_static(const moe_config_t &c, const int32_t *topk_idx,
                                   int32_t *counts, int32_t *offsets, int32_t *sorted_token,
                                   int32_t *slot_of, uint32_t *status, cudaStream_t s) {
    unsigned char *scratch = nullptr;
    cudaError_t err = static_scratch(&scratch);
    if (err != cudaSuccess) return err;
    const size_t cells = (size_t)dispatch_chunks(c) * (size_t)c.E;
    DispatchBufs b;
    b.counts = counts;
    b.offsets = offsets;
    b.sorted_token = sorted_token;
    b.slot_of = slot_of;
    b.flags = scratch;                                   // done flag + look-back words, zeroed
    b.flags_bytes = STATIC_HDR + cells * 8;              // by launch_dispatch on every call
    b.excl = reinterpret_cast<int32_t *>(scratch + STATIC_HDR + (size_t)STATIC_LOOKBACK_CELLS * 8);
    // Without a caller status word, device-side failures land in the (cleared) header.
    b.dev_status = status ? status : reinterpret_cast<uint32_t *>(scratch + 64);
    return launch_dispatch(c, topk_idx, b, s);
}

cudaError_t launch_dispatch_aux(const moe_config_t &c, const int32_t *topk_idx,
                                const DispatchBufs &b, const float *psum_part, float *aux_out,
                                float *zloss_out, cudaStream_t s) {
    if (c.T == 0 || dispatch_chunks(c) != 1) return cudaErrorInvalidValue;
    DispatchArgs a = {};
    a.idx = topk_idx;
    a.counts = b.counts;
    a.offsets = b.offsets;
    a.sorted_token = b.sorted_token;
    a.slot_of = b.slot_of;
    a.dev_status = b.dev_status;
    a.P = c.T * c.k;
    a.k = c.k;
    a.E = c.E;
    a.nchunks = 1;
    a.cap = capacity_of(c);
    a.spin_limit_ns = SPIN_LIMIT_NS;
    return launch_pdl(dispatch_aux_kernel, dim3(1), dim3(DISPATCH_THREADS), 0, s, 1, a, psum_part,
                      router_partial_rows(c), c.T, aux_out, zloss_out);
}

cudaError_t launch_permute(const moe_config_t &c, const void *h, const int32_t *slot_of,
                           void *x_perm, uint32_t *dev_status, cudaStream_t s) {
    const int64_t P = c.T * c.k;
    if (P == 0) return cudaSuccess;
    const int es = c.dtype == MOE_BF16 ? 2 : 4;
    const int vecs = c.d * es / 16;
    int64_t blocks = (c.T * vecs + 511) / 512;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(permute_kernel, dim3((unsigned)blocks), dim3(256), 0, s, 1,
                      static_cast<const uint4 *>(h), slot_of, static_cast<uint4 *>(x_perm), P, c.T,
                      c.k, vecs, dev_status);
}

}  // namespace moe
