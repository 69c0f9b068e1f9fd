// internal.cuh -- declarations shared by libmoe's translation units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// ------------------------------------------------------------------------------------------
// device status word (first 4 bytes of every workspace)
enum : uint32_t {
    DEV_ERR_TIMEOUT = 1u,  // a bounded spin-wait gave up
    DEV_ERR_INDEX = 2u,    // an expert / token / row index outside its range was read
};

// Every spin-wait in libmoe gives up after this many nanoseconds of %globaltimer.
constexpr unsigned long long SPIN_LIMIT_NS = 2000000000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void report(uint32_t *dev_status, uint32_t bits) {
    if (dev_status) atomicOr(dev_status, bits);
}

// Programmatic dependent launch. Every kernel of the library is launched with it allowed
// (launch_pdl), so it may be scheduled while the previous kernel on the stream finishes; it calls
// pdl_wait() before it touches memory that earlier stream work writes (the wait returns once that
// work has completed and its writes are visible), and pdl_trigger() after its own work, so that
// the next kernel's launch overlaps this one's tail. Both are no-ops without a dependent launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Test hook: a shorter spin limit and one withheld signal, so that a bounded wait runs out
// (the kernel then records DEV_ERR_TIMEOUT and returns). Normal calls use the defaults.
struct FaultHook {
    unsigned long long spin_limit_ns = SPIN_LIMIT_NS;
    int withhold = 0;  // dispatch: chunk 0 never publishes; GEMM: the producer issues no loads
};

// ------------------------------------------------------------------------------------------
// shapes and the workspace layout
constexpr int DISPATCH_THREADS = 1024;  // slots per dispatch chunk
constexpr int GEMM_BM = 128;            // rows per tensor-core tile

// The workspace header: the status word at offset 0 and, from WS_ARRIVE_OFFSET, the arrival
// counters of the fused f32 combine (one per output column tile). moe_workspace_init zeroes it.
constexpr size_t WS_HEADER_BYTES = 2048;
constexpr size_t WS_ARRIVE_OFFSET = 1024;
constexpr int F32_COMBINE_TILES = (int)((WS_HEADER_BYTES - WS_ARRIVE_OFFSET) / 4);

struct WsLayout {
    size_t status;        // header: u32 device status word, combine arrival counters
    size_t disp_flags;    // u32 done flag + pad, then nchunks*E u64 look-back words
    size_t disp_flags_bytes;
    size_t disp_excl;     // nchunks*E int32 (per-chunk exclusive counts)
    size_t psum;          // router partial sums [rows, E] f32
    size_t router;        // router scratch (split weights of the tensor-core router)
    size_t topk_idx, gates, counts, offsets, sorted_token, slot_of, aux;
    size_t x_perm, H, y_perm;
    size_t total;
};

// Per-expert capacity in routing slots: floor(factor T k / E), or -1 when dropless.
inline int64_t capacity_of(const moe_config_t &c) {
    if (!(c.capacity_factor > 0.f)) return -1;
    const double C = (double)c.capacity_factor * (double)c.T * (double)c.k / (double)c.E;
    return (int64_t)floor(C);
}

inline int64_t dispatch_chunks(const moe_config_t &c) {
    const int64_t P = c.T * c.k;
    return (P + DISPATCH_THREADS - 1) / DISPATCH_THREADS;
}

// Rows of psum_part [rows, E + 1] the router writes (one per router block; depends only on the
// shape).
int64_t router_partial_rows(const moe_config_t &c);
// Workspace bytes the router needs (tensor-core path: the split router weights and the partial
// logits).
size_t router_scratch_bytes(const moe_config_t &c);
// Kernels one router call launches for T > 0 (the tensor-core path: W_r split, logits, select).
int router_launches(const moe_config_t &c);
constexpr int ROUTER_TC_MAX_E = 128;   // tensor-core router: bf16 h, E <= 128
constexpr int ROUTER_TC_TOKENS = 128;  // tokens per tensor-core logits tile
size_t router_tc_scratch_bytes(const moe_config_t &c);
// K chunks of the tensor-core logits (a pure function of the shape), the padded expert count
// (row stride of the partial logits), and where the partial logits [S][T][Epad] f32 live.
int router_tc_splits(const moe_config_t &c);
int router_tc_epad(const moe_config_t &c);
float *router_tc_logits(void *scratch, const moe_config_t &c);

WsLayout ws_layout(const moe_config_t &c);
// The argument checks every entry point applies to a configuration (MOE_OK when valid).
moe_status_t validate_config(const moe_config_t *c);
// Kernels one moe_backward call launches for c (bf16); saved: the pre-activations come from
// moe_forward_train (no recompute).
int backward_launches(const moe_config_t &c, bool saved);
// Backward workspace: its size, and where moe_forward_train stores the pre-activations A1, A3
// ([P, f] bf16 each; A3 for SwiGLU only).
size_t backward_ws_bytes(const moe_config_t &c);
size_t backward_pre_offset(const moe_config_t &c, int which);

int num_sms();

// <<<grid, block, smem, s>>> with programmatic dependent launch allowed (and a cluster of
// cluster_x CTAs along x when > 1).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, int cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int n = 1;
    if (cluster_x > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster_x;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (kernel, device, size).
cudaError_t set_max_dynamic_smem(const void *kernel, size_t bytes);
// Resident blocks per SM of the dispatch kernel on the current device (queried once).
int dispatch_blocks_per_sm();

// ------------------------------------------------------------------------------------------
// launchers (each returns the launch's cudaError_t)
cudaError_t launch_router_topk(const moe_config_t &c, const void *h, const float *W_r,
                               const float *b_r, const float *sel_bias, int32_t *topk_idx,
                               float *gates, float *psum_part, void *scratch,
                               uint32_t *dev_status, cudaStream_t s);
// W_r split and the partial logits on the tensor cores (the selection follows in router.cu).
cudaError_t launch_router_tc(const moe_config_t &c, const void *h, const float *W_r,
                             void *scratch, uint32_t *dev_status, cudaStream_t s);

struct DispatchBufs {
    int32_t *counts, *offsets, *sorted_token, *slot_of;
    void *flags;        // workspace look-back region (zeroed by the launcher)
    size_t flags_bytes;
    int32_t *excl;
    uint32_t *dev_status;
};
cudaError_t launch_dispatch(const moe_config_t &c, const int32_t *topk_idx, const DispatchBufs &b,
                            cudaStream_t s, const FaultHook &hook = FaultHook());
// Dispatch whose scratch is a file-scope device array (no workspace); nchunks * E must not
// exceed STATIC_LOOKBACK_CELLS.
constexpr int64_t STATIC_LOOKBACK_CELLS = 65536;
cudaError_t launch_dispatch_static(const moe_config_t &c, const int32_t *topk_idx,
                                   int32_t *counts, int32_t *offsets, int32_t *sorted_token,
                                   int32_t *slot_of, uint32_t *status, cudaStream_t s);
// x_perm[slot_of[s]] = h[s / k] for every kept slot s (slot_of = -1: dropped by a capacity).
cudaError_t launch_permute(const moe_config_t &c, const void *h, const int32_t *slot_of,
                           void *x_perm, uint32_t *dev_status, cudaStream_t s);
cudaError_t launch_combine(const moe_config_t &c, const void *y_perm, const int32_t *slot_of,
                           const float *gates, void *y, uint32_t *dev_status, cudaStream_t s);
// aux_out: E sum f P; zloss_out (may be nullptr): the router z-loss.
cudaError_t launch_aux(const moe_config_t &c, const int32_t *counts, const float *psum_part,
                       float *aux_out, float *zloss_out, cudaStream_t s);
// Dispatch and auxiliary value of a layer whose slots fit one dispatch chunk (T k <= 1024), in
// one single-block kernel: the results of launch_dispatch followed by launch_aux.
cudaError_t launch_dispatch_aux(const moe_config_t &c, const int32_t *topk_idx,
                                const DispatchBufs &b, const float *psum_part, float *aux_out,
                                float *zloss_out, cudaStream_t s);
cudaError_t launch_update_sel_bias(const moe_config_t &c, const int32_t *counts, float *sel_bias,
                                   float gamma, cudaStream_t s);

struct FfnBufs {
    const void *x_perm;
    const int32_t *offsets;
    const void *W1, *W3, *W2;
    const float *b1, *b2;
    void *H;       // [P, f] workspace
    void *y_perm;  // [P, d]
    uint32_t *dev_status;
    // fused variants (tensor-core path, moe_forward only):
    const void *gather_h = nullptr;          // GEMM1 reads A rows h[sorted_token[r]] directly
    const int32_t *sorted_token = nullptr;
    void *scatter_y = nullptr;               // top-1: GEMM2 writes y[token] = g * expert(h)
    const float *gates = nullptr;
    // f32, ffn_f32_combine_ok: the second launch also forms y = sum_j g_j y_perm[slot_of] in the
    // last block of every column tile (arrive: zeroed counters in the workspace header, one per
    // column tile, left zero again)
    void *combine_y = nullptr;
    const int32_t *slot_of = nullptr;
    uint32_t *arrive = nullptr;
    // training forward (tensor-core path): GEMM1 also stores its pre-activations, [P, f] bf16
    // each (pre3: SwiGLU only)
    void *pre1 = nullptr, *pre3 = nullptr;
};
// The f32 combine fused into the second expert launch: at most this many slot elements (T k d),
// which the last block of each column tile reads and combines.
constexpr int64_t F32_COMBINE_MAX = 256 * 1024;
bool ffn_f32_combine_ok(const moe_config_t &c);
cudaError_t launch_ffn_f32(const moe_config_t &c, const FfnBufs &b, cudaStream_t s);
cudaError_t launch_ffn_tc(const moe_config_t &c, const FfnBufs &b, cudaStream_t s,
                          const FaultHook &hook = FaultHook());

// Row-grouped tensor-core GEMM with a plain store: out[r, n] = A_r . B[e N + n] (+ bias[e, n])
// for r in expert e's rows [offsets[e], offsets[e+1]); A row r is row A_rows[r] of a
// [A_src_rows, K] tensor when A_rows is given (TMA gathers), else row r of A [P, K]. bf16.
cudaError_t launch_gemm_rows(const void *A, const int32_t *A_rows, int64_t A_src_rows,
                             const void *B, int64_t P, int E, int K, int N,
                             const int32_t *offsets, const float *bias, void *out,
                             uint32_t *dev_status, cudaStream_t s);
// The same with B read MN-major from its natural layout: expert e's B is rows
// [e b_krows, (e + 1) b_krows) of a [E b_krows, N] tensor (rows = the K index); with
// b_ksplit = b_krows / 64 > 0, B is that tensor stacked along K on B3's rows (K = 2 b_krows),
// else K = b_krows. No bias, no gather.
cudaError_t launch_gemm_rows_bmn(const void *A, const void *B, const void *B3, int b_krows,
                                 int b_ksplit, int64_t P, int E, int K, int N,
                                 const int32_t *offsets, void *out, uint32_t *dev_status,
                                 cudaStream_t s);
// K-grouped tensor-core GEMM (weight gradients): out[e M + m, n] = sum over the rows k in
// [kseg[e], kseg[e+1]) of A[k, m] B[k, n], both operands MN-major in the padded row layout:
// A [rows, M] with row stride lda and B [rows, N] with row stride ldb (bf16, zero pad rows);
// kseg device int32 [E+1], multiples of 64. Empty segments give zero tiles.
// map_rows > 0: rows of A and B at or past map_rows read as zeros (K extent `rows` rounded up
// past the data); out_f32 (may be null): f32 output [E M, N] instead of the bf16 out.
cudaError_t launch_gemm_kgroup_mn(const void *A, int64_t lda, const void *B, int64_t ldb,
                                  const int32_t *kseg, int E, int M, int N, int64_t rows,
                                  void *out, uint32_t *dev_status, cudaStream_t s,
                                  int64_t map_rows = 0, float *out_f32 = nullptr);
// Row-grouped GEMM with K-major A and B and an f32 output [P, N] (no bias).
cudaError_t launch_gemm_rows_f32(const void *A, const void *B, int64_t P, int E, int K, int N,
                                 const int32_t *offsets, float *out, uint32_t *dev_status,
                                 cudaStream_t s);

}  // namespace moe
