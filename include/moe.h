/*
 * moe.h -- C ABI of libmoe: the forward pass of one top-k routed mixture-of-experts FFN layer on
 * one NVIDIA B300 (sm_103a).
 *
 * The layer (llm.curionode.com "Mixture of Experts.", Plate 4, opening text; lensaml.com
 * "Mixture of Experts", Steps 2-4) replaces one FFN with E expert MLPs and a router:
 *   1. router      z = h . W_r (+ b_r), p = softmax_E(z), in f32
 *   2. top-k       the k largest logits per token and their gates
 *   3. dispatch    per-expert histogram, prefix sum, and a permutation grouping token copies by expert
 *   4. expert FFN  every expert's MLP over its contiguous block of rows
 *   5. combine     y[t] = sum_j g[t,j] . FFN_{idx[t,j]}(h[t]), plus the auxiliary value E . sum f P
 *
 * Conventions for every entry point
 *   - Pointers to tensors are DEVICE pointers (cudaMalloc'd or PyTorch-owned), caller-owned.
 *     The library allocates nothing and keeps no state between calls; all scratch lives in the
 *     caller's workspace `ws` (see moe_workspace_size) -- except for moe_build_dispatch_static,
 *     whose scratch is a static device array inside the library, and the pipeline objects of
 *     moe_pipeline.h, which own their device buffers and streams.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Every call is
 *     asynchronous on that stream; results are valid once the stream reaches the call. A
 *     workspace serves one call at a time: calls that may overlap (on different streams) need
 *     different workspaces.
 *   - All tensors are dense row-major. "dtype" below is cfg->dtype: MOE_F32 (float) or MOE_BF16
 *     (bfloat16, raw 16-bit storage). Router weights, router bias, expert biases and gates are
 *     always float. Integer tensors are int32.
 *   - Device pointers must be 16-byte aligned.
 *   - Errors: argument checks run on the host before anything is launched and return a status
 *     without touching the device. A failed launch returns MOE_ERR_CUDA. Failures detected on the
 *     device (a spin-wait that ran out of its time limit, an out-of-range expert index) never trap:
 *     the kernel records a bit in a status word inside `ws` and returns; moe_device_status() reads
 *     and clears it. There is no CPU fallback.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t moe_status_t;
enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer, k outside [1, E] */
    MOE_ERR_UNSUPPORTED = 2,  /* a dtype / activation / gate / bias combination not built */
    MOE_ERR_WORKSPACE = 3,    /* ws smaller than moe_workspace_size() */
    MOE_ERR_CUDA = 4,         /* a CUDA launch or runtime call failed */
    MOE_ERR_TIMEOUT = 5,      /* (device) a bounded spin-wait gave up; outputs are invalid */
    MOE_ERR_DEVICE_INDEX = 6  /* (device) an expert index outside [0, E) was read */
};

enum { MOE_F32 = 0, MOE_BF16 = 1 };
enum { MOE_ACT_GELU_TANH = 0, MOE_ACT_SWIGLU = 1 };
enum { MOE_GATE_RENORM = 0, MOE_GATE_RAW_PROB = 1 };

/* Layer shape and variant.
 *   T tokens (>= 0); d model width; f expert hidden width; E experts; k experts per token.
 *   Limits: 1 <= E <= 256, 1 <= k <= E, d and f multiples of 64 (>= 64), T * k < 2^31.
 *   act  MOE_ACT_GELU_TANH : expert(x) = W2 GELU_tanh(W1 x + b1) + b2   (2 matrices)
 *        MOE_ACT_SWIGLU    : expert(x) = W2 (SiLU(W1 x) * (W3 x))       (3 matrices, no biases)
 *   gate MOE_GATE_RENORM   : g = softmax over the chosen logits (Mixtral form, sums to 1)
 *        MOE_GATE_RAW_PROB : g = p, the full-softmax probability (Switch top-1 form)
 *   has_bias : expert biases b1 [E, f] and b2 [E, d] (float) are present; GELU form only.
 *   capacity_factor : 0 = dropless. > 0: every expert processes at most
 *            C = floor(capacity_factor * T * k / E) routing slots -- the first C in token order --
 *            and the other slots are dropped: they contribute nothing to y (a token whose slots
 *            are all dropped gets y = 0, its residual passing around the layer), the kept gates
 *            are not renormalised, and the auxiliary value still uses the routed counts
 *            (lensaml.com "Mixture of Experts", Step 5 "Capacity & Dropped Tokens").
 *   fuse_gather : 0 or 1 (else MOE_ERR_INVALID_ARG); bf16 only, ignored for f32. 1: moe_forward
 *            does not build the permuted copy x_perm; the first expert GEMM reads its rows of h
 *            through sorted_token with 4-row TMA gathers, and the workspace holds no x_perm
 *            (P d 2 bytes less). Same bits as 0, but slower on the shapes measured here: the
 *            gather repeats for each of the f/128 column tiles of an expert, where the permute
 *            kernel gathers every row once. */
typedef struct {
    int64_t T;
    int32_t d, f, E, k;
    int32_t dtype;
    int32_t act;
    int32_t gate;
    int32_t has_bias;
    float capacity_factor;
    int32_t fuse_gather;
} moe_config_t;

/* Bytes of workspace every call below needs for `cfg` (the largest of their needs, so one
 * workspace serves them all). The workspace must be zero-filled once after allocation (or passed
 * through moe_workspace_init); afterwards the library keeps its status word consistent itself.
 * Returns MOE_ERR_INVALID_ARG for an invalid cfg. */
moe_status_t moe_workspace_size(const moe_config_t *cfg, size_t *bytes);

/* Zero the workspace header -- its first 2048 bytes: the device status word and the counters of
 * the combine that moe_forward fuses into the expert launch of small f32 layers -- on `stream`.
 * MOE_ERR_INVALID_ARG if ws is not 16-byte aligned or ws_bytes < 2048. */
moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Rows of the router's per-block partial sums psum_part [rows, E + 1]. */
moe_status_t moe_router_partials(const moe_config_t *cfg, int64_t *rows);

/* Steps 1-2. Router, softmax and top-k (lensaml.com "Mixture of Experts", Step 2 "The Router"
 * and Step 3 "Top-k Routing"; arjunjaggi.com "Mixture of Experts in LLMs", "Switch Transformers":
 * the router is kept in f32).
 *   h        [T, d] dtype           input activations
 *   W_r      [d, E] float           router weight;  b_r [E] float or NULL
 *   sel_bias [E] float or NULL      selection-only routing bias b (lensaml.com Step 4 names
 *            DeepSeek-V3's per-expert routing bias that replaces the auxiliary loss; the rule is
 *            the DeepSeek-V3 Technical Report's auxiliary-loss-free balancing): the k experts are
 *            chosen by p + b instead of the logits; the gates, p (hence psum_part and the
 *            auxiliary value) stay those of the unbiased router. See moe_update_sel_bias.
 *   topk_idx [T, k] int32  (out)    chosen experts, keys descending (the logits, or p + b),
 *                                   ties to the lower index
 *   gates    [T, k] float  (out)    gate of each chosen expert (RENORM or RAW_PROB)
 *   psum_part [moe_router_partials rows, E + 1] float (out) per-block sums in a fixed order:
 *            columns 0..E-1 the sums of p over the block's tokens (input of the auxiliary value),
 *            column E the sum of (log sum_e exp z[t, e])^2 (input of the router z-loss).
 *   ws       workspace (moe_workspace_size bytes): for bf16 h and E <= 128 with more tokens than
 *            the few-token path takes, the logits run on the tensor cores with W_r split exactly
 *            into three bf16 pieces stored in ws, and their partial sums are staged in ws.
 * Logits are accumulated in f32 from the stored h (every product exact); exp and log are CUDA's
 * expf and logf. */
moe_status_t moe_router_topk(const moe_config_t *cfg, const void *h, const float *W_r,
                             const float *b_r, const float *sel_bias, int32_t *topk_idx,
                             float *gates, float *psum_part, void *ws, size_t ws_bytes,
                             void *stream);

/* Step 3. Dispatch (lensaml.com "Mixture of Experts", Step 4 "Load Balancing": the histogram of
 * routing slots per expert; Step 5 "Capacity & Dropped Tokens": dropless grouping of any number
 * of tokens per expert). A stable counting sort of the slots s = t*k + j by topk_idx[s]:
 *   counts       [E]    int32 (out)  slots routed to each expert
 *   offsets      [E+1]  int32 (out)  exclusive prefix sum of counts; offsets[E] = T k
 *                                    (with a capacity C: of min(counts, C); offsets[E] = kept)
 *   sorted_token [T k]  int32 (out)  token of each sorted row, order (expert, token) ascending
 *                                    (rows [0, offsets[E]) are written)
 *   slot_of      [T k]  int32 (out)  sorted row of slot s (the inverse permutation); -1 for a
 *                                    slot dropped by the capacity
 *   x_perm       [T k, d] dtype (out, may be NULL): x_perm[r] = h[sorted_token[r]] for the
 *                                    offsets[E] kept rows
 *   h            [T, d] dtype, read only when x_perm is not NULL.
 * One cooperative kernel (histogram without atomics, decoupled look-back scan over blocks) and,
 * when x_perm is given, one gather kernel. Bit-exact and deterministic. */
moe_status_t moe_build_dispatch(const moe_config_t *cfg, const int32_t *topk_idx, const void *h,
                                int32_t *counts, int32_t *offsets, int32_t *sorted_token,
                                int32_t *slot_of, void *x_perm, void *ws, size_t ws_bytes,
                                void *stream);

/* Step 3 for callers that cannot allocate device memory -- for instance a custom operator inside
 * a host runtime that owns every device buffer and hands the operator only its inputs and
 * outputs, or a latency-critical loop that must never call cudaMalloc (which can synchronise the
 * device). The pages have no counterpart of this call; it exists only for such callers.
 * Same arguments, outputs and results as moe_build_dispatch, but no workspace: the dispatch
 * scratch (look-back words, per-chunk counts, the done flag) is a file-scope device array inside
 * libmoe of STATIC_SCRATCH = 256 + 12 * 65536 bytes (768.25 KiB), which every GPU that loads the
 * library holds until the process exits. It serves at most 65536 look-back cells:
 *   ceil(T k / 1024) * E <= 65536   (e.g. T k <= 1M slots for E = 64, 256K slots for E = 256);
 * larger shapes are rejected with MOE_ERR_WORKSPACE before anything is launched.
 *   status  (device, may be NULL) one uint32 the caller zeroes; device-side failures are OR-ed
 *           into it (1 = a spin-wait ran out of time, 2 = an index out of range). With NULL they
 *           are not reported.
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress) and
 * caches it per device and context (a later call looks it up again only if the device's context
 * changed, e.g. after cudaDeviceReset); the cache is guarded by a mutex, so host threads may make
 * their first calls concurrently. Make the first call on a device before any stream capture. No
 * call allocates or frees memory.
 * All calls share the one array: each call clears the parts that must start at zero, and calls
 * whose kernels overlap on the GPU (different streams without ordering) race on it. */
moe_status_t moe_build_dispatch_static(const moe_config_t *cfg, const int32_t *topk_idx,
                                       const void *h, int32_t *counts, int32_t *offsets,
                                       int32_t *sorted_token, int32_t *slot_of, void *x_perm,
                                       uint32_t *status, void *stream);

/* Step 4. Every expert's MLP over its block of rows of x_perm (llm.curionode.com "Mixture of
 * Experts.", "Workshop": the experts are MLPs; lensaml.com "Mixture of Experts", Step 1 and
 * Step 6: a full expert is three d x f matrices).
 *   x_perm  [T k, d] dtype          rows grouped by expert, as moe_build_dispatch writes them
 *   offsets [E+1] int32             expert e owns rows [offsets[e], offsets[e+1])
 *   W1 [E, f, d], W3 [E, f, d] (SwiGLU only, else NULL), W2 [E, d, f]: dtype, out x in
 *   b1 [E, f], b2 [E, d] float, only when cfg->has_bias (else NULL)
 *   y_perm  [T k, d] dtype (out)    expert output of every row
 * The hidden activations H [T k, f] (dtype) live in ws. bf16: tcgen05 tensor cores, f32
 * accumulation, H rounded to bf16. f32: CUDA-core f32 FMA. */
moe_status_t moe_expert_ffn(const moe_config_t *cfg, const void *x_perm, const int32_t *offsets,
                            const void *W1, const float *b1, const void *W3, const void *W2,
                            const float *b2, void *y_perm, void *ws, size_t ws_bytes,
                            void *stream);

/* Step 5a. Gate-weighted combine (lensaml.com "Mixture of Experts", Step 3: y = sum g . E(h)):
 *   y[t, :] = sum_{j<k} gates[t, j] * y_perm[slot_of[t k + j], :], in f32, j ascending, then
 *   rounded to dtype; slots with slot_of = -1 (dropped) are skipped.  y [T, d] dtype (out). */
moe_status_t moe_combine(const moe_config_t *cfg, const void *y_perm, const int32_t *slot_of,
                         const float *gates, void *y, void *stream);

/* Step 5b. Auxiliary load-balancing value (lensaml.com "Mixture of Experts", Step 4):
 *   aux = E . sum_e f_e P_e,  f_e = counts[e] / (T k),  P_e = (1/T) sum_t p[t, e]
 * (the weight alpha is the caller's), and the router z-loss (arjunjaggi.com "Mixture of Experts
 * in LLMs" names ST-MoE's z-loss, a penalty on large router logits; the formula is ST-MoE's,
 * Zoph et al. 2022):
 *   zloss = (1/T) sum_t (log sum_e exp z[t, e])^2     (z the router logits, b_r included)
 * Both reduced in a fixed order. aux_out: one float (device); zloss_out: one float or NULL.
 * T = 0 gives 0 for both. */
moe_status_t moe_aux_loss(const moe_config_t *cfg, const int32_t *counts, const float *psum_part,
                          float *aux_out, float *zloss_out, void *stream);

/* One step of the selection-only routing bias (DeepSeek-V3's rule, as for sel_bias above):
 * sel_bias[e] += gamma when expert e received fewer routing slots than the mean T k / E,
 * -= gamma when more, unchanged when equal (compared exactly in integers). counts [E] int32 and
 * sel_bias [E] float are device pointers; gamma must be finite. */
moe_status_t moe_update_sel_bias(const moe_config_t *cfg, const int32_t *counts, float *sel_bias,
                                 float gamma, void *stream);

/* Steps 1-5 in one call. sel_bias [E] float or NULL as for moe_router_topk. y [T, d] dtype
 * (out); aux_out one float (out); zloss_out one float (out) or NULL; topk_idx_out [T, k] and
 * counts_out [E] are optional copies of the routing (NULL to skip). Everything else lives in ws.
 * Same results as the step calls in sequence, bit for bit, except for a dropless (capacity_factor
 * 0) top-1 bf16 layer: there the second expert GEMM writes y[t] = g * expert(h[t]) itself, with
 * one bf16 rounding instead of two (no y_perm, no combine kernel). Fewer kernels than the step
 * calls where the shape allows: a layer whose T k slots fit one dispatch chunk (<= 1024) reduces
 * the auxiliary value in the dispatch's kernel; f32 layers read their expert rows of h directly
 * (no permuted copy), and small f32 layers (T k d <= 262144, d <= 8192) form y in the second
 * expert launch (no combine kernel). moe_forward_launch_count tells how many kernels run. */
moe_status_t moe_forward(const moe_config_t *cfg, const void *h, const float *W_r,
                         const float *b_r, const float *sel_bias, const void *W1,
                         const float *b1, const void *W3, const void *W2, const float *b2,
                         void *y, float *aux_out, float *zloss_out, int32_t *topk_idx_out,
                         int32_t *counts_out, void *ws, size_t ws_bytes, void *stream);

/* moe_forward that also records two caller-created CUDA events (cudaEvent_t, passed as void*) on
 * `stream`: ffn_begin right before the expert-FFN launches and ffn_end right after them, so that
 * a caller can time the dominant step live inside a longer run. Same results as moe_forward. */
moe_status_t moe_forward_events(const moe_config_t *cfg, const void *h, const float *W_r,
                                const float *b_r, const float *sel_bias, const void *W1,
                                const float *b1, const void *W3, const void *W2,
                                const float *b2, void *y, float *aux_out, float *zloss_out,
                                int32_t *topk_idx_out, int32_t *counts_out, void *ws,
                                size_t ws_bytes, void *stream, void *ffn_begin, void *ffn_end);

/* Number of kernels one moe_forward call with `cfg` launches (device memsets not counted; 0 for
 * T = 0). Host-only: reads no device state. MOE_ERR_INVALID_ARG for an invalid cfg or a NULL
 * `kernels`. */
moe_status_t moe_forward_launch_count(const moe_config_t *cfg, int32_t *kernels);

/* Synchronise `stream`, read the device status word in ws, clear it, and return MOE_OK,
 * MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_INDEX (MOE_ERR_CUDA if the copy itself fails). */
moe_status_t moe_device_status(void *ws, void *stream);

/* A static string naming a status code. */
const char *moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
