// router.cu -- steps 1-2 of the MoE layer: router logits, softmax, top-k and gates.
//
// lensaml.com "Mixture of Experts", Step 2 "The Router": logits = h . W_r and a softmax over the
// E experts. Step 3 "Top-k Routing": the k highest-scoring experts run; their gates are either a
// softmax over the chosen logits (Mixtral: softmax(TopK(h . W_g))) or the raw probability p_i
// (Switch top-1). arjunjaggi.com "Mixture of Experts in LLMs", "Switch Transformers": the router
// is kept in float32 while the rest runs in bfloat16.
//
// One block owns BT tokens and all E experts. Phase 1 is a register-blocked f32 contraction of
// the [BT, d] activation tile with W_r [d, E] (both staged through shared memory in K-steps of
// 32; every logit is a sequential FMA chain over i = 0..d-1). Phase 2 gives each warp one token:
// max, sum of exponentials and k rounds of a warp arg-max (larger logit first, lower index on
// equal logits), all by butterfly shuffles, so the result is deterministic. The block then sums
// its tokens' probabilities per expert in token order into one row of psum_part, the input of
// the auxiliary value.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int RT_THREADS = 256;
constexpr int DK = 32;  // K-step of the contraction

template <typename Tin> __device__ __forceinline__ float to_f32(Tin v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

struct RouterArgs {
    const void *h;
    const float *W_r, *b_r;
    int32_t *idx;
    float *gates, *psum;
    int64_t T;
    int d, E, k, gate_mode;
};

// Tile geometry for E experts: threads form TR rows x TC columns, each computing RT tokens x RE
// experts (experts strided by TC so that shared-memory reads of W_r are conflict-free).
struct Geo {
    int RT, RE, TC, TR, BT;
};
__host__ __device__ inline Geo geometry(int E) {
    Geo g;
    if (E % 4 == 0 && E >= 32) { g.RT = 8; g.RE = 4; } else { g.RT = 1; g.RE = 1; }
    g.TC = E / g.RE;
    g.TR = RT_THREADS / g.TC;
    g.BT = g.TR * g.RT;
    return g;
}

template <int RT, int RE, typename Tin>
__global__ void __launch_bounds__(RT_THREADS) router_topk_kernel(RouterArgs a) {
    extern __shared__ float sm[];
    const int E = a.E, d = a.d;
    const int TC = E / RE;
    const int TR = RT_THREADS / TC;
    const int BT = TR * RT;
    const int tid = threadIdx.x;
    const int64_t t0 = (int64_t)blockIdx.x * BT;
    const Tin *h = reinterpret_cast<const Tin *>(a.h);

    float *hs = sm;                       // [BT][DK + 1]
    float *wsm = sm + BT * (DK + 1);      // [DK][E]
    float *zs = sm;                       // [BT][E], reuses the staging area after phase 1

    const bool active = tid < TR * TC;
    const int r = tid / TC, c = tid % TC;
    float acc[RT][RE];
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
        for (int j = 0; j < RE; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < d; k0 += DK) {
        for (int q = tid; q < BT * DK; q += RT_THREADS) {
            const int row = q / DK, col = q % DK;
            const int64_t tok = t0 + row;
            hs[row * (DK + 1) + col] = tok < a.T ? to_f32<Tin>(h[tok * d + k0 + col]) : 0.f;
        }
        for (int q = tid; q < DK * E; q += RT_THREADS)
            wsm[q] = a.W_r[(int64_t)k0 * E + q];
        __syncthreads();
        if (active) {
#pragma unroll 4
            for (int kk = 0; kk < DK; ++kk) {
                float hv[RT], wv[RE];
#pragma unroll
                for (int i = 0; i < RT; ++i) hv[i] = hs[(r + TR * i) * (DK + 1) + kk];
#pragma unroll
                for (int j = 0; j < RE; ++j) wv[j] = wsm[kk * E + c + TC * j];
#pragma unroll
                for (int i = 0; i < RT; ++i)
#pragma unroll
                    for (int j = 0; j < RE; ++j) acc[i][j] = fmaf(hv[i], wv[j], acc[i][j]);
            }
        }
        __syncthreads();
    }
    if (active) {
#pragma unroll
        for (int i = 0; i < RT; ++i)
#pragma unroll
            for (int j = 0; j < RE; ++j) {
                const int e = c + TC * j;
                zs[(r + TR * i) * E + e] = acc[i][j] + (a.b_r ? a.b_r[e] : 0.f);
            }
    }
    __syncthreads();

    // Phase 2: one warp per token.
    const int warp = tid >> 5, lane = tid & 31;
    constexpr int NW = RT_THREADS / 32;
    constexpr int MAXM = 8;  // E <= 256 -> at most 8 logits per lane
    for (int row = warp; row < BT; row += NW) {
        const int64_t tok = t0 + row;
        float *zr = zs + row * E;
        if (tok >= a.T) {
            for (int e = lane; e < E; e += 32) zr[e] = 0.f;
            continue;
        }
        float v[MAXM];
        float zmax = -INFINITY;
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            const int e = lane + 32 * m;
            v[m] = e < E ? zr[e] : -INFINITY;
            zmax = fmaxf(zmax, v[m]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
        float ssum = 0.f;
#pragma unroll
        for (int m = 0; m < MAXM; ++m)
            if (lane + 32 * m < E) ssum += expf(v[m] - zmax);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);

        // k rounds of arg-max; lane j keeps the j-th winner.
        uint32_t chosen = 0;
        int sel_e = -1;
        float sel_v = 0.f;
        for (int j = 0; j < a.k; ++j) {
            float bv = -INFINITY;
            int be = 0x7fffffff;
#pragma unroll
            for (int m = 0; m < MAXM; ++m) {
                const int e = lane + 32 * m;
                if (e < E && !((chosen >> m) & 1u) && (v[m] > bv || (v[m] == bv && e < be))) {
                    bv = v[m];
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
            }
            if ((be & 31) == lane) chosen |= 1u << (be >> 5);
            if (lane == j) { sel_e = be; sel_v = bv; }
        }
        float g;
        if (a.gate_mode == MOE_GATE_RAW_PROB) {
            g = expf(sel_v - zmax) / ssum;
        } else {
            const float ex = lane < a.k ? expf(sel_v - zmax) : 0.f;
            float gs = ex;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, o);
            g = ex / gs;
        }
        if (lane < a.k) {
            a.idx[tok * a.k + lane] = sel_e;
            a.gates[tok * a.k + lane] = g;
        }
        __syncwarp();
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            const int e = lane + 32 * m;
            if (e < E) zr[e] = expf(v[m] - zmax) / ssum;
        }
    }
    __syncthreads();
    if (tid < E) {
        float s = 0.f;
        for (int row = 0; row < BT; ++row) s += zs[row * E + tid];
        a.psum[(int64_t)blockIdx.x * E + tid] = s;
    }
}

template <int RT, int RE, typename Tin>
cudaError_t launch_t(const RouterArgs &a, int blocks, size_t smem, cudaStream_t s) {
    auto kern = router_topk_kernel<RT, RE, Tin>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    kern<<<blocks, RT_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

int router_block_tokens(int E) { return geometry(E).BT; }

cudaError_t launch_router_topk(const moe_config_t &c, const void *h, const float *W_r,
                               const float *b_r, int32_t *topk_idx, float *gates,
                               float *psum_part, cudaStream_t s) {
    if (c.T == 0) return cudaSuccess;
    const Geo g = geometry(c.E);
    const int64_t blocks = (c.T + g.BT - 1) / g.BT;
    const size_t stage = sizeof(float) * ((size_t)g.BT * (DK + 1) + (size_t)DK * c.E);
    const size_t logits = sizeof(float) * (size_t)g.BT * c.E;
    const size_t smem = stage > logits ? stage : logits;
    RouterArgs a{h, W_r, b_r, topk_idx, gates, psum_part, c.T, c.d, c.E, c.k, c.gate};
    const bool wide = g.RE == 4;
    if (c.dtype == MOE_BF16)
        return wide ? launch_t<8, 4, __nv_bfloat16>(a, (int)blocks, smem, s)
                    : launch_t<1, 1, __nv_bfloat16>(a, (int)blocks, smem, s);
    return wide ? launch_t<8, 4, float>(a, (int)blocks, smem, s)
                : launch_t<1, 1, float>(a, (int)blocks, smem, s);
}

}  // namespace moe
