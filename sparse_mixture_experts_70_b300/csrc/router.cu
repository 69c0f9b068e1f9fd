// router.cu -- steps 1-2 of the MoE layer: router logits, softmax, top-k and gates.
//
// lensaml.com "Mixture of Experts", Step 2 "The Router": logits = h . W_r and a softmax over the
// E experts. Step 3 "Top-k Routing": the k highest-scoring experts run; their gates are either a
// softmax over the chosen logits (Mixtral: softmax(TopK(h . W_g))) or the raw probability p_i
// (Switch top-1). arjunjaggi.com "Mixture of Experts in LLMs", "Switch Transformers": the router
// is kept in float32 while the rest runs in bfloat16.
//
// Four paths share the work by shape (the choice is a pure function of the shape, so
// moe_router_partials can tell the caller how many partial-sum rows there will be):
//   router_splitd_kernel E <= 32 and few tokens: one token per block, the warps split d and read
//                        W_r from L2 (latency-bound shapes such as decode).
//   router_small_kernel  f32 h, E <= 32, W_r fits in shared memory: one warp per token, lanes across
//                        d with 16-byte loads of h, W_r resident in shared memory in a
//                        lane-interleaved layout (conflict-free 16-byte reads); the E partial sums
//                        are folded across lanes by a butterfly then a reduce-scatter, leaving
//                        lane e with logit e. Bandwidth-bound on h.
//   router_logits_kernel bf16 h, E <= 128, more tokens than the split-d kernel takes: partial
//                        logits on the tensor cores (router_tc.cu), then router_select_kernel,
//                        warp per token, for the per-token step below.
//   router_tile_kernel   everything else: a block owns BT tokens x all E experts and runs a
//                        register-blocked f32 FMA contraction staged through shared memory.
// All four end with the same per-token step: max, sum of exponentials and k rounds of arg-max
// (larger logit first, lower index on equal logits; with a selection-only routing bias b, larger
// p + b first), and per-block sums in a fixed order: one row of psum_part [rows, E + 1] per block
// holding the sums of p per expert (input of the auxiliary value) and the sum of the squared
// log-sum-exp of the logits (input of the router z-loss).
#include "internal.cuh"

namespace moe {
namespace {

constexpr int RT_THREADS = 256;
constexpr int DK = 32;  // K-step of the tiled contraction

template <typename Tin> __device__ __forceinline__ float to_f32(Tin v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

struct RouterArgs {
    const void *h;
    const float *W_r, *b_r;
    const float *sel_bias;  // selection-only routing bias [E] or nullptr
    int32_t *idx;
    float *gates, *psum;
    int64_t T;
    int d, E, k, gate_mode, tokens_per_block;
};

// A float's bits as an unsigned key with the same order (-inf lowest; no NaN here).
__device__ __forceinline__ uint32_t order_key(float x) {
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Per-token step of every router path (warp per token). Lane l holds the logits v[m] of experts
// l + 32 m (-inf where absent) and, when `biased`, their selection biases sb[m]. Every
// exponential ex = exp(z - zmax) is taken once and serves the softmax sum, the gates and p. The
// k experts are chosen by the largest keys -- the logits, or p + b with a selection bias -- in
// k rounds of arg-max on the redux unit over order-preserving integer keys (exact: the largest
// key, then the lowest index among equal ones); lane j keeps the j-th. Gates: RENORM = the
// softmax over the chosen logits (ex_j / sum of the chosen ex), RAW_PROB = p_j. Writes idx and
// gates, returns p[m] = ex / sum and the log-sum-exp of the logits.
template <int MAXM>
__device__ __forceinline__ void route_token(const float (&v)[MAXM], const float (&sb)[MAXM],
                                            bool biased, int E, int k, int gate_mode,
                                            int64_t tok, int32_t *idx, float *gates,
                                            float (&p)[MAXM], float &lse) {
    const int lane = threadIdx.x & 31;
    float lmax = -INFINITY;
#pragma unroll
    for (int m = 0; m < MAXM; ++m) lmax = fmaxf(lmax, v[m]);
    const float zmax = key_float(__reduce_max_sync(0xffffffffu, order_key(lmax)));
    float ex[MAXM], ssum = 0.f;
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
        ex[m] = lane + 32 * m < E ? expf(v[m] - zmax) : 0.f;
        ssum += ex[m];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    const float inv = 1.f / ssum;
    lse = zmax + logf(ssum);
    float key[MAXM];
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
        p[m] = ex[m] * inv;
        key[m] = biased ? p[m] + sb[m] : v[m];
    }
    uint32_t chosen = 0;
    int sel_e = -1;
    float sel_x = 0.f;
    for (int j = 0; j < k; ++j) {
        // this lane's best remaining candidate (its lowest index among equal keys)
        float bv = -INFINITY, bx = 0.f;
        int be = 0x7fffffff;
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            const int e = lane + 32 * m;
            if (e < E && !((chosen >> m) & 1u) && (key[m] > bv || be == 0x7fffffff)) {
                bv = key[m];
                be = e;
                bx = ex[m];
            }
        }
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, order_key(bv));
        const int win = (int)__reduce_min_sync(
            0xffffffffu, (be != 0x7fffffff && order_key(bv) == kmax) ? (uint32_t)be : 0xffffffffu);
        const float wx = __shfl_sync(0xffffffffu, bx, win & 31);
        if ((win & 31) == lane) chosen |= 1u << (win >> 5);
        if (lane == j) {
            sel_e = win;
            sel_x = wx;
        }
    }
    float g;
    if (gate_mode == MOE_GATE_RAW_PROB) {
        g = sel_x * inv;
    } else {
        float gs = lane < k ? sel_x : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, o);
        g = sel_x / gs;
    }
    if (lane < k) {
        idx[tok * k + lane] = sel_e;
        gates[tok * k + lane] = g;
    }
}

// ---------------------------------------------------------------------------------------------
// small E: warp per token, W_r resident in shared memory

constexpr int SMALL_WARPS = 8;
constexpr size_t SMALL_SMEM_MAX = 192 * 1024;

__host__ __device__ inline int small_emax(int E) { return E <= 8 ? 8 : (E <= 16 ? 16 : 32); }

// Eight consecutive inputs of one token, widened to f32 (one 16-byte load for bf16, two for f32).
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&x)[8]) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        x[2 * q] = __uint_as_float(w[q] << 16);
        x[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8(const float *p, float (&x)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Lane l of a warp covers inputs i = 256 j + 8 l + q (q < 8). W_r[i, e] (padded to EMAX experts)
// sits at float4 index ((j * 8 + q) * EMAX/4 + e/4) * 32 + l, so the 32 lanes of a warp read 32
// consecutive 16-byte words for every (j, q, e/4).
template <typename Tin, int EMAX>
__global__ void __launch_bounds__(RT_THREADS) router_small_kernel(RouterArgs a) {
    extern __shared__ float4 w4[];
    __shared__ float red[SMALL_WARPS][32];
    constexpr int V = EMAX / 4;
    const int E = a.E, d = a.d, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float *wf = reinterpret_cast<float *>(w4);
    pdl_wait();
    if (E == EMAX) {
        // one float4 of W_r (4 experts of one input row) lands in one float4 slot; 8 in flight
        const int n4 = d * EMAX / 4;
        const float4 *src = reinterpret_cast<const float4 *>(a.W_r);
        for (int q0 = tid; q0 < n4; q0 += 8 * RT_THREADS) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (q0 + u * RT_THREADS < n4) v[u] = __ldg(src + q0 + u * RT_THREADS);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int q = q0 + u * RT_THREADS;
                if (q < n4) {
                    const int i = q / V, vv = q % V;
                    const int j = i >> 8, l = (i >> 3) & 31, qq = i & 7;
                    w4[((j * 8 + qq) * V + vv) * 32 + l] = v[u];
                }
            }
        }
    } else {
        for (int q = tid; q < d * EMAX; q += RT_THREADS) {
            const int i = q / EMAX, e = q % EMAX;
            const int j = i >> 8, l = (i >> 3) & 31, qq = i & 7;
            wf[((((j * 8 + qq) * V + (e >> 2)) * 32 + l) << 2) + (e & 3)] =
                e < E ? a.W_r[(int64_t)i * E + e] : 0.f;
        }
    }
    __syncthreads();
    const Tin *h = reinterpret_cast<const Tin *>(a.h);
    const int nj = (d + 255) / 256;
    const int64_t t_begin = (int64_t)blockIdx.x * a.tokens_per_block;
    const int64_t t_end = min(a.T, t_begin + (int64_t)a.tokens_per_block);
    const int my_e = lane & (EMAX - 1);
    const float bias = (a.b_r && my_e < E) ? a.b_r[my_e] : 0.f;
    float sbv[1];
    sbv[0] = (a.sel_bias && my_e < E) ? a.sel_bias[my_e] : 0.f;
    float psum_lane = 0.f, lse2 = 0.f;
    // Each warp takes two tokens at a time: every W_r read from shared memory feeds both.
    for (int64_t t = t_begin + 2 * warp; t < t_end; t += 2 * SMALL_WARPS) {
        const bool two = t + 1 < t_end;
        float acc[2][EMAX];
#pragma unroll
        for (int e = 0; e < EMAX; ++e) acc[0][e] = acc[1][e] = 0.f;
        const Tin *hrow0 = h + t * d;
        const Tin *hrow1 = two ? hrow0 + d : hrow0;
        // software pipeline: the loads of slice j + 1 are in flight while slice j is computed
        // (two register buffers, the loop unrolled by two so that both stay in registers)
        float xa[2][8], xb[2][8];
        auto load_slice = [&](int j, float (&xx)[2][8]) {
            const int i0 = 256 * j + 8 * lane;
            if (j < nj && i0 < d) {
                load8(hrow0 + i0, xx[0]);
                load8(hrow1 + i0, xx[1]);
            }
        };
        auto fma_slice = [&](int j, const float (&xx)[2][8]) {
            if (j < nj && 256 * j + 8 * lane < d) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const float4 w = w4[((j * 8 + q) * V + v) * 32 + lane];
#pragma unroll
                        for (int tt = 0; tt < 2; ++tt) {
                            acc[tt][4 * v + 0] = fmaf(xx[tt][q], w.x, acc[tt][4 * v + 0]);
                            acc[tt][4 * v + 1] = fmaf(xx[tt][q], w.y, acc[tt][4 * v + 1]);
                            acc[tt][4 * v + 2] = fmaf(xx[tt][q], w.z, acc[tt][4 * v + 2]);
                            acc[tt][4 * v + 3] = fmaf(xx[tt][q], w.w, acc[tt][4 * v + 3]);
                        }
                    }
                }
            }
        };
        load_slice(0, xa);
        for (int j = 0; j < nj; j += 2) {
            load_slice(j + 1, xb);
            fma_slice(j, xa);
            load_slice(j + 2, xa);
            fma_slice(j + 1, xb);
        }
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
            if (tt == 1 && !two) break;  // warp-uniform
            float *av = acc[tt];
            // Fold the lanes: butterfly over the lane bits >= EMAX, then a reduce-scatter over
            // the lower bits; afterwards lane l holds logit (l & (EMAX - 1)).
#pragma unroll
            for (int o = 16; o >= EMAX; o >>= 1)
#pragma unroll
                for (int e = 0; e < EMAX; ++e) av[e] += __shfl_xor_sync(0xffffffffu, av[e], o);
#pragma unroll
            for (int o = EMAX / 2; o >= 1; o >>= 1) {
                const bool up = (lane & o) != 0;
#pragma unroll
                for (int m = 0; m < o; ++m) {
                    const float send = up ? av[m] : av[m + o];
                    const float keep = up ? av[m + o] : av[m];
                    av[m] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            float v[1];
            v[0] = (lane < EMAX && my_e < E) ? av[0] + bias : -INFINITY;
            float p[1], lse;
            route_token<1>(v, sbv, a.sel_bias != nullptr, E, a.k, a.gate_mode, t + tt, a.idx,
                           a.gates, p, lse);
            if (lane < E) psum_lane += p[0];
            lse2 += lse * lse;
        }
    }
    red[warp][lane] = psum_lane;
    __shared__ float red_lse[SMALL_WARPS];
    if (lane == 0) red_lse[warp] = lse2;
    __syncthreads();
    if (tid < E) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < SMALL_WARPS; ++w) s += red[w][tid];
        a.psum[(int64_t)blockIdx.x * (E + 1) + tid] = s;
    } else if (tid == E) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < SMALL_WARPS; ++w) s += red_lse[w];
        a.psum[(int64_t)blockIdx.x * (E + 1) + E] = s;
    }
    pdl_trigger();
}

// Few tokens: one token per block, the 8 warps take the 256-wide slices of d in turn and read
// W_r straight from L2 (it is shared by all blocks), so no block pays for staging W_r; the warps'
// partial logits meet in shared memory and warp 0 finishes the token. psum_part gets one row per
// token.
template <typename Tin, int EMAX>
__global__ void __launch_bounds__(RT_THREADS) router_splitd_kernel(RouterArgs a) {
    __shared__ float part[SMALL_WARPS][EMAX];
    const int E = a.E, d = a.d, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t = blockIdx.x;
    pdl_wait();
    const Tin *hrow = reinterpret_cast<const Tin *>(a.h) + t * d;
    const int nj = (d + 255) / 256;
    const bool vec = (E & 3) == 0;
    float acc[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) acc[e] = 0.f;
    for (int j = warp; j < nj; j += SMALL_WARPS) {
        const int i0 = 256 * j + 8 * lane;
        if (i0 >= d) continue;
        float x[8];
        load8(hrow + i0, x);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float *wrow = a.W_r + (int64_t)(i0 + q) * E;
            if (vec) {
#pragma unroll
                for (int v = 0; v < EMAX / 4; ++v) {
                    if (4 * v < E) {
                        const float4 w = __ldg(reinterpret_cast<const float4 *>(wrow) + v);
                        acc[4 * v + 0] = fmaf(x[q], w.x, acc[4 * v + 0]);
                        acc[4 * v + 1] = fmaf(x[q], w.y, acc[4 * v + 1]);
                        acc[4 * v + 2] = fmaf(x[q], w.z, acc[4 * v + 2]);
                        acc[4 * v + 3] = fmaf(x[q], w.w, acc[4 * v + 3]);
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < EMAX; ++e)
                    if (e < E) acc[e] = fmaf(x[q], __ldg(wrow + e), acc[e]);
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= EMAX; o >>= 1)
#pragma unroll
        for (int e = 0; e < EMAX; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
#pragma unroll
    for (int o = EMAX / 2; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int m = 0; m < o; ++m) {
            const float send = up ? acc[m] : acc[m + o];
            const float keep = up ? acc[m + o] : acc[m];
            acc[m] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    if (lane < EMAX) part[warp][lane] = acc[0];
    __syncthreads();
    if (warp == 0) {
        float z = 0.f;
        if (lane < EMAX) {
#pragma unroll
            for (int w = 0; w < SMALL_WARPS; ++w) z += part[w][lane];
        }
        float v[1], sbv[1];
        v[0] = (lane < EMAX && lane < E) ? z + (a.b_r ? a.b_r[lane] : 0.f) : -INFINITY;
        sbv[0] = (a.sel_bias && lane < E) ? a.sel_bias[lane] : 0.f;
        float p[1], lse;
        route_token<1>(v, sbv, a.sel_bias != nullptr, E, a.k, a.gate_mode, t, a.idx, a.gates, p,
                       lse);
        if (lane < E) a.psum[t * (E + 1) + lane] = p[0];
        if (lane == 0) a.psum[t * (E + 1) + E] = lse * lse;
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------------------------
// general shapes: tiled f32 contraction

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
__global__ void __launch_bounds__(RT_THREADS) router_tile_kernel(RouterArgs a) {
    extern __shared__ float sm[];
    pdl_wait();
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
    float *lse_s = zs + BT * E;           // [BT] squared log-sum-exp per token

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

    // one warp per token
    const int warp = tid >> 5, lane = tid & 31;
    constexpr int NW = RT_THREADS / 32;
    constexpr int MAXM = 8;  // E <= 256 -> at most 8 logits per lane
    float sbv[MAXM];
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
        const int e = lane + 32 * m;
        sbv[m] = (a.sel_bias && e < E) ? a.sel_bias[e] : 0.f;
    }
    for (int row = warp; row < BT; row += NW) {
        const int64_t tok = t0 + row;
        float *zr = zs + row * E;
        if (tok >= a.T) {
            for (int e = lane; e < E; e += 32) zr[e] = 0.f;
            if (lane == 0) lse_s[row] = 0.f;
            continue;
        }
        float v[MAXM];
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            const int e = lane + 32 * m;
            v[m] = e < E ? zr[e] : -INFINITY;
        }
        float p[MAXM], lse;
        route_token<MAXM>(v, sbv, a.sel_bias != nullptr, E, a.k, a.gate_mode, tok, a.idx,
                          a.gates, p, lse);
        __syncwarp();
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            const int e = lane + 32 * m;
            if (e < E) zr[e] = p[m];
        }
        if (lane == 0) lse_s[row] = lse * lse;
    }
    __syncthreads();
    for (int e = tid; e <= E; e += RT_THREADS) {
        float s = 0.f;
        if (e < E)
            for (int row = 0; row < BT; ++row) s += zs[row * E + e];
        else
            for (int row = 0; row < BT; ++row) s += lse_s[row];
        a.psum[(int64_t)blockIdx.x * (E + 1) + e] = s;
    }
    pdl_trigger();
}

template <typename K>
cudaError_t launch_k(K kern, const RouterArgs &a, int64_t blocks, size_t smem, cudaStream_t s) {
    if (smem > 48 * 1024) {
        cudaError_t err = set_max_dynamic_smem((const void *)kern, smem);
        if (err != cudaSuccess) return err;
    }
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(RT_THREADS), smem, s, 1, a);
}

// ---------------------------------------------------------------------------------------------
// selection after the tensor-core logits (router_tc.cu): warp per token

constexpr int SEL_WARPS = 16;

// Tokens per selection block: about two blocks per SM of a 148-SM part (a pure function of T,
// which fixes the rows of psum_part), whole multiples of the warps.
int select_tokens_per_block(int64_t T) {
    int64_t tpb = (T + 295) / 296;
    tpb = (tpb + SEL_WARPS - 1) / SEL_WARPS * SEL_WARPS;
    return (int)(tpb < SEL_WARPS ? SEL_WARPS : tpb);
}

// Lane's logits of token tok before the bias: the sum over the S K chunks of zpart[s][tok][e]
// (s = 0..S-1 in order), -inf for absent experts. With one chunk the loads are left in flight
// (nothing consumes them here), so a call for the next token overlaps the current one.
template <int MAXM>
__device__ __forceinline__ void load_logits(const float *__restrict__ zpart, int S, int Epad,
                                            int64_t T, int64_t tok, int E, float (&v)[MAXM]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
        const int e = lane + 32 * m;
        if (e >= E) {
            v[m] = -INFINITY;
        } else if (S == 1) {
            v[m] = __ldg(zpart + tok * Epad + e);
        } else {
            float z = 0.f;
            for (int s = 0; s < S; ++s) z += __ldg(zpart + ((int64_t)s * T + tok) * Epad + e);
            v[m] = z;
        }
    }
}

// Warp per token over this block's tokens (the next token's logits loaded while the current one
// is processed), then the block's sums of p per expert (per warp in token order, then over the
// warps in order).
template <int MAXM>
__global__ void __launch_bounds__(SEL_WARPS * 32)
    router_select_kernel(const float *__restrict__ zpart, int S, int Epad, int tpb,
                         const RouterArgs a) {
    __shared__ float wsum[SEL_WARPS][MAXM * 32];
    __shared__ float wlse[SEL_WARPS];
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E;
    const int64_t t0 = (int64_t)blockIdx.x * tpb;
    int64_t t_end = t0 + tpb;
    if (t_end > a.T) t_end = a.T;
    float bias[MAXM], sbv[MAXM], acc[MAXM], lse2 = 0.f;
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
        const int e = lane + 32 * m;
        bias[m] = (a.b_r && e < E) ? __ldg(a.b_r + e) : 0.f;
        sbv[m] = (a.sel_bias && e < E) ? __ldg(a.sel_bias + e) : 0.f;
        acc[m] = 0.f;
    }
    int64_t tok = t0 + warp;
    float v[MAXM];
    if (tok < t_end) load_logits<MAXM>(zpart, S, Epad, a.T, tok, E, v);
    while (tok < t_end) {
        const int64_t nxt = tok + SEL_WARPS;
        float vn[MAXM];
#pragma unroll
        for (int m = 0; m < MAXM; ++m) vn[m] = -INFINITY;
        if (nxt < t_end) load_logits<MAXM>(zpart, S, Epad, a.T, nxt, E, vn);
#pragma unroll
        for (int m = 0; m < MAXM; ++m) v[m] += bias[m];  // -inf stays -inf for absent experts
        float p[MAXM], lse;
        route_token<MAXM>(v, sbv, a.sel_bias != nullptr, E, a.k, a.gate_mode, tok, a.idx,
                          a.gates, p, lse);
        lse2 += lse * lse;
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            if (lane + 32 * m < E) acc[m] += p[m];
            v[m] = vn[m];
        }
        tok = nxt;
    }
#pragma unroll
    for (int m = 0; m < MAXM; ++m) wsum[warp][lane + 32 * m] = acc[m];
    if (lane == 0) wlse[warp] = lse2;
    __syncthreads();
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        float s = 0.f;
        for (int w = 0; w < SEL_WARPS; ++w) s += e < E ? wsum[w][e] : wlse[w];
        a.psum[(int64_t)blockIdx.x * (E + 1) + e] = s;
    }
    pdl_trigger();
}

enum RouterPath { PATH_SPLITD, PATH_SMALL, PATH_TC, PATH_TILE };

RouterPath router_path(const moe_config_t &c) {
    // few tokens: every block reads all of W_r from L2; keep that traffic within 64 MiB
    if (c.E <= 32 && c.T <= 1024 &&
        (double)c.T * c.d * small_emax(c.E) * 4 <= 64.0 * 1024 * 1024)
        return PATH_SPLITD;
    // bf16 with many tokens: the tensor cores (exact three-piece split of W_r)
    if (c.dtype == MOE_BF16 && c.E <= ROUTER_TC_MAX_E) return PATH_TC;
    if (c.E <= 32 && (size_t)((c.d + 255) / 256) * 256 * small_emax(c.E) * 4 <= SMALL_SMEM_MAX)
        return PATH_SMALL;
    return PATH_TILE;
}

// Tokens per block of the small kernel: about one block per SM, two tokens per warp at least.
int small_tokens_per_block(int64_t T) {
    int64_t tpb = (T + 147) / 148;
    tpb = (tpb + 2 * SMALL_WARPS - 1) / (2 * SMALL_WARPS) * (2 * SMALL_WARPS);
    return (int)(tpb < 2 * SMALL_WARPS ? 2 * SMALL_WARPS : tpb);
}

}  // namespace

int64_t router_partial_rows(const moe_config_t &c) {
    switch (router_path(c)) {
        case PATH_SPLITD: return c.T;
        case PATH_SMALL: {
            const int tpb = small_tokens_per_block(c.T);
            return (c.T + tpb - 1) / tpb;
        }
        case PATH_TC: {
            const int tpb = select_tokens_per_block(c.T);
            return (c.T + tpb - 1) / tpb;
        }
        default: {
            const int bt = geometry(c.E).BT;
            return (c.T + bt - 1) / bt;
        }
    }
}

size_t router_scratch_bytes(const moe_config_t &c) {
    return router_path(c) == PATH_TC ? router_tc_scratch_bytes(c) : 0;
}

int router_launches(const moe_config_t &c) { return router_path(c) == PATH_TC ? 3 : 1; }

cudaError_t launch_router_topk(const moe_config_t &c, const void *h, const float *W_r,
                               const float *b_r, const float *sel_bias, int32_t *topk_idx,
                               float *gates, float *psum_part, void *scratch,
                               uint32_t *dev_status, cudaStream_t s) {
    if (c.T == 0) return cudaSuccess;
    RouterArgs a{h, W_r, b_r, sel_bias, topk_idx, gates, psum_part, c.T, c.d, c.E, c.k, c.gate, 0};
    const RouterPath path = router_path(c);
    if (path == PATH_TC) {
        cudaError_t err = launch_router_tc(c, h, W_r, scratch, dev_status, s);
        if (err != cudaSuccess) return err;
        const float *zpart = router_tc_logits(scratch, c);
        const int S = router_tc_splits(c), Epad = router_tc_epad(c);
        const int tpb = select_tokens_per_block(c.T);
        const unsigned blocks = (unsigned)((c.T + tpb - 1) / tpb);
        const dim3 grid(blocks), thr(SEL_WARPS * 32);
        switch ((c.E + 31) / 32) {
            case 1: return launch_pdl(router_select_kernel<1>, grid, thr, 0, s, 1, zpart, S, Epad, tpb, a);
            case 2: return launch_pdl(router_select_kernel<2>, grid, thr, 0, s, 1, zpart, S, Epad, tpb, a);
            case 3: return launch_pdl(router_select_kernel<3>, grid, thr, 0, s, 1, zpart, S, Epad, tpb, a);
            default: return launch_pdl(router_select_kernel<4>, grid, thr, 0, s, 1, zpart, S, Epad, tpb, a);
        }
    }
    const bool bf16 = c.dtype == MOE_BF16;
    if (path == PATH_SPLITD) {
        switch (small_emax(c.E)) {
            case 8:
                return bf16 ? launch_k(router_splitd_kernel<__nv_bfloat16, 8>, a, c.T, 0, s)
                            : launch_k(router_splitd_kernel<float, 8>, a, c.T, 0, s);
            case 16:
                return bf16 ? launch_k(router_splitd_kernel<__nv_bfloat16, 16>, a, c.T, 0, s)
                            : launch_k(router_splitd_kernel<float, 16>, a, c.T, 0, s);
            default:
                return bf16 ? launch_k(router_splitd_kernel<__nv_bfloat16, 32>, a, c.T, 0, s)
                            : launch_k(router_splitd_kernel<float, 32>, a, c.T, 0, s);
        }
    }
    if (path == PATH_SMALL) {
        a.tokens_per_block = small_tokens_per_block(c.T);
        const int emax = small_emax(c.E);
        const size_t smem = (size_t)((c.d + 255) / 256) * 256 * emax * 4;
        const int64_t blocks = (c.T + a.tokens_per_block - 1) / a.tokens_per_block;
        switch (emax) {
            case 8:
                return bf16 ? launch_k(router_small_kernel<__nv_bfloat16, 8>, a, blocks, smem, s)
                            : launch_k(router_small_kernel<float, 8>, a, blocks, smem, s);
            case 16:
                return bf16 ? launch_k(router_small_kernel<__nv_bfloat16, 16>, a, blocks, smem, s)
                            : launch_k(router_small_kernel<float, 16>, a, blocks, smem, s);
            default:
                return bf16 ? launch_k(router_small_kernel<__nv_bfloat16, 32>, a, blocks, smem, s)
                            : launch_k(router_small_kernel<float, 32>, a, blocks, smem, s);
        }
    }
    const Geo g = geometry(c.E);
    const int64_t blocks = (c.T + g.BT - 1) / g.BT;
    const size_t stage = sizeof(float) * ((size_t)g.BT * (DK + 1) + (size_t)DK * c.E);
    const size_t logits = sizeof(float) * (size_t)g.BT * (c.E + 1);
    const size_t smem = stage > logits ? stage : logits;
    const bool wide = g.RE == 4;
    if (bf16)
        return wide ? launch_k(router_tile_kernel<8, 4, __nv_bfloat16>, a, blocks, smem, s)
                    : launch_k(router_tile_kernel<1, 1, __nv_bfloat16>, a, blocks, smem, s);
    return wide ? launch_k(router_tile_kernel<8, 4, float>, a, blocks, smem, s)
                : launch_k(router_tile_kernel<1, 1, float>, a, blocks, smem, s);
}

}  // namespace moe
