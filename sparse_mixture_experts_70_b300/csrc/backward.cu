// backward.cu -- the backward pass of the MoE layer (bf16 layers, tensor-core GEMMs).
//
// The pages: selecting the top-k experts is not differentiable, so the gradient reaches the
// router only through the weights of the chosen experts -- for Switch top-1 through the router
// probability p_i (llm.curionode.com "Mixture of Experts.", opening text; lensaml.com "Mixture of
// Experts", Step 3 "Top-k Routing"); of the auxiliary term only P_i is differentiable (Step 4
// "Load Balancing"); the router trains by ordinary backpropagation (arjunjaggi.com "Mixture of
// Experts in LLMs", "How Routing Works"). So idx, the routed counts and the capacity drops of the
// forward are constants here, and the loss differentiated is
//     L = sum dy * y + aux_weight * (E sum_e f_e P_e) + zloss_weight * zloss.
//
// With X the permuted rows of h, a slot r of expert e with gate g_r, and dYu[r] = dy[token(r)]:
//   A1 = X W1_e^T (+ b1), A3 = X W3_e^T     saved by the training forward, or recomputed (two
//                                           row-grouped GEMMs)
//   dHu = dYu W2_e                           row-grouped GEMM
//   SwiGLU: Hact = SiLU(A1) A3, dA1 = g dHu A3 SiLU'(A1), dA3 = g dHu SiLU(A1)
//   GELU  : Hact = GELU(A1),    dA1 = g dHu GELU'(A1)
//   dg_r = dHu . Hact (+ dy . b2_e)          gradient of the slot's gate
//   dX = dA1 W1_e + dA3 W3_e                  one row-grouped GEMM over K = [dA1 | dA3]
//   dW2_e = dYu^T (g Hact), dW1_e = dA1^T X, dW3_e = dA3^T X   K-grouped GEMMs over the slots
//   db2_e = sum_r g_r dYu[r], db1_e = sum_r dA1[r]
//   router: dz from dg through the gate softmax (RENORM) or p (RAW_PROB), plus the auxiliary
//           term and the z-loss; dh = sum_j dX[slot] + dz W_r^T, dW_r = h^T dz, db_r = sum dz.
// Layout: the per-slot tensors of the backward (rows of h and dy, dHu, dA, g Hact, dX) live in a
// padded row layout, expert e's slots at rows [kseg[e], kseg[e+1]) with kseg[e+1] - kseg[e] =
// roundup64(count_e) and zero pad rows. Every GEMM reads its operands in their stored layouts:
// the data-gradient GEMMs take W2, W1 and W3 as MN-major B operands, and the weight-gradient
// GEMMs, which contract over each expert's slots (the rows), take both operands MN-major in
// 64-row K blocks that never straddle two experts. The router's two contractions (dz W_r^T,
// h^T dz) run on the tensor cores with dz and W_r split into hi + lo bf16 pieces. f32 layers take
// the same steps with every product on the CUDA cores (gemm_f32_kernel).
#include <nvtx3/nvToolsExt.h>

#include <type_traits>

#include "internal.cuh"
#include "moe_backward.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int BT = 64;  // rows per padded segment block and tile edge of the element-wise kernels

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ void unpack8(const uint4 u, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
        v[2 * i] = __low2float(p);
        v[2 * i + 1] = __high2float(p);
    }
}

// 8 consecutive elements of a bf16 or f32 row (16-byte aligned) as f32, and back.
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
    unpack8(__ldg(reinterpret_cast<const uint4 *>(p)), v);
}
__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float (&v)[8]) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]),
                                               pack2(v[4], v[5]), pack2(v[6], v[7]));
}
__device__ __forceinline__ void store8(float *p, const float (&v)[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
// 8 elements in their stored form (16 bytes of bf16, 32 of f32): loaded ahead of their use, so
// that a thread has all its loads in flight before it computes.
template <typename Elt>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
        u = __ldg(reinterpret_cast<const uint4 *>(p));
    }
    __device__ __forceinline__ void get(float (&v)[8]) const { unpack8(u, v); }
};
template <>
struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float *p) {
        a = __ldg(reinterpret_cast<const float4 *>(p));
        b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    }
    __device__ __forceinline__ void get(float (&v)[8]) const {
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f(float v) { return v; }

// The expert whose padded segment holds padded row c (kseg in shared memory, E+1 entries).
__device__ __forceinline__ int segment_of(const int32_t *kseg, int E, int c) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (kseg[mid] <= c) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ---------------------------------------------------------------------------------------------
// prep: gate of every sorted row (gate_r[slot_of[s]] = gates[s] for kept slots), and in block 0
// the padded segment offsets kseg and the router GEMMs' one-group segments seg.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const int32_t *slot_of, const float *gates,
                                                       const int32_t *offsets, int64_t P, int E,
                                                       int64_t T, int nsplit, float *gate_r,
                                                       int32_t *kseg, int32_t *seg,
                                                       uint32_t *dev_status) {
    pdl_wait();
    const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int rows = offsets[E];
    if (s < P) {
        const int r = slot_of[s];
        if (r >= rows || (int64_t)r >= P) report(dev_status, DEV_ERR_INDEX);
        else if (r >= 0) gate_r[r] = gates[s];
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        // segments of the router GEMMs: rows [0, T) as one group for dz W_r^T, and the K range
        // [0, roundup64(T)) of h^T dz cut into nsplit groups of whole 64-row blocks
        seg[0] = 0;
        seg[1] = (int32_t)T;
        const int64_t blocks = (T + BT - 1) / BT;
        for (int g = 0; g <= nsplit; ++g) seg[2 + g] = (int32_t)(blocks * g / nsplit * BT);
        int acc = 0;
        kseg[0] = 0;
        for (int e = 0; e < E; ++e) {
            const int cnt = offsets[e + 1] - offsets[e];
            acc += (cnt + BT - 1) / BT * BT;
            kseg[e + 1] = acc;
        }
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------------------------
// Padded-row gathers: for padded row c = kseg[e] + l of expert e, when l < count_e (sorted row
// r = offsets[e] + l, token t = sorted_token[r]): Xp[c] = h[t] and dYp[c] = dy[t]; pad rows are
// zero. When db2_part is given, db2_part[tile][o] is the tile's sum of gate_r[r] dy[t, o].
// Block (x, y): the 64 rows of tile x, columns [2048 y, 2048 y + 2048), 8 per thread.
constexpr int GP_COLS = 2048;
template <typename Elt>
__global__ void __launch_bounds__(256) gather_pad_kernel(const Elt *h, const Elt *dy,
                                                         const int32_t *sorted_token,
                                                         const int32_t *offsets,
                                                         const int32_t *kseg_g,
                                                         const float *gate_r, int E, int64_t T,
                                                         int64_t P, int d, Elt *Xp, Elt *dYp,
                                                         float *db2_part, uint32_t *dev_status) {
    __shared__ int32_t kseg[257];
    __shared__ int32_t tok[BT];
    __shared__ float scl[BT];
    pdl_wait();
    for (int e = threadIdx.x; e <= E; e += blockDim.x) kseg[e] = kseg_g[e];
    __syncthreads();
    const int c0 = blockIdx.x * BT;
    if (c0 >= kseg[E]) {
        pdl_trigger();
        return;
    }
    const int e = segment_of(kseg, E, c0);
    const int cnt = offsets[e + 1] - offsets[e];
    const int local0 = c0 - kseg[e];
    if (threadIdx.x < BT) {
        const int l = local0 + threadIdx.x;
        const int r = offsets[e] + l;
        int t = -1;
        float sc = 0.f;
        if (l < cnt && (r < 0 || (int64_t)r >= P)) report(dev_status, DEV_ERR_INDEX);
        if (l < cnt && r >= 0 && (int64_t)r < P) {
            t = sorted_token[r];
            if (t < 0 || t >= T) {
                report(dev_status, DEV_ERR_INDEX);
                t = -1;
            } else {
                sc = gate_r[r];
            }
        }
        tok[threadIdx.x] = t;
        scl[threadIdx.x] = sc;
    }
    __syncthreads();
    const int col = blockIdx.y * GP_COLS + threadIdx.x * 8;
    if (col < d) {
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.f;
#pragma unroll 4
        for (int jr = 0; jr < BT; ++jr) {
            const int t = tok[jr];
            float hv[8], dv[8];
            if (t >= 0) {
                load8(h + (int64_t)t * d + col, hv);
                load8(dy + (int64_t)t * d + col, dv);
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) hv[q] = dv[q] = 0.f;
            }
            const int64_t o = (int64_t)(c0 + jr) * d + col;
            store8(Xp + o, hv);
            store8(dYp + o, dv);
            if (db2_part) {
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = fmaf(scl[jr], dv[q], acc[q]);
            }
        }
        if (db2_part) {
#pragma unroll
            for (int q = 0; q < 8; ++q) db2_part[(int64_t)blockIdx.x * d + col + q] = acc[q];
        }
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------------------------
// Activation backward on one 64-row x 64-feature tile: padded rows [c0, c0 + 64) of one expert
// (blockIdx.x), features [n0, n0 + 64) (blockIdx.y). Reads the pre-activations A1 (and A3) of
// sorted row r = offsets[e] + l, dHu of padded row c = kseg[e] + l, and the row's gate g; writes
// padded rows of dA [kw, K2] (dA1 in columns [0, f), dA3 in [f, 2f) for SwiGLU) and of
// Hs = g Hact [kw, f] (pad rows zero), dg_part[n-tile][r] = the tile's part of dHu . Hact, and
// (when db1_part is given) the tile's column sums of dA1.
template <typename Elt>
struct ActBwd {
    const Elt *A1, *A3, *dHu;
    const float *gate_r;
    const int32_t *offsets, *kseg;
    Elt *dA, *Hs;
    float *dg_part;   // [f/64, P]
    float *db1_part;  // [kw/64, f] or null
    int64_t P;
    int E, f, swiglu;
};

// FAST: the special-function unit's tanh and exp (the forward's GELU and SiLU use the same), for
// bf16 layers; f32 layers keep the accurate library functions.
template <bool FAST>
__device__ __forceinline__ float gelu_tanh_acc(float x, float &slope) {
    const float c = 0.7978845608028654f;
    const float u = c * (x + 0.044715f * x * x * x);
    const float th = FAST ? tc::tanh_approx(u) : tanhf(u);
    slope = 0.5f * (1.f + th) + 0.5f * x * (1.f - th * th) * c * (1.f + 3.f * 0.044715f * x * x);
    return 0.5f * x * (1.f + th);
}

template <typename Elt>
__global__ void __launch_bounds__(256) act_bwd_kernel(const ActBwd<Elt> a, uint32_t *dev_status) {
    __shared__ float s1[BT][BT + 1];  // dA1 (f32) for the bias sums
    __shared__ int32_t kseg[257];
    pdl_wait();
    for (int e = threadIdx.x; e <= a.E; e += blockDim.x) kseg[e] = a.kseg[e];
    __syncthreads();
    // block b: padded rows [64 (b / (f/64)), +64), features [64 (b % (f/64)), +64) -- the
    // feature block runs fastest, so the blocks resident at one time cover whole rows (runs of
    // contiguous memory) rather than a 128-byte piece of every row
    const int ncb = a.f / BT;
    const int rb = (int)(blockIdx.x / (unsigned)ncb), cb = (int)(blockIdx.x % (unsigned)ncb);
    const int c0 = rb * BT;
    if (c0 >= kseg[a.E]) {
        pdl_trigger();
        return;
    }
    const int e = segment_of(kseg, a.E, c0);
    const int rbase = a.offsets[e] + (c0 - kseg[e]);  // sorted row of padded row c0
    const int rend = a.offsets[e + 1];
    if (rend > a.P || rbase < 0) {
        report(dev_status, DEV_ERR_INDEX);
        pdl_trigger();
        return;
    }
    const int n0 = cb * BT;
    const int K2 = a.swiglu ? 2 * a.f : a.f;
    // every thread first issues the loads of its IT vectors of 8, then computes them
    constexpr int IT = BT * (BT / 8) / 256;
    static_assert(BT * (BT / 8) % 256 == 0, "the block's vectors of 8 split evenly");
    Raw8<Elt> ra1[IT], ra3[IT], rdu[IT];
    float gv[IT];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int i = (int)threadIdx.x + it * 256;
        const int jr = i >> 3, ch = i & 7;
        const int r = rbase + jr;
        if (r < rend) {
            const int64_t off = (int64_t)r * a.f + n0 + ch * 8;
            ra1[it].load(a.A1 + off);
            rdu[it].load(a.dHu + (int64_t)(c0 + jr) * a.f + n0 + ch * 8);
            if (a.swiglu) ra3[it].load(a.A3 + off);
            gv[it] = a.gate_r[r];
        }
    }
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int i = (int)threadIdx.x + it * 256;
        const int jr = i >> 3, ch = i & 7;
        const int r = rbase + jr;
        const bool valid = r < rend;
        float d1[8], d3[8], hs[8];
        float dg = 0.f;
        if (valid) {
            float x1[8], x3[8], du[8];
            ra1[it].get(x1);
            rdu[it].get(du);
            if (a.swiglu) ra3[it].get(x3);
            const float g = gv[it];
            constexpr bool FAST = !std::is_same<Elt, float>::value;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float hv;
                if (a.swiglu) {
                    const float sg = FAST ? __fdividef(1.f, 1.f + __expf(-x1[q]))
                                          : 1.f / (1.f + expf(-x1[q]));
                    const float si = x1[q] * sg;
                    hv = si * x3[q];
                    d1[q] = g * du[q] * x3[q] * sg * (1.f + x1[q] * (1.f - sg));
                    d3[q] = g * du[q] * si;
                } else {
                    float slope;
                    hv = gelu_tanh_acc<FAST>(x1[q], slope);
                    d1[q] = g * du[q] * slope;
                    d3[q] = 0.f;
                }
                hs[q] = g * hv;
                dg += du[q] * hv;
            }
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) d1[q] = d3[q] = hs[q] = 0.f;
        }
        Elt *row = a.dA + (int64_t)(c0 + jr) * K2 + n0 + ch * 8;
        store8(row, d1);
        if (a.swiglu) store8(row + a.f, d3);
        store8(a.Hs + (int64_t)(c0 + jr) * a.f + n0 + ch * 8, hs);
        if (a.db1_part) {
#pragma unroll
            for (int q = 0; q < 8; ++q) s1[jr][ch * 8 + q] = d1[q];
        }
        // the row's 8 feature groups are 8 consecutive lanes: sum them in a fixed order
        dg += __shfl_xor_sync(0xffffffffu, dg, 1);
        dg += __shfl_xor_sync(0xffffffffu, dg, 2);
        dg += __shfl_xor_sync(0xffffffffu, dg, 4);
        if (valid && ch == 0) a.dg_part[(int64_t)cb * a.P + r] = dg;
    }
    if (a.db1_part) {
        __syncthreads();
        if (threadIdx.x < BT) {
            float sum = 0.f;
            for (int jr = 0; jr < BT; ++jr) sum += s1[jr][threadIdx.x];
            a.db1_part[(int64_t)rb * a.f + n0 + threadIdx.x] = sum;
        }
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------------------------
// Router logits z[t, e] = h[t] . W_r[:, e] (no bias) for layers whose forward router is not the
// tensor-core one (few tokens, or f32): one block per token (striding over the tokens), its 8
// warps splitting d; experts 8 at a time, each thread's 8 partial dots summed over its warp by
// shuffles and then over the warps in order.
template <typename Elt>
__global__ void __launch_bounds__(256) router_logits_direct_kernel(const Elt *h, const float *W_r,
                                                                   int64_t T, int d, int E,
                                                                   float *z) {
    __shared__ float wpart[8][8];
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        const Elt *ht = h + t * d;
        for (int e0 = 0; e0 < E; e0 += 8) {
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.f;
            for (int i = threadIdx.x; i < d; i += blockDim.x) {
                const float hv = to_f(ht[i]);
                const float *wr = W_r + (int64_t)i * E + e0;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (e0 + q < E) acc[q] = fmaf(hv, __ldg(wr + q), acc[q]);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float v = acc[q];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0) wpart[warp][q] = v;
            }
            __syncthreads();
            if (threadIdx.x < 8 && e0 + (int)threadIdx.x < E) {
                float v = 0.f;
                for (int w = 0; w < 8; ++w) v += wpart[w][threadIdx.x];
                z[t * E + e0 + threadIdx.x] = v;
            }
            __syncthreads();
        }
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------------------------
// Router backward, one warp per token: the logits z (summed over the partial logits
// part[S][T][ldp]: the tensor-core router's K chunks, or S = 1 from router_logits_direct_kernel),
// p, lse, the gate gradients dg_j of the k slots
// (the tiles' parts summed, plus dy . b2_e when b2 is given), then dz = dL/dz. dz leaves as bf16
// pieces for the two router GEMMs: Zp[t] = [hi(dz) | lo(dz) | hi(dz) | 0 ...] (Kp columns), with
// hi = bf16(dz) and lo = bf16(dz - hi), so that dz W_r^T ~ hi Whi + lo Whi + hi Wlo and
// h^T dz ~ h^T hi + h^T lo hold to about 2^-16; the per-block sums of dz (db_r) go to dbr_part.
constexpr int RB_MAXEW = 8;  // experts per lane: E <= 256
template <typename Elt>
struct RouterBwd {
    const Elt *h, *dy;
    const float *W_r, *b_r, *b2;
    const float *part;  // partial logits [S][T][ldp]
    int S, ldp;
    const int32_t *topk_idx, *slot_of, *counts;
    const float *gates, *dg_part;
    int n_part;         // f / 64 partial rows of dg
    int64_t T, P;
    int d, E, k, raw_prob;
    float aux_weight, zloss_weight;
    __nv_bfloat16 *Zp;  // [T, Kp] bf16 pieces (bf16 layers), or
    float *dz;          // [T, E] f32 (f32 layers)
    int Kp;
    float *dbr_part;    // [gridDim.x, E]
};

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// dz of token t into this lane's experts lane + 32 i.
template <typename Elt>
__device__ __forceinline__ void router_token_grad(const RouterBwd<Elt> &a, int64_t t, int lane,
                                                  float (&dz)[RB_MAXEW], uint32_t *dev_status) {
    const int E = a.E;
    float z[RB_MAXEW], p[RB_MAXEW];
#pragma unroll
    for (int i = 0; i < RB_MAXEW; ++i) z[i] = 0.f;
    {
#pragma unroll
        for (int i = 0; i < RB_MAXEW; ++i) {
            const int e = lane + 32 * i;
            if (e < E)
                for (int s = 0; s < a.S; ++s) z[i] += a.part[((int64_t)s * a.T + t) * a.ldp + e];
        }
    }
    float zmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < RB_MAXEW; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            if (a.b_r) z[i] += a.b_r[e];
            zmax = fmaxf(zmax, z[i]);
        }
    }
    zmax = warp_max_f(zmax);
    float se = 0.f;
#pragma unroll
    for (int i = 0; i < RB_MAXEW; ++i) {
        const int e = lane + 32 * i;
        p[i] = e < E ? expf(z[i] - zmax) : 0.f;
        se += p[i];
    }
    se = warp_sum_f(se);
    const float lse = zmax + logf(se);
#pragma unroll
    for (int i = 0; i < RB_MAXEW; ++i) {
        p[i] /= se;
        dz[i] = 0.f;
    }
    // gate gradients: the warp sums slot j's partial rows (and its bias term) in a fixed order
    float dg_mine = 0.f;  // lane j < k keeps dg_j
    int e_mine = 0;
    float g_mine = 0.f;
    for (int j = 0; j < a.k; ++j) {
        const int64_t sidx = t * a.k + j;
        const int r = a.slot_of[sidx];
        const int ej = a.topk_idx[sidx];
        if (ej < 0 || ej >= E || r >= a.P) report(dev_status, DEV_ERR_INDEX);
        float v = 0.f;
        if (r >= 0 && r < a.P && ej >= 0 && ej < E) {
            for (int q = lane; q < a.n_part; q += 32) v += a.dg_part[(int64_t)q * a.P + r];
            if (a.b2) {
                const Elt *dyt = a.dy + t * a.d;
                const float *b2e = a.b2 + (int64_t)ej * a.d;
                for (int o = lane; o < a.d; o += 32) v = fmaf(to_f(dyt[o]), b2e[o], v);
            }
        }
        v = warp_sum_f(v);
        if (lane == j) {
            dg_mine = v;
            e_mine = ej < 0 || ej >= E ? 0 : ej;
            g_mine = a.gates[sidx];
        }
    }
    // the probability p[e_j] of every slot's expert, gathered from its owner lane
    float pj = 0.f;
    for (int j = 0; j < a.k; ++j) {
        const int ej = __shfl_sync(0xffffffffu, e_mine, j);
        float pe = 0.f;
#pragma unroll
        for (int i = 0; i < RB_MAXEW; ++i)
            if (ej == lane + 32 * i) pe = p[i];
        pe = warp_sum_f(pe);
        if (lane == j) pj = pe;
    }
    const bool has = lane < a.k;
    float add_j;  // dz contribution of slot j at its own expert
    if (a.raw_prob) {
        const float S = warp_sum_f(has ? dg_mine * pj : 0.f);
#pragma unroll
        for (int i = 0; i < RB_MAXEW; ++i) dz[i] = -p[i] * S;
        add_j = dg_mine * pj;
    } else {
        const float S = warp_sum_f(has ? g_mine * dg_mine : 0.f);
        add_j = g_mine * (dg_mine - S);
    }
    for (int j = 0; j < a.k; ++j) {
        const int ej = __shfl_sync(0xffffffffu, e_mine, j);
        const float v = __shfl_sync(0xffffffffu, add_j, j);
#pragma unroll
        for (int i = 0; i < RB_MAXEW; ++i)
            if (ej == lane + 32 * i) dz[i] += v;
    }
    if (a.aux_weight != 0.f) {
        // dL/dp[t, e] = aux_weight E f_e / T with f_e = counts[e] / (T k)
        const float scale = a.aux_weight * (float)E / ((float)a.T * (float)a.T * (float)a.k);
        float c[RB_MAXEW];
        float sdot = 0.f;
#pragma unroll
        for (int i = 0; i < RB_MAXEW; ++i) {
            const int e = lane + 32 * i;
            c[i] = e < E ? scale * (float)a.counts[e] : 0.f;
            sdot += c[i] * p[i];
        }
        sdot = warp_sum_f(sdot);
#pragma unroll
        for (int i = 0; i < RB_MAXEW; ++i) dz[i] += p[i] * (c[i] - sdot);
    }
    if (a.zloss_weight != 0.f) {
        const float zs = a.zloss_weight * 2.f / (float)a.T * lse;
#pragma unroll
        for (int i = 0; i < RB_MAXEW; ++i) dz[i] += zs * p[i];
    }
}

// Warps stride over the tokens; each block sums dz over its tokens (per warp in token order,
// then over the warps in order) into dbr_part[blockIdx.x].
template <typename Elt>
__global__ void __launch_bounds__(256) router_bwd_kernel(const RouterBwd<Elt> a,
                                                         uint32_t *dev_status) {
    __shared__ float wsum[8][256];
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int E = a.E;
    float acc[RB_MAXEW];
#pragma unroll
    for (int i = 0; i < RB_MAXEW; ++i) acc[i] = 0.f;
    for (int64_t t = (int64_t)blockIdx.x * 8 + warp; t < a.T; t += (int64_t)gridDim.x * 8) {
        float dz[RB_MAXEW];
        router_token_grad(a, t, lane, dz, dev_status);
        if (a.dz) {
#pragma unroll
            for (int i = 0; i < RB_MAXEW; ++i) {
                const int e = lane + 32 * i;
                if (e < E) {
                    a.dz[t * E + e] = dz[i];
                    acc[i] += dz[i];
                }
            }
            continue;
        }
        __nv_bfloat16 *zp = a.Zp + t * a.Kp;
#pragma unroll
        for (int i = 0; i < RB_MAXEW; ++i) {
            const int e = lane + 32 * i;
            if (e < E) {
                const __nv_bfloat16 hi = __float2bfloat16_rn(dz[i]);
                const __nv_bfloat16 lo = __float2bfloat16_rn(dz[i] - __bfloat162float(hi));
                zp[e] = hi;
                zp[E + e] = lo;
                zp[2 * E + e] = hi;
                acc[i] += dz[i];
            }
        }
        for (int c = 3 * E + lane; c < a.Kp; c += 32) zp[c] = __float2bfloat16_rn(0.f);
    }
#pragma unroll
    for (int i = 0; i < RB_MAXEW; ++i) {
        const int e = lane + 32 * i;
        if (e < E) wsum[warp][e] = acc[i];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float v = 0.f;
        for (int w = 0; w < 8; ++w) v += wsum[w][e];
        a.dbr_part[(int64_t)blockIdx.x * E + e] = v;
    }
    pdl_trigger();
}

// Wp[i] = [hi(W_r[i, :]) | hi(W_r[i, :]) | lo(W_r[i, :]) | 0 ...] (Kp columns): the router weight
// as bf16 pieces matching Zp, for dz W_r^T on the tensor cores.
__global__ void __launch_bounds__(256) wr_pieces_kernel(const float *W_r, int d, int E, int Kp,
                                                        __nv_bfloat16 *Wp) {
    pdl_wait();
    const int64_t n = (int64_t)d * Kp;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n;
         x += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = x / Kp;
        const int c = (int)(x - i * Kp);
        float v = 0.f;
        if (c < 3 * E) {
            const int e = c % E;
            const float w = W_r[i * E + e];
            const float hi = __bfloat162float(__float2bfloat16_rn(w));
            v = c < 2 * E ? hi : w - hi;
        }
        Wp[x] = __float2bfloat16_rn(v);
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------------------------
// dh[t, i] = dhr[t, i] + sum_j dX[c(t, j), i]: the router's term dz W_r^T (f32, from the tensor
// cores) plus the k slots' input gradients, where c(t, j) = kseg[e] + slot_of[t k + j] -
// offsets[e] with e = idx[t k + j] is the slot's padded row (dropped slots contribute nothing).
// One thread per 8 features of a token.
template <typename Elt, int G>
__global__ void __launch_bounds__(256) dh_kernel(const Elt *dX, const float *dhr,
                                                 const int32_t *slot_of, const int32_t *idx,
                                                 const int32_t *offsets_g, const int32_t *kseg_g,
                                                 int64_t T, int d, int E, int k, Elt *dh,
                                                 uint32_t *dev_status) {
    __shared__ int32_t kseg[257], offs[257];
    pdl_wait();
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        kseg[e] = kseg_g[e];
        offs[e] = offsets_g[e];
    }
    __syncthreads();
    const int vecs = d / 8;
    const int64_t n = T * vecs;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n;
         x += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = x / vecs;
        const int i0 = (int)(x - t * vecs) * 8;
        const float4 r0 = *reinterpret_cast<const float4 *>(dhr + t * d + i0);
        const float4 r1 = *reinterpret_cast<const float4 *>(dhr + t * d + i0 + 4);
        float acc[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        // slots in groups of G: the group's padded rows, then its dX loads, then the sums in
        // slot order (G = 1 for top-1 layers, where grouping only costs registers)
        for (int j0 = 0; j0 < k; j0 += G) {
            int cr[G];
#pragma unroll
            for (int u = 0; u < G; ++u) {
                const int j = j0 + u;
                cr[u] = -1;
                if (j >= k) continue;
                const int r = slot_of[t * k + j];
                if (r < 0) continue;  // dropped by the capacity
                const int e = idx[t * k + j];
                const int c = (e >= 0 && e < E) ? kseg[e] + (r - offs[e]) : -1;
                if (e < 0 || e >= E || r < offs[e] || c >= kseg[e + 1]) {
                    report(dev_status, DEV_ERR_INDEX);
                    continue;
                }
                cr[u] = c;
            }
            Raw8<Elt> raw[G];
#pragma unroll
            for (int u = 0; u < G; ++u)
                if (cr[u] >= 0) raw[u].load(dX + (int64_t)cr[u] * d + i0);
#pragma unroll
            for (int u = 0; u < G; ++u) {
                if (cr[u] < 0) continue;
                float v[8];
                raw[u].get(v);
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] += v[q];
            }
        }
        store8(dh + t * d + i0, acc);
    }
    pdl_trigger();
}

// dW_r[i, e] = sum over the K groups g of o[g][i, e] + o[g][i, E + e], from the GEMM
// h^T [hi | lo] split into nsplit groups of rows (o [nsplit, d, ldo] f32, summed in group order);
// db_r[e] = the sum of the router blocks' dz sums (when db_r is given): warp e of the blocks past
// the dW_r threads strides over the blocks' sums and adds its lanes in a fixed order.
__global__ void __launch_bounds__(256) router_final_kernel(const float *o, int ldo, int d, int E,
                                                           int nsplit, const float *dbr_part,
                                                           int nblk, float *dW_r, float *db_r) {
    // o == nullptr: dW_r is already final (f32 layers), only db_r is reduced
    pdl_wait();
    const int64_t n = (int64_t)d * E;
    const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (o && x < n) {
        const int64_t i = x / E;
        const int e = (int)(x - i * E);
        float v = 0.f;
        for (int g = 0; g < nsplit; ++g) {
            const float *og = o + ((int64_t)g * d + i) * ldo;
            v += og[e] + og[E + e];
        }
        dW_r[x] = v;
    }
    const int64_t nb = o ? (n + blockDim.x - 1) / blockDim.x : 0;  // blocks of the dW_r part
    if (db_r && blockIdx.x >= nb) {
        const int64_t e = (int64_t)(blockIdx.x - nb) * (blockDim.x >> 5) + (threadIdx.x >> 5);
        const int lane = threadIdx.x & 31;
        if (e < E) {
            float v = 0.f;
            for (int b = lane; b < nblk; b += 32) v += dbr_part[(int64_t)b * E + e];
            v = warp_sum_f(v);
            if (lane == 0) db_r[e] = v;
        }
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------------------------
// f32 grouped GEMM on the CUDA cores (the backward of f32 layers): C(m, n) (+)= sum_k A(m, k)
// B(k, n) (+ bias[g][n]), A(m, k) = A[m sam + k sak], B(k, n) = B[k sbk + n sbn], per group g:
//   rows mode (kmode = 0): rows [seg[g], seg[g+1]) of A and C (A's row a_rows[m] when given), B
//     offset by g sbg, K = the whole K;
//   K mode: the K range [seg[g], seg[g+1]), C offset by g cg, rows [0, M).
// 64 x 64 output tiles, thread (tx, ty) of 16 x 16 owning 4 x 4 outputs, K in chunks of 16
// through shared memory (loaded along whichever operand axis is contiguous).
struct GemmF32 {
    const float *A, *B, *bias;
    float *C;
    const int32_t *seg, *a_rows;
    int64_t sam, sak, sbk, sbn, sbg, ldc, cg, a_src_rows;
    int G, kmode, M, N, K, beta;
};

__global__ void __launch_bounds__(256) gemm_f32_kernel(const GemmF32 a, uint32_t *dev_status) {
    __shared__ __align__(16) float As[16][BT + 4];
    __shared__ __align__(16) float Bs[16][BT + 4];
    __shared__ int32_t sseg[257], cum[257];
    pdl_wait();
    for (int q = threadIdx.x; q <= a.G; q += blockDim.x) sseg[q] = a.seg[q];
    __syncthreads();
    int g, m0, mend, kbeg, kend;
    if (!a.kmode) {
        if (threadIdx.x == 0) {
            int acc = 0;
            for (int q = 0; q < a.G; ++q) {
                cum[q] = acc;
                const int cnt = sseg[q + 1] - sseg[q];
                acc += cnt > 0 ? (cnt + BT - 1) / BT : 0;
            }
            cum[a.G] = acc;
        }
        __syncthreads();
        const int y = blockIdx.y;
        if (y >= cum[a.G]) {
            pdl_trigger();
            return;
        }
        int lo = 0, hi = a.G - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cum[mid] <= y) lo = mid; else hi = mid - 1;
        }
        g = lo;
        m0 = sseg[g] + (y - cum[g]) * BT;
        mend = sseg[g + 1];
        kbeg = 0;
        kend = a.K;
    } else {
        g = blockIdx.z;
        m0 = blockIdx.y * BT;
        mend = a.M;
        kbeg = sseg[g];
        kend = sseg[g + 1];
    }
    const int n0 = blockIdx.x * BT;
    const float *Bg = a.B + (a.kmode ? 0 : (int64_t)g * a.sbg);
    float *Cg = a.C + (a.kmode ? (int64_t)g * a.cg : 0);
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int k0 = kbeg; k0 < kend; k0 += 16) {
        __syncthreads();
        for (int x = threadIdx.x; x < 16 * BT; x += blockDim.x) {
            int kk, mm;
            if (a.sak == 1) { kk = x & 15; mm = x >> 4; } else { mm = x & 63; kk = x >> 6; }
            const int m = m0 + mm, k = k0 + kk;
            float v = 0.f;
            if (m < mend && k < kend) {
                int64_t arow = m;
                if (a.a_rows) {
                    arow = a.a_rows[m];
                    if (arow < 0 || arow >= a.a_src_rows) {
                        report(dev_status, DEV_ERR_INDEX);
                        arow = -1;
                    }
                }
                if (arow >= 0) v = a.A[arow * a.sam + (int64_t)k * a.sak];
            }
            As[kk][mm] = v;
        }
        for (int x = threadIdx.x; x < 16 * BT; x += blockDim.x) {
            int kk, nn;
            if (a.sbn == 1) { nn = x & 63; kk = x >> 6; } else { kk = x & 15; nn = x >> 4; }
            const int n = n0 + nn, k = k0 + kk;
            Bs[kk][nn] = (n < a.N && k < kend) ? Bg[(int64_t)k * a.sbk + (int64_t)n * a.sbn] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const float4 a4 = *reinterpret_cast<const float4 *>(&As[kk][ty * 4]);
            const float4 b4 = *reinterpret_cast<const float4 *>(&Bs[kk][tx * 4]);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
            const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= mend) break;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= a.N) break;
            float v = acc[i][j];
            if (a.bias) v += a.bias[(int64_t)g * a.N + n];
            float *cp = Cg + (int64_t)m * a.ldc + n;
            *cp = a.beta ? *cp + v : v;
        }
    }
    pdl_trigger();
}

// Bias gradients from the per-tile sums: out[e][n] = sum over the 64-row tiles of expert e's
// padded segment of part[tile][n], in tile order (zero for an expert without slots).
__global__ void __launch_bounds__(256) seg_sum_kernel(const float *part, int width,
                                                      const int32_t *kseg, int E, float *out) {
    pdl_wait();
    const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x < (int64_t)E * width) {
        const int e = (int)(x / width), n = (int)(x - (int64_t)e * width);
        float v = 0.f;
        for (int c = kseg[e] / BT; c < kseg[e + 1] / BT; ++c) v += part[(int64_t)c * width + n];
        out[x] = v;
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------------------------
// host side

size_t al(size_t x) { return (x + 1023) & ~(size_t)1023; }



// Blocks of the router backward (their dz sums make db_r).
constexpr int RB_BLOCKS_MAX = 4096;
int router_bwd_blocks(int64_t T) {
    const int64_t b = (T + 7) / 8;
    return (int)(b < RB_BLOCKS_MAX ? (b > 0 ? b : 1) : RB_BLOCKS_MAX);
}

struct BwdLayout {
    size_t gate_r, kseg, seg, A1, A3, Xp, dYp, dHu, dA, Hs, dX, dg_part, db1_part, db2_part, Zp,
        Wp, dz, zl, dhr, dwr_out, dbr_part, total;
    int64_t kw;  // padded slot width: roundup64(P) + 64 E >= sum_e roundup64(count_e)
    int K2, n_part;
    int Kp;      // columns of the bf16 pieces of dz and W_r: roundup64(3 E)
    int Nr;      // columns of h^T [hi | lo]: roundup64(2 E)
    int nsplit;  // K groups of h^T [hi | lo]
};

BwdLayout bwd_layout(const moe_config_t &c) {
    BwdLayout L = {};
    const int64_t P = c.T * c.k;
    const bool sw = c.act == MOE_ACT_SWIGLU;
    L.kw = (P + BT - 1) / BT * BT + (int64_t)BT * c.E;
    L.K2 = sw ? 2 * c.f : c.f;
    L.n_part = c.f / BT;
    L.Kp = (3 * c.E + BT - 1) / BT * BT;
    L.Nr = (2 * c.E + BT - 1) / BT * BT;
    {
        // enough K groups that the d/128 x Nr/256 output tiles of h^T [hi | lo] fill the SMs,
        // each group at least 512 rows
        const int64_t tiles = (int64_t)((c.d + 127) / 128) * ((L.Nr + 255) / 256);
        int64_t g = (148 + tiles - 1) / tiles;
        const int64_t gmax = (c.T + 511) / 512;
        if (g > gmax) g = gmax;
        if (g < 1) g = 1;
        if (g > 64) g = 64;
        L.nsplit = (int)g;
    }
    const size_t E = (size_t)c.E, d = (size_t)c.d, f = (size_t)c.f, kw = (size_t)L.kw;
    const size_t nt = kw / BT;
    const bool f32 = c.dtype == MOE_F32;
    const size_t es = f32 ? 4 : 2;  // per-slot tensors in the layer's type
    size_t off = 0;
    L.gate_r = off;     off = al(off + (size_t)P * 4);
    L.kseg = off;       off = al(off + (E + 1) * 4);
    L.seg = off;        off = al(off + (size_t)(3 + L.nsplit) * 4);
    L.A1 = off;         off = al(off + (size_t)P * f * es);
    L.A3 = off;         off = al(off + (sw ? (size_t)P * f * es : 0));
    // padded row layout [kw, .]: expert e's slots at rows [kseg[e], kseg[e+1]), pad rows zero
    L.Xp = off;         off = al(off + kw * d * es);
    L.dYp = off;        off = al(off + kw * d * es);
    L.dHu = off;        off = al(off + kw * f * es);
    L.dA = off;         off = al(off + kw * (size_t)L.K2 * es);
    L.Hs = off;         off = al(off + kw * f * es);
    L.dX = off;         off = al(off + kw * d * es);
    L.dg_part = off;    off = al(off + (size_t)L.n_part * (size_t)P * 4);
    L.db1_part = off;   off = al(off + (c.has_bias ? nt * f * 4 : 0));
    L.db2_part = off;   off = al(off + (c.has_bias ? nt * d * 4 : 0));
    L.Zp = off;         off = al(off + (f32 ? 0 : (size_t)c.T * L.Kp * 2));
    L.Wp = off;         off = al(off + (f32 ? 0 : d * L.Kp * 2));
    L.dz = off;         off = al(off + (f32 ? (size_t)c.T * E * 4 : 0));
    // logits for layers without the tensor-core router
    L.zl = off;         off = al(off + (router_launches(c) == 3 ? 0 : (size_t)c.T * E * 4));
    L.dhr = off;        off = al(off + (size_t)c.T * d * 4);
    L.dwr_out = off;    off = al(off + (f32 ? 0 : (size_t)L.nsplit * d * L.Nr * 4));
    L.dbr_part = off;   off = al(off + (size_t)router_bwd_blocks(c.T) * E * 4);
    L.total = off;
    return L;
}

bool al16(const void *p) { return p && ((uintptr_t)p & 15u) == 0; }
bool al4(const void *p) { return p && ((uintptr_t)p & 3u) == 0; }

}  // namespace

size_t backward_ws_bytes(const moe_config_t &c) { return bwd_layout(c).total; }

size_t backward_pre_offset(const moe_config_t &c, int which) {
    const BwdLayout L = bwd_layout(c);
    return which == 0 ? L.A1 : L.A3;
}

int backward_launches(const moe_config_t &c, bool saved) {
    if (c.T == 0) return 0;
    const bool sw = c.act == MOE_ACT_SWIGLU;
    if (c.dtype == MOE_F32)  // CUDA-core GEMMs; the pre-activations are always recomputed
        return 1 /*prep*/ + (sw ? 2 : 1) /*A1, A3*/ + 1 /*padded gathers*/ + 1 /*dHu*/ +
               1 /*act*/ + (sw ? 2 : 1) /*dX*/ + (sw ? 3 : 2) /*dW*/ + 2 /*logits, router bwd*/ +
               2 /*dz W_r^T, dh*/ + 1 /*h^T dz*/ + 1 /*db_r*/ + (c.has_bias ? 2 : 0);
    // the logits: the forward's tensor-core partials, still in the router scratch of ws, or the
    // direct kernel
    const int router = router_launches(c) == 3 ? 0 : 1;
    return 2 /*prep, W_r pieces*/ + (saved ? 0 : sw ? 2 : 1) /*A1, A3*/ +
           2 /*padded gathers, dHu*/ + 1 /*act*/ + 1 /*dX*/ + (sw ? 3 : 2) /*dW*/ +
           router + 1 /*router bwd*/ + 2 /*dz W_r^T, dh*/ + 2 /*h^T dz, dW_r and db_r*/ +
           (c.has_bias ? 2 : 0);
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_backward_workspace_size(const moe_config_t *cfg, size_t *bytes) {
    const moe_status_t st = validate_config(cfg);
    if (st != MOE_OK) return st;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = bwd_layout(*cfg).total;
    return MOE_OK;
}

moe_status_t moe_backward_launch_count(const moe_config_t *cfg, int32_t saved_preact,
                                       int32_t *kernels) {
    const moe_status_t st = validate_config(cfg);
    if (st != MOE_OK) return st;
    if (!kernels || (saved_preact != 0 && saved_preact != 1)) return MOE_ERR_INVALID_ARG;
    if (cfg->dtype == MOE_F32 && saved_preact) return MOE_ERR_UNSUPPORTED;
    *kernels = backward_launches(*cfg, saved_preact != 0);
    return MOE_OK;
}

moe_status_t moe_backward(const moe_config_t *cfg, const void *h, const float *W_r,
                          const float *b_r, const void *W1, const float *b1, const void *W3,
                          const void *W2, const float *b2, const int32_t *topk_idx,
                          const int32_t *counts, const void *dy, float aux_weight,
                          float zloss_weight, void *dh, float *dW_r, float *db_r, void *dW1,
                          float *db1, void *dW3, void *dW2, float *db2, void *ws, size_t ws_bytes,
                          void *bws, size_t bws_bytes, int32_t saved_preact, void *stream) {
    moe_status_t st = validate_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config_t &c = *cfg;
    const bool sw = c.act == MOE_ACT_SWIGLU;
    const bool f32 = c.dtype == MOE_F32;
    if (!isfinite(aux_weight) || !isfinite(zloss_weight)) return MOE_ERR_INVALID_ARG;
    if (saved_preact != 0 && saved_preact != 1) return MOE_ERR_INVALID_ARG;
    if (f32 && saved_preact) return MOE_ERR_UNSUPPORTED;  // f32 layers recompute them
    if (!al16(ws) || !al16(bws) || !al4(dW_r) || !al16(dW1) || !al16(dW2) ||
        (sw && !al16(dW3)) || ((b_r != nullptr) != (db_r != nullptr)) || (db_r && !al4(db_r)) ||
        (c.has_bias && (!al4(db1) || !al4(db2) || !al4(b1) || !al4(b2))))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(c);
    const BwdLayout B = bwd_layout(c);
    if (ws_bytes < L.total || bws_bytes < B.total) return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t E = c.E, d = c.d, f = c.f;
    const size_t wes = f32 ? 4 : 2;  // weight-gradient element size
    if (c.T == 0) {
        // no tokens: every gradient is zero
        cudaError_t e = cudaMemsetAsync(dW_r, 0, (size_t)d * E * 4, s);
        if (e == cudaSuccess && db_r) e = cudaMemsetAsync(db_r, 0, (size_t)E * 4, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dW1, 0, (size_t)(E * f * d) * wes, s);
        if (e == cudaSuccess && sw) e = cudaMemsetAsync(dW3, 0, (size_t)(E * f * d) * wes, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dW2, 0, (size_t)(E * f * d) * wes, s);
        if (e == cudaSuccess && c.has_bias) e = cudaMemsetAsync(db1, 0, (size_t)(E * f) * 4, s);
        if (e == cudaSuccess && c.has_bias) e = cudaMemsetAsync(db2, 0, (size_t)(E * d) * 4, s);
        return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    if (!al16(h) || !al4(W_r) || (b_r && !al4(b_r)) || !al16(W1) || !al16(W2) ||
        (sw && !al16(W3)) || !al16(dy) || !al16(dh) || (topk_idx && !al4(topk_idx)) ||
        (counts && !al4(counts)))
        return MOE_ERR_INVALID_ARG;
    char *w = static_cast<char *>(ws);
    char *b = static_cast<char *>(bws);
    uint32_t *dev_status = reinterpret_cast<uint32_t *>(w + L.status);
    const int32_t *idx = topk_idx ? topk_idx : reinterpret_cast<const int32_t *>(w + L.topk_idx);
    const int32_t *cnt = counts ? counts : reinterpret_cast<const int32_t *>(w + L.counts);
    const float *gates = reinterpret_cast<const float *>(w + L.gates);
    const int32_t *offsets = reinterpret_cast<const int32_t *>(w + L.offsets);
    const int32_t *sorted_token = reinterpret_cast<const int32_t *>(w + L.sorted_token);
    const int32_t *slot_of = reinterpret_cast<const int32_t *>(w + L.slot_of);
    const bool have_xperm = !c.fuse_gather;
    const int64_t P = c.T * c.k;
    auto bf = [&](size_t o) { return reinterpret_cast<__nv_bfloat16 *>(b + o); };
    auto fl = [&](size_t o) { return reinterpret_cast<float *>(b + o); };
    float *gate_r = fl(B.gate_r);
    int32_t *kseg = reinterpret_cast<int32_t *>(b + B.kseg);
    // profilers can select the backward's kernels by this range (no cost without a tool)
    struct Range {
        Range() { nvtxRangePushA("moe_backward"); }
        ~Range() { nvtxRangePop(); }
    } range;
#define MOE_TRY(x)                                     \
    do {                                               \
        if ((x) != cudaSuccess) return MOE_ERR_CUDA;   \
    } while (0)
    // 1. sorted-row gates and the padded segment offsets
    int32_t *seg = reinterpret_cast<int32_t *>(b + B.seg);
    MOE_TRY(launch_pdl(bwd_prep_kernel, dim3((unsigned)((P + 255) / 256)), dim3(256), 0, s, 1,
                       slot_of, gates, offsets, P, c.E, c.T, B.nsplit, gate_r, kseg, seg,
                       dev_status));
    if (f32) {
        // f32 layers: the same steps on the CUDA cores (gemm_f32_kernel), no weight pieces
        if (B.kw / BT + c.E >= 65535 || (P + BT - 1) / BT + c.E >= 65535 ||
            (c.T + BT - 1) / BT + 1 >= 65535)
            return MOE_ERR_UNSUPPORTED;
        auto F = [&](size_t o) { return reinterpret_cast<float *>(b + o); };
        auto gemm = [&](const float *A, int64_t sam, int64_t sak, const int32_t *a_rows,
                        int64_t a_src_rows, const float *Bm, int64_t sbk, int64_t sbn,
                        int64_t sbg, const float *bias, float *C, int64_t ldc, int64_t cg,
                        const int32_t *sg, int G, int kmode, int M, int N, int K,
                        int64_t rows_bound, int beta) -> cudaError_t {
            GemmF32 ga;
            ga.A = A;
            ga.B = Bm;
            ga.bias = bias;
            ga.C = C;
            ga.seg = sg;
            ga.a_rows = a_rows;
            ga.sam = sam;
            ga.sak = sak;
            ga.sbk = sbk;
            ga.sbn = sbn;
            ga.sbg = sbg;
            ga.ldc = ldc;
            ga.cg = cg;
            ga.a_src_rows = a_src_rows;
            ga.G = G;
            ga.kmode = kmode;
            ga.M = M;
            ga.N = N;
            ga.K = K;
            ga.beta = beta;
            const dim3 grid((unsigned)((N + BT - 1) / BT),
                            (unsigned)(kmode ? (M + BT - 1) / BT : (rows_bound + BT - 1) / BT + G),
                            (unsigned)(kmode ? G : 1));
            return launch_pdl(gemm_f32_kernel, grid, dim3(256), 0, s, 1, ga, dev_status);
        };
        const float *hf = static_cast<const float *>(h), *dyf = static_cast<const float *>(dy);
        const float *W1f = static_cast<const float *>(W1), *W3f = static_cast<const float *>(W3);
        const float *W2f = static_cast<const float *>(W2);
        // A1 = h[token] W1_e^T (+ b1), A3 = h[token] W3_e^T over the sorted rows
        MOE_TRY(gemm(hf, d, 1, sorted_token, c.T, W1f, 1, d, f * d, c.has_bias ? b1 : nullptr,
                     F(B.A1), f, 0, offsets, c.E, 0, 0, c.f, c.d, P, 0));
        if (sw)
            MOE_TRY(gemm(hf, d, 1, sorted_token, c.T, W3f, 1, d, f * d, nullptr, F(B.A3), f, 0,
                         offsets, c.E, 0, 0, c.f, c.d, P, 0));
        // padded rows of h and dy (+ db2 parts)
        MOE_TRY(launch_pdl(gather_pad_kernel<float>,
                           dim3((unsigned)(B.kw / BT), (unsigned)((c.d + GP_COLS - 1) / GP_COLS)),
                           dim3(256), 0, s, 1, hf, dyf, sorted_token, offsets,
                           static_cast<const int32_t *>(kseg), static_cast<const float *>(gate_r),
                           c.E, c.T, P, c.d, F(B.Xp), F(B.dYp),
                           c.has_bias ? F(B.db2_part) : nullptr, dev_status));
        // dHu = dYp W2_e (W2_e [d, f]: B(k = o, n) = W2[e][o][n]) over the padded rows
        MOE_TRY(gemm(F(B.dYp), d, 1, nullptr, 0, W2f, f, 1, d * f, nullptr, F(B.dHu), f, 0, kseg,
                     c.E, 0, 0, c.f, c.d, B.kw, 0));
        ActBwd<float> ab;
        ab.A1 = F(B.A1);
        ab.A3 = sw ? F(B.A3) : nullptr;
        ab.dHu = F(B.dHu);
        ab.gate_r = gate_r;
        ab.offsets = offsets;
        ab.kseg = kseg;
        ab.dA = F(B.dA);
        ab.Hs = F(B.Hs);
        ab.dg_part = F(B.dg_part);
        ab.db1_part = c.has_bias ? F(B.db1_part) : nullptr;
        ab.P = P;
        ab.E = c.E;
        ab.f = c.f;
        ab.swiglu = sw ? 1 : 0;
        MOE_TRY(launch_pdl(act_bwd_kernel<float>, dim3((unsigned)((B.kw / BT) * (c.f / BT))),
                           dim3(256), 0, s, 1, ab, dev_status));
        // dX = dA1 W1_e (+ dA3 W3_e) (W1_e [f, d]: B(k = j, n = i) = W1[e][j][i])
        MOE_TRY(gemm(F(B.dA), B.K2, 1, nullptr, 0, W1f, d, 1, f * d, nullptr, F(B.dX), d, 0, kseg,
                     c.E, 0, 0, c.d, c.f, B.kw, 0));
        if (sw)
            MOE_TRY(gemm(F(B.dA) + c.f, B.K2, 1, nullptr, 0, W3f, d, 1, f * d, nullptr, F(B.dX), d,
                         0, kseg, c.E, 0, 0, c.d, c.f, B.kw, 1));
        // weight gradients over each expert's padded rows
        MOE_TRY(gemm(F(B.dYp), 1, d, nullptr, 0, F(B.Hs), f, 1, 0, nullptr,
                     static_cast<float *>(dW2), f, d * f, kseg, c.E, 1, c.d, c.f, 0, 0, 0));
        MOE_TRY(gemm(F(B.dA), 1, B.K2, nullptr, 0, F(B.Xp), d, 1, 0, nullptr,
                     static_cast<float *>(dW1), d, f * d, kseg, c.E, 1, c.f, c.d, 0, 0, 0));
        if (sw)
            MOE_TRY(gemm(F(B.dA) + c.f, 1, B.K2, nullptr, 0, F(B.Xp), d, 1, 0, nullptr,
                         static_cast<float *>(dW3), d, f * d, kseg, c.E, 1, c.f, c.d, 0, 0, 0));
        // router: dz (f32), dz W_r^T, dh, h^T dz, db_r
        RouterBwd<float> rb;
        rb.h = hf;
        rb.dy = dyf;
        rb.W_r = W_r;
        rb.b_r = b_r;
        rb.b2 = c.has_bias ? b2 : nullptr;
        {
            const int64_t blocks = c.T < 4 * (int64_t)num_sms() ? c.T : 4 * (int64_t)num_sms();
            MOE_TRY(launch_pdl(router_logits_direct_kernel<float>, dim3((unsigned)blocks),
                               dim3(256), 0, s, 1, hf, W_r, c.T, c.d, c.E, F(B.zl)));
        }
        rb.part = F(B.zl);
        rb.S = 1;
        rb.ldp = c.E;
        rb.topk_idx = idx;
        rb.slot_of = slot_of;
        rb.counts = cnt;
        rb.gates = gates;
        rb.dg_part = F(B.dg_part);
        rb.n_part = B.n_part;
        rb.T = c.T;
        rb.P = P;
        rb.d = c.d;
        rb.E = c.E;
        rb.k = c.k;
        rb.raw_prob = c.gate == MOE_GATE_RAW_PROB ? 1 : 0;
        rb.aux_weight = aux_weight;
        rb.zloss_weight = zloss_weight;
        rb.Zp = nullptr;
        rb.dz = F(B.dz);
        rb.Kp = 0;
        rb.dbr_part = F(B.dbr_part);
        const int rblocks = router_bwd_blocks(c.T);
        MOE_TRY(launch_pdl(router_bwd_kernel<float>, dim3((unsigned)rblocks), dim3(256), 0, s, 1,
                           rb, dev_status));
        // dz W_r^T: B(k = e, n = i) = W_r[i][e]; one group of T rows (seg = {0, T})
        MOE_TRY(gemm(F(B.dz), E, 1, nullptr, 0, W_r, 1, E, 0, nullptr, F(B.dhr), d, 0, seg, 1, 0,
                     0, c.d, c.E, c.T, 0));
        {
            const int64_t n = c.T * (d / 8);
            int64_t blocks = (n + 255) / 256;
            if (blocks > 8 * (int64_t)num_sms()) blocks = 8 * (int64_t)num_sms();
            const auto dhk = c.k == 1 ? dh_kernel<float, 1> : dh_kernel<float, 4>;
            MOE_TRY(launch_pdl(dhk, dim3((unsigned)blocks), dim3(256), 0, s, 1,
                               static_cast<const float *>(F(B.dX)),
                               static_cast<const float *>(F(B.dhr)), slot_of, idx, offsets,
                               static_cast<const int32_t *>(kseg), c.T, c.d, c.E, c.k,
                               static_cast<float *>(dh), dev_status));
        }
        // h^T dz straight into dW_r (K = the T tokens, seg = {0, T})
        MOE_TRY(gemm(hf, 1, d, nullptr, 0, F(B.dz), E, 1, 0, nullptr, dW_r, E, 0, seg, 1, 1, c.d,
                     c.E, 0, 0, 0));
        MOE_TRY(launch_pdl(router_final_kernel, dim3((unsigned)((E + 7) / 8)), dim3(256), 0, s, 1,
                           static_cast<const float *>(nullptr), 0, c.d, c.E, 1,
                           static_cast<const float *>(F(B.dbr_part)), rblocks, dW_r, db_r));
        if (c.has_bias) {
            MOE_TRY(launch_pdl(seg_sum_kernel, dim3((unsigned)((E * f + 255) / 256)), dim3(256), 0,
                               s, 1, static_cast<const float *>(F(B.db1_part)), c.f,
                               static_cast<const int32_t *>(kseg), c.E, db1));
            MOE_TRY(launch_pdl(seg_sum_kernel, dim3((unsigned)((E * d + 255) / 256)), dim3(256), 0,
                               s, 1, static_cast<const float *>(F(B.db2_part)), c.d,
                               static_cast<const int32_t *>(kseg), c.E, db2));
        }
        return MOE_OK;
    }
    // 2. the router weight as bf16 pieces (for dz W_r^T on the tensor cores)
    {
        const int64_t n = d * B.Kp;
        int64_t blocks = (n + 255) / 256;
        if (blocks > 4 * (int64_t)num_sms()) blocks = 4 * (int64_t)num_sms();
        MOE_TRY(launch_pdl(wr_pieces_kernel, dim3((unsigned)blocks), dim3(256), 0, s, 1, W_r, c.d,
                           c.E, B.Kp, bf(B.Wp)));
    }
    // 3. pre-activations A1 = X W1^T (+ b1), A3 = X W3^T: left in bws by moe_forward_train, or
    // recomputed here
    if (!saved_preact) {
        const void *xa = have_xperm ? static_cast<const void *>(w + L.x_perm) : h;
        const int32_t *xrows = have_xperm ? nullptr : sorted_token;
        MOE_TRY(launch_gemm_rows(xa, xrows, c.T, W1, P, c.E, c.d, c.f, offsets,
                                 c.has_bias ? b1 : nullptr, bf(B.A1), dev_status, s));
        if (sw)
            MOE_TRY(launch_gemm_rows(xa, xrows, c.T, W3, P, c.E, c.d, c.f, offsets, nullptr,
                                     bf(B.A3), dev_status, s));
    }
    // 4. padded rows of h and dy (+ db2 parts), then dHu = dYp W2_e over each expert's padded
    // rows (W2_e read MN-major: rows o of W2 [E d, f] are the K index)
    const int32_t *ksegc = kseg;
    MOE_TRY(launch_pdl(gather_pad_kernel<__nv_bfloat16>,
                       dim3((unsigned)(B.kw / BT), (unsigned)((c.d + GP_COLS - 1) / GP_COLS)),
                       dim3(256), 0, s, 1, static_cast<const __nv_bfloat16 *>(h),
                       static_cast<const __nv_bfloat16 *>(dy), sorted_token, offsets, ksegc,
                       static_cast<const float *>(gate_r), c.E, c.T, P, c.d, bf(B.Xp), bf(B.dYp),
                       c.has_bias ? fl(B.db2_part) : nullptr, dev_status));
    MOE_TRY(launch_gemm_rows_bmn(bf(B.dYp), W2, nullptr, c.d, 0, B.kw, c.E, c.d, c.f, ksegc,
                                 bf(B.dHu), dev_status, s));
    // 5. activation backward: dA, Hs = g Hact (padded rows), dg parts, db1 parts
    ActBwd<__nv_bfloat16> ab;
    ab.A1 = bf(B.A1);
    ab.A3 = sw ? bf(B.A3) : nullptr;
    ab.dHu = bf(B.dHu);
    ab.gate_r = gate_r;
    ab.offsets = offsets;
    ab.kseg = ksegc;
    ab.dA = bf(B.dA);
    ab.Hs = bf(B.Hs);
    ab.dg_part = fl(B.dg_part);
    ab.db1_part = c.has_bias ? fl(B.db1_part) : nullptr;
    ab.P = P;
    ab.E = c.E;
    ab.f = c.f;
    ab.swiglu = sw ? 1 : 0;
    MOE_TRY(launch_pdl(act_bwd_kernel<__nv_bfloat16>, dim3((unsigned)((B.kw / BT) * (c.f / BT))),
                       dim3(256), 0, s, 1, ab, dev_status));
    // 6. dX = dA1 W1_e + dA3 W3_e over the padded rows: one GEMM over K2 = [dA1 | dA3], B = W1
    // then W3 read MN-major
    MOE_TRY(launch_gemm_rows_bmn(bf(B.dA), W1, sw ? W3 : nullptr, c.f, sw ? c.f / BT : 0, B.kw,
                                 c.E, B.K2, c.d, ksegc, bf(B.dX), dev_status, s));
    // 7. weight gradients over each expert's padded rows, every operand MN-major:
    //    dW2_e = dYp^T Hs, dW1_e = dA1^T Xp, dW3_e = dA3^T Xp
    MOE_TRY(launch_gemm_kgroup_mn(bf(B.dYp), c.d, bf(B.Hs), c.f, ksegc, c.E, c.d, c.f, B.kw, dW2,
                                  dev_status, s));
    MOE_TRY(launch_gemm_kgroup_mn(bf(B.dA), B.K2, bf(B.Xp), c.d, ksegc, c.E, c.f, c.d, B.kw, dW1,
                                  dev_status, s));
    if (sw)
        MOE_TRY(launch_gemm_kgroup_mn(bf(B.dA) + c.f, B.K2, bf(B.Xp), c.d, ksegc, c.E, c.f, c.d,
                                      B.kw, dW3, dev_status, s));
    // 9. router: logits (the forward's tensor-core partials when its router ran on the tensor
    // cores, else the direct kernel), dz
    RouterBwd<__nv_bfloat16> rb;
    rb.h = static_cast<const __nv_bfloat16 *>(h);
    rb.dy = static_cast<const __nv_bfloat16 *>(dy);
    rb.W_r = W_r;
    rb.b_r = b_r;
    rb.b2 = c.has_bias ? b2 : nullptr;
    if (router_launches(c) == 3) {
        // h . W_r without the bias, [S][T][Epad] f32 partials over K chunks, as the forward's
        // router left them (the same h and W_r, so the same values a recompute would give)
        void *scratch = w + L.router;
        rb.part = router_tc_logits(scratch, c);
        rb.S = router_tc_splits(c);
        rb.ldp = router_tc_epad(c);
    } else {
        const int64_t blocks = c.T < 4 * (int64_t)num_sms() ? c.T : 4 * (int64_t)num_sms();
        MOE_TRY(launch_pdl(router_logits_direct_kernel<__nv_bfloat16>, dim3((unsigned)blocks),
                           dim3(256), 0, s, 1, static_cast<const __nv_bfloat16 *>(h), W_r, c.T,
                           c.d, c.E, fl(B.zl)));
        rb.part = fl(B.zl);
        rb.S = 1;
        rb.ldp = c.E;
    }
    rb.topk_idx = idx;
    rb.slot_of = slot_of;
    rb.counts = cnt;
    rb.gates = gates;
    rb.dg_part = fl(B.dg_part);
    rb.n_part = B.n_part;
    rb.T = c.T;
    rb.P = P;
    rb.d = c.d;
    rb.E = c.E;
    rb.k = c.k;
    rb.raw_prob = c.gate == MOE_GATE_RAW_PROB ? 1 : 0;
    rb.aux_weight = aux_weight;
    rb.zloss_weight = zloss_weight;
    rb.Zp = bf(B.Zp);
    rb.dz = nullptr;
    rb.Kp = B.Kp;
    rb.dbr_part = fl(B.dbr_part);
    const int rblocks = router_bwd_blocks(c.T);
    MOE_TRY(launch_pdl(router_bwd_kernel<__nv_bfloat16>, dim3((unsigned)rblocks), dim3(256), 0, s, 1, rb,
                       dev_status));
    // 10. the router's h-gradient dz W_r^T = Zp Wp^T (f32, one group of T rows), then
    // dh = that + sum_j dX[padded row of slot j]
    MOE_TRY(launch_gemm_rows_f32(bf(B.Zp), bf(B.Wp), c.T, 1, B.Kp, c.d, seg, fl(B.dhr),
                                 dev_status, s));
    {
        const int64_t n = c.T * (d / 8);
        int64_t blocks = (n + 255) / 256;
        if (blocks > 8 * (int64_t)num_sms()) blocks = 8 * (int64_t)num_sms();
        const auto dhk = c.k == 1 ? dh_kernel<__nv_bfloat16, 1> : dh_kernel<__nv_bfloat16, 4>;
        MOE_TRY(launch_pdl(dhk, dim3((unsigned)blocks), dim3(256), 0, s, 1,
                           static_cast<const __nv_bfloat16 *>(bf(B.dX)),
                           static_cast<const float *>(fl(B.dhr)), slot_of, idx, offsets, ksegc,
                           c.T, c.d, c.E, c.k, static_cast<__nv_bfloat16 *>(dh), dev_status));
    }
    // 11. dW_r = h^T dz as h^T [hi | lo] on the tensor cores (MN-major operands, one group of
    // K = T rows, rows past T read as zeros), then the two halves added and db_r reduced
    MOE_TRY(launch_gemm_kgroup_mn(h, c.d, bf(B.Zp), B.Kp, seg + 2, B.nsplit, c.d, B.Nr,
                                  (c.T + BT - 1) / BT * BT, nullptr, dev_status, s, c.T,
                                  fl(B.dwr_out)));
    {
        const int64_t nb = (d * E + 255) / 256, eb = b_r ? (E + 7) / 8 : 0;
        MOE_TRY(launch_pdl(router_final_kernel, dim3((unsigned)(nb + eb)), dim3(256), 0, s, 1,
                           static_cast<const float *>(fl(B.dwr_out)), B.Nr, c.d, c.E, B.nsplit,
                           static_cast<const float *>(fl(B.dbr_part)), rblocks, dW_r, db_r));
    }
    // 12. bias gradients
    if (c.has_bias) {
        MOE_TRY(launch_pdl(seg_sum_kernel, dim3((unsigned)((E * f + 255) / 256)), dim3(256), 0, s,
                           1, static_cast<const float *>(fl(B.db1_part)), c.f,
                           static_cast<const int32_t *>(kseg), c.E, db1));
        MOE_TRY(launch_pdl(seg_sum_kernel, dim3((unsigned)((E * d + 255) / 256)), dim3(256), 0, s,
                           1, static_cast<const float *>(fl(B.db2_part)), c.d,
                           static_cast<const int32_t *>(kseg), c.E, db2));
    }
#undef MOE_TRY
    return MOE_OK;
}

}  // extern "C"
