// ffn_f32.cu -- step 4 of the MoE layer in f32 on the CUDA cores (the f32 workloads).
//
// Every expert e is an MLP over its contiguous block of permuted rows [offsets[e], offsets[e+1])
// (llm.curionode.com "Mixture of Experts.", "Workshop"; lensaml.com "Mixture of Experts",
// Step 1 and Step 6: a full expert is three d x f matrices):
//   GELU form   : H = GELU_tanh(X W1_e^T + b1_e),   Y = H W2_e^T + b2_e
//   SwiGLU form : H = SiLU(X W1_e^T) * (X W3_e^T),  Y = H W2_e^T
// Two launches of one tiled FFMA kernel. A block computes a TBM x TBN output tile of one expert
// (thread tile TM x TN, 256 threads); it finds its (expert, row tile) from the offsets, staged in
// shared memory, so the grid is sized on the host without knowing the per-expert counts.
// The K loop streams 32-wide slices of the A rows and of the weight rows into shared memory with
// cp.async, several slices in flight, so the loads of later slices overlap the FMAs of the
// current one; within a slice the next k group's operands are read while the current one's FMAs
// run. Small layers (few output tiles) take 32 x 32 tiles, so that more SMs get work. Every output
// is one f32 FMA chain in ascending k, the same for both tile shapes.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int FK = 32;          // K slice
constexpr int FLD = FK + 4;     // shared row stride in floats: 16-byte aligned rows, and eight
                                // consecutive rows start in eight different 16-byte bank groups
constexpr int FTHREADS = 256;

enum { EPI_STORE = 0, EPI_GELU = 1, EPI_SWIGLU = 2 };

struct F32Args {
    const float *A;               // [P, K]
    const float *B, *B3;          // [E, N, K]
    const float *bias;            // [E, N] or null
    float *out;                   // [P, N]
    const int32_t *offsets;       // [E+1]
    uint32_t *dev_status;
    int E, K, N;
    int64_t P;
    // gathered A rows (first launch of moe_forward): row r of the A tile is row a_rows[r] of A
    // (a [a_src_rows, K] tensor, h) instead of row r of a permuted copy
    const int32_t *a_rows;
    int64_t a_src_rows;
    // combine fused into the second launch (cmb_y not null): the last block of every column tile
    // forms y[t, cols] = sum_j gates[t, j] out[slot_of[t k + j], cols] for every token
    const int32_t *cmb_slot;
    const float *cmb_gates;
    float *cmb_y;
    uint32_t *cmb_arrive;  // one counter per column tile, zero between launches
    int64_t cmb_T;
    int cmb_k;
};

template <int TBM, int TBN, int NS, int EPI>
struct FTile {
    static constexpr int NB = EPI == EPI_SWIGLU ? 2 : 1;          // weight matrices per tile
    static constexpr int STAGE_FLOATS = (TBM + NB * TBN) * FLD;
    static constexpr size_t SMEM = (size_t)NS * STAGE_FLOATS * sizeof(float);  // NS slices
};

__device__ __forceinline__ float gelu_tanh(float x) {
    return 0.5f * x * (1.f + tanhf(0.7978845608028654f * (x + 0.044715f * x * x * x)));
}
__device__ __forceinline__ float silu(float x) { return x / (1.f + expf(-x)); }

// 16-byte asynchronous copy global -> shared; src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The output tile (row0, rows) of expert e: the K loop and the epilogue of ffn_f32_kernel.
template <int TBM, int TBN, int TM, int TN, int NS, int EPI>
__device__ __forceinline__ void ffn_tile(const F32Args &a, const int e, const int row0,
                                         const int rows, float *fsm) {
    using Tl = FTile<TBM, TBN, NS, EPI>;
    constexpr int RSTEP = TBM / TM, CSTEP = TBN / TN;  // a thread's rows / columns are strided
    constexpr int CHUNKS = FK / 4;                      // 16-byte pieces per row slice
    const int tid = threadIdx.x;
    const int n0 = blockIdx.y * TBN;
    const int ty = tid / CSTEP, tx = tid % CSTEP;
    const float *Be = a.B + (int64_t)e * a.N * a.K;
    const float *B3e = EPI == EPI_SWIGLU ? a.B3 + (int64_t)e * a.N * a.K : nullptr;
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(fsm));
    // the A rows this thread copies (the same in every K slice): rows past the tile's last valid
    // row copy zeros from a real row; a gathered row comes from h through a_rows
    constexpr int A_PER = TBM * CHUNKS / FTHREADS;
    static_assert(A_PER * FTHREADS == TBM * CHUNKS, "whole A pieces per thread");
    const float *arow[A_PER];
#pragma unroll
    for (int i = 0; i < A_PER; ++i) {
        const int r = (tid + i * FTHREADS) / CHUNKS;
        int64_t src = r < rows ? row0 + r : row0;
        if (a.a_rows) {
            int tok = r < rows ? __ldg(a.a_rows + row0 + r) : 0;
            if (tok < 0 || (int64_t)tok >= a.a_src_rows) {
                report(a.dev_status, DEV_ERR_INDEX);
                tok = 0;
            }
            src = tok;
        }
        arow[i] = a.A + src * a.K;
    }

    // One K slice into stage `st`: TBM A rows (zeros past the tile's last row), then TBN rows of
    // each weight matrix.
    auto load_slice = [&](int st, int k0) {
        const uint32_t sA = sbase + st * Tl::STAGE_FLOATS * 4;
#pragma unroll
        for (int i = 0; i < A_PER; ++i) {
            const int c = tid + i * FTHREADS;
            const int r = c / CHUNKS, q = c % CHUNKS;
            cp_async16(sA + (r * FLD + 4 * q) * 4, arow[i] + k0 + 4 * q, r < rows ? 16 : 0);
        }
        const uint32_t sB = sA + TBM * FLD * 4;
        for (int c = tid; c < Tl::NB * TBN * CHUNKS; c += FTHREADS) {
            const int r = c / CHUNKS, q = c % CHUNKS;
            const float *W = (EPI == EPI_SWIGLU && r >= TBN) ? B3e + (int64_t)(n0 + r - TBN) * a.K
                                                              : Be + (int64_t)(n0 + r) * a.K;
            cp_async16(sB + (r * FLD + 4 * q) * 4, W + k0 + 4 * q, 16);
        }
    };

    float acc[TM][TN], acc3[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = acc3[i][j] = 0.f;

    const int nk = a.K / FK;
#pragma unroll
    for (int s = 0; s < NS - 1; ++s) {
        if (s < nk) load_slice(s, s * FK);
        cp_async_commit();
    }
    for (int kb = 0; kb < nk; ++kb) {
        cp_async_wait<NS - 2>();       // this thread's copies of slice kb have landed
        __syncthreads();               // everyone's have, and slice kb-1 is no longer read
        const int nxt = kb + NS - 1;
        if (nxt < nk) load_slice(nxt % NS, nxt * FK);
        cp_async_commit();
        const float *As = fsm + (kb % NS) * Tl::STAGE_FLOATS;
        const float *Bs = As + TBM * FLD;
        const float *B3s = Bs + TBN * FLD;
        // operands of the next 4-wide k group are read from shared memory while the FMAs of the
        // current group run (two register sets, alternating)
        float4 x[2][TM], w[2][TN], w3[2][TN];
        auto fetch = [&](int b, int kk) {
#pragma unroll
            for (int i = 0; i < TM; ++i)
                x[b][i] = *reinterpret_cast<const float4 *>(As + (ty + RSTEP * i) * FLD + kk);
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                w[b][j] = *reinterpret_cast<const float4 *>(Bs + (tx + CSTEP * j) * FLD + kk);
                if (EPI == EPI_SWIGLU)
                    w3[b][j] = *reinterpret_cast<const float4 *>(B3s + (tx + CSTEP * j) * FLD + kk);
            }
        };
        fetch(0, 0);
#pragma unroll
        for (int g = 0; g < FK / 4; ++g) {
            const int b = g & 1;
            if (g + 1 < FK / 4) fetch(b ^ 1, 4 * (g + 1));
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) {
                    acc[i][j] = fmaf(x[b][i].x, w[b][j].x, acc[i][j]);
                    acc[i][j] = fmaf(x[b][i].y, w[b][j].y, acc[i][j]);
                    acc[i][j] = fmaf(x[b][i].z, w[b][j].z, acc[i][j]);
                    acc[i][j] = fmaf(x[b][i].w, w[b][j].w, acc[i][j]);
                    if (EPI == EPI_SWIGLU) {
                        acc3[i][j] = fmaf(x[b][i].x, w3[b][j].x, acc3[i][j]);
                        acc3[i][j] = fmaf(x[b][i].y, w3[b][j].y, acc3[i][j]);
                        acc3[i][j] = fmaf(x[b][i].z, w3[b][j].z, acc3[i][j]);
                        acc3[i][j] = fmaf(x[b][i].w, w3[b][j].w, acc3[i][j]);
                    }
                }
        }
    }
    cp_async_wait<0>();
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int r = ty + RSTEP * i;
        if (r >= rows) continue;
        float *orow = a.out + (int64_t)(row0 + r) * a.N;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int n = n0 + tx + CSTEP * j;
            float v = acc[i][j];
            if (EPI == EPI_SWIGLU) {
                v = silu(v) * acc3[i][j];
            } else {
                if (a.bias) v += a.bias[(int64_t)e * a.N + n];
                if (EPI == EPI_GELU) v = gelu_tanh(v);
            }
            orow[n] = v;
        }
    }
}

// Combine fused into the second expert launch of a small f32 layer (lensaml.com "Mixture of
// Experts", Step 3: y = sum_j g_j E_j(h)). Every block, done with its output tile, makes its
// stores visible and counts itself in on its column tile's counter; the last block of a column
// tile then forms y[t, n0 .. n0 + TBN) = sum_j gates[t, j] out[slot_of[t k + j], n0 ..] for every
// token t -- f32 FMA in j order from 0, dropped slots skipped: the combine kernel's arithmetic, so
// the same bits -- with four (token, 4-column) units in flight per thread, and puts its counter
// back to zero for the next launch. Blocks without a tile count themselves in too.
template <int TBN>
__device__ __forceinline__ void combine_tail(const F32Args &a, int32_t *s_last) {
    __threadfence();  // this block's output stores are visible before it counts itself in
    __syncthreads();
    if (threadIdx.x == 0) *s_last = atomicAdd(a.cmb_arrive + blockIdx.y, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!*s_last) return;
    __threadfence();  // the other blocks' stores of this column tile are visible to this one
    constexpr int C4 = TBN / 4, U = 4;
    const int N = a.N, k = a.cmb_k;
    const int c0 = blockIdx.y * C4;  // first float4 column of the tile
    const int64_t units = a.cmb_T * C4;
    for (int64_t u0 = threadIdx.x; u0 < units; u0 += U * FTHREADS) {
        float4 acc[U];
        int64_t t[U];
        int col[U];
#pragma unroll
        for (int q = 0; q < U; ++q) {
            acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            const int64_t u = u0 + q * FTHREADS;
            t[q] = u < units ? u / C4 : -1;
            col[q] = c0 + (int)(u - (u / C4) * C4);
        }
        for (int j = 0; j < k; ++j) {
            float4 v[U];
            float g[U];
            bool has[U];
#pragma unroll
            for (int q = 0; q < U; ++q) {
                has[q] = false;
                if (t[q] < 0) continue;
                const int32_t r = a.cmb_slot[t[q] * k + j];
                if (r == -1) continue;  // dropped by a capacity
                if (r < 0 || r >= a.P) {
                    report(a.dev_status, DEV_ERR_INDEX);
                    continue;
                }
                has[q] = true;
                g[q] = a.cmb_gates[t[q] * k + j];
                v[q] = __ldcg(reinterpret_cast<const float4 *>(a.out + (int64_t)r * N) + col[q]);
            }
#pragma unroll
            for (int q = 0; q < U; ++q) {
                if (!has[q]) continue;
                acc[q].x = fmaf(g[q], v[q].x, acc[q].x);
                acc[q].y = fmaf(g[q], v[q].y, acc[q].y);
                acc[q].z = fmaf(g[q], v[q].z, acc[q].z);
                acc[q].w = fmaf(g[q], v[q].w, acc[q].w);
            }
        }
#pragma unroll
        for (int q = 0; q < U; ++q)
            if (t[q] >= 0) reinterpret_cast<float4 *>(a.cmb_y + t[q] * N)[col[q]] = acc[q];
    }
    if (threadIdx.x == 0) a.cmb_arrive[blockIdx.y] = 0u;
}

template <int TBM, int TBN, int TM, int TN, int NS, int EPI, bool CMB>
__global__ void __launch_bounds__(FTHREADS) ffn_f32_kernel(F32Args a) {
    static_assert((TBM / TM) * (TBN / TN) == FTHREADS, "one thread per TM x TN outputs");
    extern __shared__ __align__(16) float fsm[];
    __shared__ int32_t s_off[257];
    __shared__ int32_t s_e, s_row0, s_rows, s_last;
    const int tid = threadIdx.x;
    pdl_wait();
    for (int i = tid; i <= a.E; i += FTHREADS) s_off[i] = a.offsets[i];
    __syncthreads();
    if (tid == 0) {
        int cum = 0, e_found = -1, m = 0;
        for (int e = 0; e < a.E; ++e) {
            const int lo = s_off[e], hi = s_off[e + 1];
            if (hi < lo || lo < 0 || hi > a.P) {
                report(a.dev_status, DEV_ERR_INDEX);
                break;
            }
            const int mt = (hi - lo + TBM - 1) / TBM;
            if ((int)blockIdx.x < cum + mt) {
                e_found = e;
                m = blockIdx.x - cum;
                break;
            }
            cum += mt;
        }
        s_e = e_found;
        if (e_found >= 0) {
            s_row0 = s_off[e_found] + m * TBM;
            s_rows = min(TBM, s_off[e_found + 1] - s_row0);
        }
    }
    __syncthreads();
    const int e = s_e;
    if (e >= 0) ffn_tile<TBM, TBN, TM, TN, NS, EPI>(a, e, s_row0, s_rows, fsm);
    if (CMB) combine_tail<TBN>(a, &s_last);
    pdl_trigger();
}

template <int TBM, int TBN, int TM, int TN, int NS, int EPI, bool CMB>
cudaError_t launch_tiles(const F32Args &a, int64_t P, cudaStream_t s) {
    constexpr size_t smem = FTile<TBM, TBN, NS, EPI>::SMEM;
    const void *k = (const void *)ffn_f32_kernel<TBM, TBN, TM, TN, NS, EPI, CMB>;
    cudaError_t err = set_max_dynamic_smem(k, smem);
    if (err != cudaSuccess) return err;
    // at most one partial row tile per expert beyond P / TBM full ones
    const int64_t mtiles = (P + TBM - 1) / TBM + a.E;
    dim3 grid((unsigned)mtiles, (unsigned)(a.N / TBN));
    return launch_pdl(ffn_f32_kernel<TBM, TBN, TM, TN, NS, EPI, CMB>, grid, dim3(FTHREADS), smem, s,
                      1, a);
}

template <int EPI, bool CMB = false>
cudaError_t launch_f32(const F32Args &a, int64_t P, cudaStream_t s) {
    // 64 x 64 tiles (4 x 4 per thread, 3 slices in flight) when they give every SM two blocks,
    // else 32 x 32 tiles (2 x 2 per thread, 4 slices in flight: less work per slice to hide the
    // load latency behind)
    const int64_t big = ((P + 63) / 64 + a.E) * (int64_t)(a.N / 64);
    if (big >= 2 * (int64_t)num_sms()) return launch_tiles<64, 64, 4, 4, 3, EPI, CMB>(a, P, s);
    return launch_tiles<32, 32, 2, 2, 4, EPI, CMB>(a, P, s);
}

}  // namespace

bool ffn_f32_combine_ok(const moe_config_t &c) {
    return c.dtype == MOE_F32 && c.T * c.k * (int64_t)c.d <= F32_COMBINE_MAX &&
           c.d / 32 <= F32_COMBINE_TILES;
}

cudaError_t launch_ffn_f32(const moe_config_t &c, const FfnBufs &b, cudaStream_t s) {
    const int64_t P = c.T * c.k;
    if (P == 0) return cudaSuccess;
    F32Args g1{static_cast<const float *>(b.gather_h ? b.gather_h : b.x_perm),
               static_cast<const float *>(b.W1), static_cast<const float *>(b.W3),
               c.has_bias ? b.b1 : nullptr, static_cast<float *>(b.H), b.offsets, b.dev_status,
               c.E, c.d, c.f, P};
    if (b.gather_h) {
        if (!b.sorted_token) return cudaErrorInvalidValue;
        g1.a_rows = b.sorted_token;
        g1.a_src_rows = c.T;
    }
    cudaError_t err = c.act == MOE_ACT_SWIGLU ? launch_f32<EPI_SWIGLU>(g1, P, s)
                                              : launch_f32<EPI_GELU>(g1, P, s);
    if (err != cudaSuccess) return err;
    F32Args g2{static_cast<const float *>(b.H), static_cast<const float *>(b.W2), nullptr,
               c.has_bias ? b.b2 : nullptr, static_cast<float *>(b.y_perm), b.offsets,
               b.dev_status, c.E, c.f, c.d, P};
    if (b.combine_y == nullptr) return launch_f32<EPI_STORE>(g2, P, s);
    if (!ffn_f32_combine_ok(c) || !b.slot_of || !b.gates || !b.arrive)
        return cudaErrorInvalidValue;
    g2.cmb_slot = b.slot_of;
    g2.cmb_gates = b.gates;
    g2.cmb_y = static_cast<float *>(b.combine_y);
    g2.cmb_arrive = b.arrive;
    g2.cmb_T = c.T;
    g2.cmb_k = c.k;
    return launch_f32<EPI_STORE, true>(g2, P, s);
}

}  // namespace moe
