// ffn_f32.cu -- step 4 of the MoE layer in f32 on the CUDA cores (the f32 workloads).
//
// Every expert e is an MLP over its contiguous block of permuted rows [offsets[e], offsets[e+1])
// (llm.curionode.com "Mixture of Experts.", "Workshop"; lensaml.com "Mixture of Experts",
// Step 1 and Step 6: a full expert is three d x f matrices):
//   GELU form   : H = GELU_tanh(X W1_e^T + b1_e),   Y = H W2_e^T + b2_e
//   SwiGLU form : H = SiLU(X W1_e^T) * (X W3_e^T),  Y = H W2_e^T
// Two launches of one tiled kernel (64 x 64 output tile, K-step 16, 4 x 4 outputs per thread).
// A block finds its (expert, row tile) from a tile table it builds from offsets, so the grid is
// sized on the host without knowing the per-expert counts.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int FB = 64;   // tile rows and columns
constexpr int FK = 16;   // K-step

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
};

__device__ __forceinline__ float gelu_tanh(float x) {
    return 0.5f * x * (1.f + tanhf(0.7978845608028654f * (x + 0.044715f * x * x * x)));
}
__device__ __forceinline__ float silu(float x) { return x / (1.f + expf(-x)); }

template <int EPI>
__global__ void __launch_bounds__(256) ffn_f32_kernel(F32Args a) {
    __shared__ float As[FK][FB + 4];
    __shared__ float Bs[FK][FB + 4];
    __shared__ float B3s[EPI == EPI_SWIGLU ? FK : 1][FB + 4];
    __shared__ int32_t s_e, s_row0, s_rows;
    const int tid = threadIdx.x;
    pdl_wait();
    if (tid == 0) {
        int cum = 0, e_found = -1, m = 0;
        for (int e = 0; e < a.E; ++e) {
            const int lo = a.offsets[e], hi = a.offsets[e + 1];
            if (hi < lo || lo < 0 || hi > a.P) {
                report(a.dev_status, DEV_ERR_INDEX);
                break;
            }
            const int mt = (hi - lo + FB - 1) / FB;
            if ((int)blockIdx.x < cum + mt) {
                e_found = e;
                m = blockIdx.x - cum;
                break;
            }
            cum += mt;
        }
        s_e = e_found;
        if (e_found >= 0) {
            s_row0 = a.offsets[e_found] + m * FB;
            s_rows = min(FB, a.offsets[e_found + 1] - s_row0);
        }
    }
    __syncthreads();
    const int e = s_e;
    if (e < 0) return;
    const int row0 = s_row0, rows = s_rows;
    const int n0 = blockIdx.y * FB;
    const int ty = tid / 16, tx = tid % 16;
    const float *Be = a.B + (int64_t)e * a.N * a.K;
    const float *B3e = EPI == EPI_SWIGLU ? a.B3 + (int64_t)e * a.N * a.K : nullptr;

    float acc[4][4], acc3[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = acc3[i][j] = 0.f;

    const int lr = tid / 4, lk = (tid % 4) * 4;  // loader: row (or column) and K offset
    for (int k0 = 0; k0 < a.K; k0 += FK) {
        float4 av = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lr < rows) av = *reinterpret_cast<const float4 *>(a.A + (int64_t)(row0 + lr) * a.K + k0 + lk);
        const float4 bv = *reinterpret_cast<const float4 *>(Be + (int64_t)(n0 + lr) * a.K + k0 + lk);
        As[lk + 0][lr] = av.x; As[lk + 1][lr] = av.y; As[lk + 2][lr] = av.z; As[lk + 3][lr] = av.w;
        Bs[lk + 0][lr] = bv.x; Bs[lk + 1][lr] = bv.y; Bs[lk + 2][lr] = bv.z; Bs[lk + 3][lr] = bv.w;
        if (EPI == EPI_SWIGLU) {
            const float4 cv = *reinterpret_cast<const float4 *>(B3e + (int64_t)(n0 + lr) * a.K + k0 + lk);
            B3s[lk + 0][lr] = cv.x; B3s[lk + 1][lr] = cv.y; B3s[lk + 2][lr] = cv.z; B3s[lk + 3][lr] = cv.w;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < FK; ++kk) {
            float x[4], w[4], w3[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] = As[kk][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                w[j] = Bs[kk][tx + 16 * j];
                if (EPI == EPI_SWIGLU) w3[j] = B3s[kk][tx + 16 * j];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] = fmaf(x[i], w[j], acc[i][j]);
                    if (EPI == EPI_SWIGLU) acc3[i][j] = fmaf(x[i], w3[j], acc3[i][j]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = ty + 16 * i;
        if (r >= rows) continue;
        float *orow = a.out + (int64_t)(row0 + r) * a.N;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx + 16 * j;
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
    pdl_trigger();
}

template <int EPI>
cudaError_t launch_f32(const F32Args &a, int64_t P, cudaStream_t s) {
    const int64_t mtiles = (P + FB - 1) / FB + a.E;
    dim3 grid((unsigned)mtiles, (unsigned)(a.N / FB));
    return launch_pdl(ffn_f32_kernel<EPI>, grid, dim3(256), 0, s, 1, a);
}

}  // namespace

cudaError_t launch_ffn_f32(const moe_config_t &c, const FfnBufs &b, cudaStream_t s) {
    const int64_t P = c.T * c.k;
    if (P == 0) return cudaSuccess;
    F32Args g1{static_cast<const float *>(b.x_perm), static_cast<const float *>(b.W1),
               static_cast<const float *>(b.W3), c.has_bias ? b.b1 : nullptr,
               static_cast<float *>(b.H), b.offsets, b.dev_status, c.E, c.d, c.f, P};
    cudaError_t err = c.act == MOE_ACT_SWIGLU ? launch_f32<EPI_SWIGLU>(g1, P, s)
                                              : launch_f32<EPI_GELU>(g1, P, s);
    if (err != cudaSuccess) return err;
    F32Args g2{static_cast<const float *>(b.H), static_cast<const float *>(b.W2), nullptr,
               c.has_bias ? b.b2 : nullptr, static_cast<float *>(b.y_perm), b.offsets,
               b.dev_status, c.E, c.f, c.d, P};
    return launch_f32<EPI_STORE>(g2, P, s);
}

}  // namespace moe
