// combine.cu -- step 5 of the MoE layer: gate-weighted combine and the auxiliary value.
//
// lensaml.com "Mixture of Experts", Step 3 "Top-k Routing": y = sum g . E(h), the chosen
// experts' outputs blended by their gates. Step 4 "Load Balancing": the auxiliary term
// N . sum_i f_i P_i, with f_i the fraction of routing slots sent to expert i and P_i its mean
// router probability, equal to 1 under uniform routing.
#include "internal.cuh"
#include "layer_dev.cuh"

namespace moe {
namespace {

using namespace dev;

template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
    uint4 v;
    __device__ __forceinline__ void load(const void *p, int64_t i) {
        v = __ldg(reinterpret_cast<const uint4 *>(p) + i);
    }
    __device__ __forceinline__ float get(int q) const {
        const uint32_t w = (&v.x)[q >> 1];
        const uint16_t b = (q & 1) ? (uint16_t)(w >> 16) : (uint16_t)(w & 0xffffu);
        return __bfloat162float(__ushort_as_bfloat16(b));
    }
    static __device__ __forceinline__ void store(void *p, int64_t i, const float *x) {
        uint4 o;
        uint32_t *ow = &o.x;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * q], x[2 * q + 1]);
            ow[q] = *reinterpret_cast<const uint32_t *>(&b);
        }
        reinterpret_cast<uint4 *>(p)[i] = o;
    }
};
template <> struct Vec8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const void *p, int64_t i) {
        a = __ldg(reinterpret_cast<const float4 *>(p) + 2 * i);
        b = __ldg(reinterpret_cast<const float4 *>(p) + 2 * i + 1);
    }
    __device__ __forceinline__ float get(int q) const {
        return q < 4 ? (&a.x)[q] : (&b.x)[q - 4];
    }
    static __device__ __forceinline__ void store(void *p, int64_t i, const float *x) {
        reinterpret_cast<float4 *>(p)[2 * i] = make_float4(x[0], x[1], x[2], x[3]);
        reinterpret_cast<float4 *>(p)[2 * i + 1] = make_float4(x[4], x[5], x[6], x[7]);
    }
};

constexpr int CB_THREADS = 256;
constexpr int CB_SLOTS = 1024;  // slot entries a block stages in shared memory

// y[t, :] = sum_{j<k} gates[t, j] * y_perm[slot_of[t k + j], :]. A block takes tpb consecutive
// tokens: their slot indices and gates go to shared memory first (checked once), then one thread
// per (token, 8-element vector) sums its rows with f32 FMA in j order and one rounding, the slots
// in groups of 4 whose row loads are issued together.
template <typename VT>
__global__ void __launch_bounds__(CB_THREADS) combine_kernel(const void *__restrict__ y_perm,
                                                             const int32_t *__restrict__ slot_of,
                                                             const float *__restrict__ gates,
                                                             void *__restrict__ y, int64_t T,
                                                             int64_t P, int d, int k, int tpb,
                                                             uint32_t *dev_status) {
    __shared__ int32_t s_row[CB_SLOTS];
    __shared__ float s_g[CB_SLOTS];
    pdl_wait();
    const int v8 = d / 8;
    const int64_t t0 = (int64_t)blockIdx.x * tpb;
    const int nt = (int)(T - t0 < tpb ? T - t0 : tpb);
    const int ns = nt * k;
    for (int q = threadIdx.x; q < ns; q += CB_THREADS) {
        int32_t r = __ldg(slot_of + t0 * k + q);
        if (r != -1 && (r < 0 || r >= P)) {  // -1: dropped by the capacity
            report(dev_status, DEV_ERR_INDEX);
            r = -1;
        }
        s_row[q] = r;
        s_g[q] = __ldg(gates + t0 * k + q);
    }
    __syncthreads();
    const int units = nt * v8;
    for (int u = threadIdx.x; u < units; u += CB_THREADS) {
        const int tl = u / v8, i = u - tl * v8;
        const int32_t *rows = s_row + tl * k;
        const float *gs = s_g + tl * k;
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.f;
        for (int j0 = 0; j0 < k; j0 += 4) {
            Vec8<VT> v[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                if (j0 + jj < k && rows[j0 + jj] >= 0)
                    v[jj].load(y_perm, (int64_t)rows[j0 + jj] * v8 + i);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                if (j0 + jj < k && rows[j0 + jj] >= 0) {
                    const float g = gs[j0 + jj];
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[q] = fmaf(g, v[jj].get(q), acc[q]);
                }
        }
        Vec8<VT>::store(y, (t0 + tl) * v8 + i, acc);
    }
    pdl_trigger();
}

__global__ void __launch_bounds__(1024) aux_kernel(const int32_t *__restrict__ counts,
                                                   const float *__restrict__ psum, int64_t rows,
                                                   int E, int64_t T, int k, float *aux_out,
                                                   float *zloss_out) {
    __shared__ float part[1024];
    __shared__ float colsum[257];
    __shared__ int32_t s_counts[256];
    pdl_wait();
    aux_block(counts, psum, rows, E, T, k, aux_out, zloss_out, part, colsum, s_counts);
    pdl_trigger();
}

// One step of the selection-only routing bias: b[e] += gamma when expert e received fewer routing
// slots than the mean T k / E, -= gamma when more (compared exactly: counts[e] E against T k).
__global__ void update_sel_bias_kernel(const int32_t *__restrict__ counts, float *b, int E,
                                       int64_t slots, float gamma) {
    pdl_wait();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e < E) {
        const int64_t ce = (int64_t)counts[e] * E;
        if (ce < slots) b[e] += gamma;
        else if (ce > slots) b[e] -= gamma;
    }
    pdl_trigger();
}

}  // namespace

cudaError_t launch_combine(const moe_config_t &c, const void *y_perm, const int32_t *slot_of,
                           const float *gates, void *y, uint32_t *dev_status, cudaStream_t s) {
    if (c.T == 0) return cudaSuccess;
    // about 8 (token, vector) units per thread, within the staged slot budget, and at least
    // about two blocks per SM when there are enough tokens
    int64_t tpb = 8 * CB_THREADS / (c.d / 8);
    if (tpb > c.T / (2 * num_sms())) tpb = c.T / (2 * num_sms());
    if (tpb < 1) tpb = 1;
    if (tpb * c.k > CB_SLOTS) tpb = CB_SLOTS / c.k;
    const int64_t blocks = (c.T + tpb - 1) / tpb;
    const int64_t P = c.T * c.k;
    const dim3 grid((unsigned)blocks), block(CB_THREADS);
    if (c.dtype == MOE_BF16)
        return launch_pdl(combine_kernel<__nv_bfloat16>, grid, block, 0, s, 1, y_perm, slot_of,
                          gates, y, c.T, P, c.d, c.k, (int)tpb, dev_status);
    return launch_pdl(combine_kernel<float>, grid, block, 0, s, 1, y_perm, slot_of, gates, y, c.T,
                      P, c.d, c.k, (int)tpb, dev_status);
}

cudaError_t launch_aux(const moe_config_t &c, const int32_t *counts, const float *psum_part,
                       float *aux_out, float *zloss_out, cudaStream_t s) {
    if (c.T == 0) {
        cudaError_t err = cudaMemsetAsync(aux_out, 0, sizeof(float), s);
        if (err == cudaSuccess && zloss_out) err = cudaMemsetAsync(zloss_out, 0, sizeof(float), s);
        return err;
    }
    return launch_pdl(aux_kernel, dim3(1), dim3(1024), 0, s, 1, counts, psum_part,
                      router_partial_rows(c), c.E, c.T, c.k, aux_out, zloss_out);
}

cudaError_t launch_update_sel_bias(const moe_config_t &c, const int32_t *counts, float *sel_bias,
                                   float gamma, cudaStream_t s) {
    return launch_pdl(update_sel_bias_kernel, dim3((c.E + 255) / 256), dim3(256), 0, s, 1, counts,
                      sel_bias, c.E, c.T * (int64_t)c.k, gamma);
}

}  // namespace moe
