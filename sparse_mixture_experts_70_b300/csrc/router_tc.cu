// router_tc.cu -- steps 1-2 of the MoE layer on the tensor cores, for bf16 h and E <= 128.
//
// The router logits z = h . W_r (lensaml.com "Mixture of Experts", Step 2) are a dense
// [T, d] x [d, E] contraction; with E of 64-128 it is far too much f32 arithmetic for the CUDA
// cores (2 d E flop per token), so it runs as a tcgen05 GEMM; for small E it is a bandwidth-bound
// stream of h that the TMA ring feeds at full rate. The router stays f32-accurate
// (arjunjaggi.com "Mixture of Experts in LLMs", "Switch Transformers": router in float32):
//   W_r (f32) is split exactly into three bf16 pieces, w = w_hi + w_mid + w_lo (each piece keeps
//   the next 8 significant bits of the remainder; 3 x 8 bits cover f32's 24), and
//   z = h . w_hi + h . w_mid + h . w_lo, all three accumulated into one f32 TMEM accumulator.
//   Since h is bf16, every product h_i * piece is exact in f32; only the f32 accumulation rounds,
//   as it does for an FMA chain.
// router_split_kernel writes the pieces, transposed to K-major [3][Epad][d] (Epad = E rounded up
// to 16, zero rows beyond E), into the caller's workspace. router_tc_kernel is persistent over
// tiles of 128 tokens: warp 0 streams 128 x 64 tiles of h and the three 64-wide piece tiles by
// TMA into a shared-memory ring, warp 1 issues 3 x 4 MMAs (M = 128, N = Epad, K = 16) per stage
// into one of two TMEM accumulators, and warps 2-5 -- one thread per token, the token's logits in
// its TMEM lane, read back 32 columns at a time -- add the bias and do the softmax, the top-k
// (k passes of arg-max, larger logit first, lower index on equal logits), the gates, and the
// tile's per-expert sums of p (in token order, through shared memory) while the next tile's MMAs
// run.
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int RB = ROUTER_TC_TOKENS;  // tokens per CTA (MMA M)
constexpr int RK = 64;                // K per stage (one 128-byte swizzle row of bf16)
constexpr int R_THREADS = 192;
constexpr int R_CTL = 2048;
constexpr size_t R_SMEM_BUDGET = 200 * 1024;

inline int epad_of(int E) { return (E + 15) / 16 * 16; }

struct RouterTcArgs {
    const float *b_r;
    int32_t *idx;
    float *gates, *psum;
    uint32_t *dev_status;
    int64_t T;
    int d, E, Epad, k, gate_mode, stages;
};

__global__ void router_split_kernel(const float *__restrict__ W_r, __nv_bfloat16 *__restrict__ out,
                                    int d, int E, int Epad) {
    __shared__ float tile[32][33];
    const int i0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;
    for (int r = ty; r < 32; r += 8) {
        const int i = i0 + r, e = e0 + tx;
        tile[r][tx] = (i < d && e < E) ? W_r[(int64_t)i * E + e] : 0.f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int e = e0 + r, i = i0 + tx;
        if (e < Epad && i < d) {
            const float w = tile[tx][r];
            const __nv_bfloat16 hi = __float2bfloat16_rn(w);
            const float r1 = w - __bfloat162float(hi);
            const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
            const float r2 = r1 - __bfloat162float(mid);
            const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
            const int64_t plane = (int64_t)Epad * d;
            out[(int64_t)e * d + i] = hi;
            out[plane + (int64_t)e * d + i] = mid;
            out[2 * plane + (int64_t)e * d + i] = lo;
        }
    }
}

template <int NCH>  // logits per token handled as NCH chunks of 32 (32 * NCH >= Epad)
__global__ void __launch_bounds__(R_THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmH,
                     const __grid_constant__ CUtensorMap tmW, const RouterTcArgs a) {
    constexpr int NZ = 32 * NCH;
    constexpr uint32_t ACC_COLS = NZ <= 32 ? 32 : (NZ <= 64 ? 64 : 128);
    constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;  // two accumulators: epilogue overlaps MMAs
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int S = a.stages, Epad = a.Epad, E = a.E;
    const uint32_t A_ST = RB * RK * 2;                  // 16 KiB
    const uint32_t P_ST = (uint32_t)Epad * RK * 2;      // one piece tile
    const uint32_t ST = A_ST + 3 * P_ST;
    float *pbuf = reinterpret_cast<float *>(gbase + (size_t)S * ST);  // [RB][NZ + 1]
    float *sinv = pbuf + RB * (NZ + 1);                                 // [RB]
    uint8_t *ctl = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(sinv + RB) + 255) & ~static_cast<uintptr_t>(255));
    const uint32_t bar0 = smem_u32(ctl);
    const uint32_t bar_full = bar0, bar_empty = bar0 + 8 * 8;
    const uint32_t bar_tfull = bar0 + 16 * 8, bar_tempty = bar_tfull + 16;
    const uint32_t bar_drain = bar_tempty + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctl + 256);
    volatile int *s_abort = reinterpret_cast<volatile int *>(ctl + 260);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = a.d / RK;
    const int ntiles = (int)((a.T + RB - 1) / RB);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(bar_tfull + 8 * q, 1);
            mbar_init(bar_tempty + 8 * q, 128);
        }
        mbar_init(bar_drain, 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, last_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, s_abort, a.dev_status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar_full + 8 * stage;
                    const uint32_t dst = base + stage * ST;
                    mbar_expect_tx(fb, ST);
                    tma_load_2d(dst, &tmH, fb, kb * RK, tile * RB);
#pragma unroll
                    for (int p = 0; p < 3; ++p)
                        tma_load_2d(dst + A_ST + p * P_ST, &tmW, fb, kb * RK, p * Epad);
                    issued |= 1u << stage;
                    last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < S; ++s)
                if ((issued >> s) & 1u)
                    mbar_wait(bar_full + 8 * s, (last_phase >> s) & 1u, nullptr, a.dev_status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, aphase = 0;
            bool ok = true;
            const uint32_t idesc = idesc_bf16(RB, Epad);
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                if (!mbar_wait(bar_tempty + 8 * acc, aphase ^ 1u, s_abort, a.dev_status)) break;
                tc_fence_after();
                const uint32_t dt = tmem_base + (uint32_t)acc * ACC_COLS;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(bar_full + 8 * stage, phase, s_abort, a.dev_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = base + stage * ST;
                    const uint64_t ad = sdesc_k_sw128(st);
#pragma unroll
                    for (int p = 0; p < 3; ++p) {
                        const uint64_t bd = sdesc_k_sw128(st + A_ST + p * P_ST);
#pragma unroll
                        for (int kk = 0; kk < RK / 16; ++kk)
                            umma_bf16(dt, ad + 2 * kk, bd + 2 * kk, idesc,
                                      (kb | p | kk) != 0 ? 1u : 0u);
                    }
                    umma_commit(bar_empty + 8 * stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(bar_tfull + 8 * acc);
                acc ^= 1;
                if (acc == 0) aphase ^= 1u;
            }
            umma_commit(bar_drain);
            mbar_wait(bar_drain, 0, nullptr, a.dev_status);
        }
    } else {
        const int q = warp & 3;
        const int r = q * 32 + lane;
        int acc = 0;
        uint32_t aphase = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            const int64_t tok = (int64_t)tile * RB + r;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(bar_tfull + 8 * acc, aphase, s_abort, a.dev_status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            __syncwarp();
            tc_fence_after();
            const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * ACC_COLS;
            const bool valid = tok < a.T;
            // pass 1: maximum logit (with bias); pass 2: exp(z - zmax) into this row of pbuf
            float zmax = -INFINITY;
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                float v[32];
                tmem_ld32(trow + 32 * ch, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int e = 32 * ch + i;
                    if (e < E) zmax = fmaxf(zmax, v[i] + (a.b_r ? __ldg(a.b_r + e) : 0.f));
                }
            }
            float ssum = 0.f;
            float *prow = pbuf + r * (NZ + 1);
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                float v[32];
                tmem_ld32(trow + 32 * ch, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int e = 32 * ch + i;
                    const float ex =
                        e < E ? __expf(v[i] + ((a.b_r && e < E) ? __ldg(a.b_r + e) : 0.f) - zmax)
                              : 0.f;
                    ssum += ex;
                    prow[e] = ex;
                }
            }
            {
                // k passes of arg-max over the logits (larger first, lower index on ties). Every
                // lane runs them -- tcgen05.ld is warp-collective -- and only valid rows store.
                uint32_t chosen[NCH];
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) chosen[ch] = 0;
                float gsum = 0.f;
                for (int j = 0; j < a.k; ++j) {
                    float bv = -INFINITY;
                    int be = 0;
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        float v[32];
                        tmem_ld32(trow + 32 * ch, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int e = 32 * ch + i;
                            const float z = v[i] + ((a.b_r && e < E) ? __ldg(a.b_r + e) : 0.f);
                            if (e < E && !((chosen[ch] >> i) & 1u) && z > bv) {
                                bv = z;
                                be = e;
                            }
                        }
                    }
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch)
                        if (ch == (be >> 5)) chosen[ch] |= 1u << (be & 31);
                    if (valid) a.idx[tok * a.k + j] = be;
                    gsum += prow[be];
                }
                if (valid) {
                    const float inv = 1.f / (a.gate_mode == MOE_GATE_RAW_PROB ? ssum : gsum);
                    for (int j = 0; j < a.k; ++j)
                        a.gates[tok * a.k + j] = prow[a.idx[tok * a.k + j]] * inv;
                }
            }
            tc_fence_before();
            mbar_arrive(bar_tempty + 8 * acc);  // TMEM no longer read for this tile
            sinv[r] = valid ? 1.f / ssum : 0.f;
            asm volatile("bar.sync 1, 128;" ::: "memory");
            // per-expert sums of p over this tile's tokens, in token order
            if (r < E) {
                float s = 0.f;
                for (int t = 0; t < RB; ++t) s += pbuf[t * (NZ + 1) + r] * sinv[t];
                a.psum[(int64_t)tile * E + r] = s;
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            acc ^= 1;
            if (acc == 0) aphase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int NCH>
cudaError_t launch_nch(const CUtensorMap &mh, const CUtensorMap &mw, const RouterTcArgs &a,
                       int64_t blocks, size_t smem, cudaStream_t s) {
    auto kern = router_tc_kernel<NCH>;
    cudaError_t err = set_max_dynamic_smem((const void *)kern, smem);
    if (err != cudaSuccess) return err;
    kern<<<(unsigned)blocks, R_THREADS, smem, s>>>(mh, mw, a);
    return cudaGetLastError();
}

}  // namespace

size_t router_tc_scratch_bytes(const moe_config_t &c) {
    return (size_t)3 * epad_of(c.E) * c.d * 2;
}

cudaError_t launch_router_tc(const moe_config_t &c, const void *h, const float *W_r,
                             const float *b_r, int32_t *topk_idx, float *gates, float *psum_part,
                             void *scratch, uint32_t *dev_status, cudaStream_t s) {
    const int Epad = epad_of(c.E);
    auto *pieces = static_cast<__nv_bfloat16 *>(scratch);
    dim3 sg((c.d + 31) / 32, (Epad + 31) / 32);
    router_split_kernel<<<sg, dim3(32, 8), 0, s>>>(W_r, pieces, c.d, c.E, Epad);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    CUtensorMap mh, mw;
    if (!make_map(&mh, h, c.T, c.d, RB)) return cudaErrorInvalidValue;
    if (!make_map(&mw, pieces, (int64_t)3 * Epad, c.d, Epad)) return cudaErrorInvalidValue;
    RouterTcArgs a;
    a.b_r = b_r;
    a.idx = topk_idx;
    a.gates = gates;
    a.psum = psum_part;
    a.dev_status = dev_status;
    a.T = c.T;
    a.d = c.d;
    a.E = c.E;
    a.Epad = Epad;
    a.k = c.k;
    a.gate_mode = c.gate;
    const int nch = (Epad + 31) / 32;
    const size_t stage = (size_t)RB * RK * 2 + (size_t)3 * Epad * RK * 2;
    const size_t pbuf = (size_t)RB * (32 * nch + 1) * 4 + (size_t)RB * 4;
    int stages = (int)((R_SMEM_BUDGET - R_CTL - 1024 - pbuf) / stage);
    if (stages > 8) stages = 8;
    if (stages < 2) stages = 2;
    a.stages = stages;
    const size_t smem = 1024 + (size_t)stages * stage + pbuf + R_CTL;
    const int64_t tiles = (c.T + RB - 1) / RB;
    const int64_t blocks = tiles < num_sms() ? tiles : num_sms();
    switch (nch) {
        case 1: return launch_nch<1>(mh, mw, a, blocks, smem, s);
        case 2: return launch_nch<2>(mh, mw, a, blocks, smem, s);
        case 3: return launch_nch<3>(mh, mw, a, blocks, smem, s);
        default: return launch_nch<4>(mh, mw, a, blocks, smem, s);
    }
}

}  // namespace moe
