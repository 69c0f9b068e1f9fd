// router_tc.cu -- the router logits of the MoE layer on the tensor cores, for bf16 h and E <= 128.
//
// The router logits z = h . W_r (lensaml.com "Mixture of Experts", Step 2) are a dense
// [T, d] x [d, E] contraction; with E of 64-128 it is far too much f32 arithmetic for the CUDA
// cores (2 d E flop per token), and for small E it is a bandwidth-bound stream of h. The router
// stays f32-accurate (arjunjaggi.com "Mixture of Experts in LLMs", "Switch Transformers": router
// in float32):
//   W_r (f32) is split exactly into three bf16 pieces, w = w_hi + w_mid + w_lo (each piece keeps
//   the next 8 significant bits of the remainder; 3 x 8 bits cover f32's 24), and
//   z = h . w_hi + h . w_mid + h . w_lo with f32 accumulation. Since h is bf16, every product
//   h_i * piece is exact in f32; only the f32 accumulation rounds, as it does for an FMA chain.
// router_split_kernel writes the pieces, transposed to K-major [3][Epad][d] (Epad = E rounded up
// to 16, zero rows beyond E), into the caller's workspace.
//
// router_logits_kernel computes f32 partial logits zpart[s][t][e] over K chunk s of d. Work items
// are (128-token tile, K chunk) pairs, taken by persistent CTAs; the number of K chunks is chosen
// so that small token counts still spread over the SMs. Per 64-wide K stage, warp 0 streams the
// h tile and the three piece tiles by TMA; warp 1 issues, for each of the 4 K = 16 steps, one MMA
// with N = 3 Epad (hi | mid | lo side by side; two MMAs when 3 Epad > 256). Consecutive K steps
// rotate over up to 4 independent accumulators ("chains") so that dependent MMAs do not
// serialise (an MMA of N = 16-48 is far shorter than its latency). Warps 2-5 (one thread per
// token) add the chains and the three pieces of each logit in a fixed order and store the
// partial logits; with two TMEM buffers that overlaps the next item's MMAs. Softmax, top-k and
// gates follow in router_select_kernel (router.cu), warp per token.
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int RB = ROUTER_TC_TOKENS;  // tokens per tile (MMA M)
constexpr int RK = 64;                // K per stage (one 128-byte swizzle row of bf16)
constexpr int L_THREADS = 192;
constexpr int L_CTL = 1024;
constexpr size_t L_SMEM_BUDGET = 200 * 1024;
constexpr int SPLIT_SMS = 148;        // splits are chosen for this many SMs (a pure function)

inline int epad_of(int E) { return (E + 15) / 16 * 16; }

// TMEM plan: columns of one accumulator set (3 Epad), chains per set, buffers.
struct LogitsPlan {
    int Epad, cols, chains, buffers;
};
inline LogitsPlan logits_plan(int E) {
    LogitsPlan p;
    p.Epad = epad_of(E);
    p.cols = 3 * p.Epad;
    p.buffers = p.cols <= 256 ? 2 : 1;
    const int per_buffer = p.buffers == 2 ? 256 : 512;
    p.chains = p.cols * 4 <= per_buffer ? 4 : (p.cols * 2 <= per_buffer ? 2 : 1);
    return p;
}

struct LogitsArgs {
    float *zpart;  // [S][T][Epad]
    uint32_t *dev_status;
    int64_t T;
    int d, Epad, S, chains, buffers, stages;
};

__global__ void router_split_kernel(const float *__restrict__ W_r, __nv_bfloat16 *__restrict__ out,
                                    int d, int E, int Epad) {
    __shared__ float tile[32][33];
    pdl_wait();
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
    pdl_trigger();
}

__global__ void __launch_bounds__(L_THREADS, 1)
    router_logits_kernel(const __grid_constant__ CUtensorMap tmH,
                         const __grid_constant__ CUtensorMap tmW, const LogitsArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int S = a.S, Epad = a.Epad, NS = a.stages;
    const uint32_t A_ST = RB * RK * 2;             // 16 KiB of h
    const uint32_t P_ST = (uint32_t)Epad * RK * 2;  // one piece tile
    const uint32_t ST = A_ST + 3 * P_ST;
    uint8_t *ctl = gbase + (size_t)NS * ST;
    const uint32_t bar0 = smem_u32(ctl);
    const uint32_t bar_full = bar0, bar_empty = bar0 + 8 * 8;
    const uint32_t bar_tfull = bar0 + 16 * 8, bar_tempty = bar_tfull + 16;
    const uint32_t bar_drain = bar_tempty + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctl + 256);
    volatile int *s_abort = reinterpret_cast<volatile int *>(ctl + 260);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();  // h, the W_r pieces and the previous use of zpart come from earlier stream work
    const int nk = a.d / RK;
    const int kps = nk / S;  // K stages per chunk (S divides nk)
    const int ntiles = (int)((a.T + RB - 1) / RB);
    const int items = ntiles * S;
    const int cols = 3 * Epad;
    const uint32_t buf_cols = a.buffers == 2 ? 256u : 512u;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(bar_tfull + 8 * q, 1);
            mbar_init(bar_tempty + 8 * q, 4);
        }
        mbar_init(bar_drain, 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
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
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
                const int tile = it / S, kb0 = (it % S) * kps;
                for (int kb = kb0; kb < kb0 + kps; ++kb) {
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
                    if (++stage == NS) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < NS; ++s)
                if ((issued >> s) & 1u)
                    mbar_wait(bar_full + 8 * s, (last_phase >> s) & 1u, nullptr, a.dev_status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, buf = 0;
            uint32_t phase = 0, bphase = 0;
            bool ok = true;
            const bool two = cols > 256;  // hi | mid in one MMA, lo in a second
            const uint32_t id_all = idesc_bf16(RB, two ? 2 * Epad : cols);
            const uint32_t id_lo = idesc_bf16(RB, Epad);
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
                if (!mbar_wait(bar_tempty + 8 * buf, bphase ^ 1u, s_abort, a.dev_status)) break;
                tc_fence_after();
                const uint32_t dt0 = tmem_base + (uint32_t)buf * buf_cols;
                for (int j = 0; j < kps; ++j) {
                    if (!mbar_wait(bar_full + 8 * stage, phase, s_abort, a.dev_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = base + stage * ST;
                    const uint64_t ad = sdesc_k_sw128(st);
                    const uint64_t bd = sdesc_k_sw128(st + A_ST);
                    const uint64_t bd_lo = sdesc_k_sw128(st + A_ST + 2 * P_ST);
#pragma unroll
                    for (int kk = 0; kk < RK / 16; ++kk) {
                        const int ch = kk % a.chains;
                        const uint32_t dt = dt0 + (uint32_t)(ch * cols);
                        const uint32_t acc = (j > 0 || kk >= a.chains) ? 1u : 0u;
                        umma_bf16(dt, ad + 2 * kk, bd + 2 * kk, id_all, acc);
                        if (two) umma_bf16(dt + 2 * Epad, ad + 2 * kk, bd_lo + 2 * kk, id_lo, acc);
                    }
                    umma_commit(bar_empty + 8 * stage);
                    if (++stage == NS) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(bar_tfull + 8 * buf);
                if (++buf == a.buffers) {
                    buf = 0;
                    bphase ^= 1u;
                }
            }
            umma_commit(bar_drain);
            mbar_wait(bar_drain, 0, nullptr, a.dev_status);
        }
    } else {
        const int q = warp & 3;
        const int r = q * 32 + lane;
        int buf = 0;
        uint32_t bphase = 0;
        for (int it = blockIdx.x; it < items; it += gridDim.x) {
            const int tile = it / S, s = it % S;
            const int64_t tok = (int64_t)tile * RB + r;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(bar_tfull + 8 * buf, bphase, s_abort, a.dev_status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            __syncwarp();
            tc_fence_after();
            const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)buf * buf_cols;
            float *zrow = a.zpart + ((int64_t)s * a.T + tok) * Epad;
            for (int e0 = 0; e0 < Epad; e0 += 16) {
                // z = sum over chains of (hi + (mid + lo)), in that fixed order
                float z[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) z[i] = 0.f;
                for (int ch = 0; ch < a.chains; ++ch) {
                    uint32_t vh[16], vm[16], vl[16];
                    const uint32_t c0 = trow + (uint32_t)(ch * cols + e0);
                    tmem_ld16_nowait(c0, vh);
                    tmem_ld16_nowait(c0 + Epad, vm);
                    tmem_ld16_nowait(c0 + 2 * Epad, vl);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        z[i] += __uint_as_float(vh[i]) +
                                (__uint_as_float(vm[i]) + __uint_as_float(vl[i]));
                }
                if (tok < a.T) {
                    float4 *dst = reinterpret_cast<float4 *>(zrow + e0);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_float4(z[4 * i], z[4 * i + 1], z[4 * i + 2], z[4 * i + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_tempty + 8 * buf);  // TMEM no longer read
            if (++buf == a.buffers) {
                buf = 0;
                bphase ^= 1u;
            }
        }
    }

    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

size_t pieces_bytes(const moe_config_t &c) {
    return ((size_t)3 * epad_of(c.E) * c.d * 2 + 1023) & ~(size_t)1023;
}

}  // namespace

int router_tc_splits(const moe_config_t &c) {
    // split K while the work items still fit in about one wave of SPLIT_SMS SMs and every chunk
    // keeps at least 4 stages of 64
    const int64_t tiles = (c.T + RB - 1) / RB;
    const int nk = c.d / RK;
    int S = 1;
    while (tiles * S * 2 <= SPLIT_SMS && nk % (2 * S) == 0 && nk / (2 * S) >= 4) S *= 2;
    return S;
}

size_t router_tc_scratch_bytes(const moe_config_t &c) {
    return pieces_bytes(c) + (size_t)router_tc_splits(c) * (size_t)c.T * epad_of(c.E) * 4;
}

int router_tc_epad(const moe_config_t &c) { return epad_of(c.E); }

float *router_tc_logits(void *scratch, const moe_config_t &c) {
    return reinterpret_cast<float *>(static_cast<char *>(scratch) + pieces_bytes(c));
}

cudaError_t launch_router_tc(const moe_config_t &c, const void *h, const float *W_r,
                             void *scratch, uint32_t *dev_status, cudaStream_t s) {
    const LogitsPlan plan = logits_plan(c.E);
    const int Epad = plan.Epad;
    auto *pieces = static_cast<__nv_bfloat16 *>(scratch);
    dim3 sg((c.d + 31) / 32, (Epad + 31) / 32);
    cudaError_t err =
        launch_pdl(router_split_kernel, sg, dim3(32, 8), 0, s, 1, W_r, pieces, c.d, c.E, Epad);
    if (err != cudaSuccess) return err;
    CUtensorMap mh, mw;
    if (!make_map(&mh, h, c.T, c.d, RB)) return cudaErrorInvalidValue;
    if (!make_map(&mw, pieces, (int64_t)3 * Epad, c.d, Epad)) return cudaErrorInvalidValue;
    LogitsArgs a;
    a.zpart = router_tc_logits(scratch, c);
    a.dev_status = dev_status;
    a.T = c.T;
    a.d = c.d;
    a.Epad = Epad;
    a.S = router_tc_splits(c);
    a.chains = plan.chains;
    a.buffers = plan.buffers;
    const size_t stage = (size_t)RB * RK * 2 + (size_t)3 * Epad * RK * 2;
    int stages = (int)((L_SMEM_BUDGET - L_CTL - 1024) / stage);
    if (stages > 8) stages = 8;
    if (stages < 2) stages = 2;
    a.stages = stages;
    const size_t smem = 1024 + (size_t)stages * stage + L_CTL;
    const int64_t items = (c.T + RB - 1) / RB * a.S;
    const int64_t blocks = items < num_sms() ? items : num_sms();
    err = set_max_dynamic_smem((const void *)router_logits_kernel, smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(router_logits_kernel, dim3((unsigned)blocks), dim3(L_THREADS), smem, s, 1,
                      mh, mw, a);
}

}  // namespace moe
