// gemm_tc.cu -- step 4 of the MoE layer on the 5th-generation tensor cores (bf16 workloads).
//
// Every expert e is an MLP over its contiguous block of permuted rows [offsets[e], offsets[e+1])
// (llm.curionode.com "Mixture of Experts.", "Workshop"; lensaml.com "Mixture of Experts", Step 1
// and Step 6: a full expert is three d x f matrices; Step 5: dropless grouping of any number of
// tokens per expert):
//   GEMM1  SwiGLU : H[r, n] = SiLU(x_r . W1_e[n]) * (x_r . W3_e[n])      (bf16 out)
//          GELU   : H[r, n] = GELU_tanh(x_r . W1_e[n] + b1_e[n])          (bf16 out)
//   GEMM2         : y_perm[r, o] = H_r . W2_e[o] (+ b2_e[o])              (bf16 out)
// Both are "A times B-transposed" with A and B K-contiguous, which is exactly the K-major operand
// form of tcgen05.mma.
//
// Kernel design (one persistent CTA per SM, 192 threads, static round-robin tile schedule):
//   warp 0      TMA producer: 2-D tiled bulk copies (128-byte swizzle) of a 128 x 64 A tile and
//               a 256 x 64 B tile (SwiGLU: 128 rows of W1 stacked on 128 rows of W3) into a
//               4-stage shared-memory ring, signalling mbarriers with transaction counts.
//   warp 1      MMA issuer (one thread): tcgen05.mma.cta_group::1.kind::f16, M = 128, N = 256,
//               K = 16, f32 accumulation in tensor memory; tcgen05.commit releases a ring stage
//               when its MMAs have read it, and hands a finished accumulator to the epilogue.
//               Warp 1 also owns the 512-column TMEM allocation (two 128 x 256 f32 accumulators,
//               so the epilogue of tile i overlaps the MMAs of tile i + 1).
//   warps 2-9   epilogue, two warps per TMEM lane quarter (each converts half of the tile's
//               columns): tcgen05.ld of the thread's accumulator row (TMEM lane = row), bias /
//               GELU / SwiGLU in f32 on the special-function unit, round to bf16, masked 16-byte
//               stores.
// Tile order: expert-major, then N tile, then M tile, so the CTAs in flight at any moment share a
// few weight tiles (read once from HBM, then from L2) and one expert's activations.
// Rows of an expert's last M tile that belong to the next expert (or lie past the end, which TMA
// fills with zeros) are computed and masked at the store.
// Every mbarrier wait is bounded by %globaltimer: on expiry the CTA records DEV_ERR_TIMEOUT,
// stops issuing, waits (bounded) for its own copies and MMAs, frees TMEM and returns.
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = GEMM_BM, BN = 256, BK = 64, STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;  // 16 KiB
constexpr int B_STAGE = BN * BK * 2;  // 32 KiB
constexpr int TC_THREADS = 320;   // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr uint32_t TMEM_COLS = 512;
constexpr int CTL_BYTES = 4096;
constexpr size_t TC_SMEM = 1024 + (size_t)STAGES * (A_STAGE + B_STAGE) + CTL_BYTES;

enum { EPI_STORE = 0, EPI_GELU = 1, EPI_SWIGLU = 2 };

struct TcArgs {
    const int32_t *offsets;  // [E+1]
    const float *bias;       // [E, N] or null
    __nv_bfloat16 *out;      // [P, N]
    uint32_t *dev_status;
    int64_t P;
    int E, K, N, n_tiles, epi;
    unsigned long long spin_limit_ns;  // bound of every mbarrier wait
    int withhold_loads;                // test hook: the producer issues no loads
};

struct Tile {
    int e, n, row0, rows;
};
// Tile t of the schedule: s_cum[e] is the first tile of expert e (E+1 entries); within an
// expert, tiles run N-major, M-minor. eh is a cursor that only moves forward.
__device__ __forceinline__ Tile decode_tile(int t, int &eh, const int32_t *s_cum,
                                            const int32_t *s_off, int n_tiles) {
    while (s_cum[eh + 1] <= t) ++eh;
    const int e = eh;
    const int local = t - s_cum[e];
    const int mt = (s_cum[e + 1] - s_cum[e]) / n_tiles;
    const int n = local / mt;
    const int m = local - n * mt;
    Tile ti;
    ti.e = e;
    ti.n = n;
    ti.row0 = s_off[e] + m * BM;
    ti.rows = min(BM, s_off[e + 1] - ti.row0);
    return ti;
}

__global__ void __launch_bounds__(TC_THREADS, 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmB3, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + STAGES * A_STAGE;
    uint8_t *ctl = gbase + STAGES * (A_STAGE + B_STAGE);
    const uint32_t bar0 = smem_u32(ctl);
    // barriers: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
    const uint32_t bar_full = bar0, bar_empty = bar0 + 8 * STAGES;
    const uint32_t bar_tfull = bar0 + 16 * STAGES, bar_tempty = bar_tfull + 16;
    const uint32_t bar_drain = bar_tempty + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctl + 256);
    volatile int *s_abort = reinterpret_cast<volatile int *>(ctl + 260);
    int32_t *s_cum = reinterpret_cast<int32_t *>(ctl + 512);   // [E+1]
    int32_t *s_off = s_cum + 260;                             // [E+1]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(bar_tfull + 8 * q, 1);
            mbar_init(bar_tempty + 8 * q, 256);
        }
        mbar_init(bar_drain, 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 2 && lane == 0) {
        int cum = 0;
        bool bad = false;
        for (int e = 0; e < E; ++e) {
            const int lo = a.offsets[e], hi = a.offsets[e + 1];
            if (lo < 0 || hi < lo || (int64_t)hi > a.P) bad = true;
            s_off[e] = lo;
            s_cum[e] = cum;
            if (!bad) cum += ((hi - lo + BM - 1) / BM) * a.n_tiles;
        }
        s_off[E] = a.offsets[E];
        s_cum[E] = cum;
        if (bad) {
            report(a.dev_status, DEV_ERR_INDEX);
            for (int e = 0; e <= E; ++e) s_cum[e] = 0;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = s_cum[E];
    const int nk = a.K / BK;
    const unsigned long long lim = a.spin_limit_ns;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0, eh = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, last_phase = 0;  // per-stage bits
            bool ok = !a.withhold_loads;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile ti = decode_tile(t, eh, s_cum, s_off, a.n_tiles);
                const int brow = ti.e * a.N + ti.n * (a.epi == EPI_SWIGLU ? BN / 2 : BN);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, s_abort, a.dev_status, lim)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar_full + 8 * stage;
                    mbar_expect_tx(fb, A_STAGE + B_STAGE);
                    tma_load_2d(sA + stage * A_STAGE, &tmA, fb, kb * BK, ti.row0);
                    if (a.epi == EPI_SWIGLU) {
                        tma_load_2d(sB + stage * B_STAGE, &tmB, fb, kb * BK, brow);
                        tma_load_2d(sB + stage * B_STAGE + B_STAGE / 2, &tmB3, fb, kb * BK, brow);
                    } else {
                        tma_load_2d(sB + stage * B_STAGE, &tmB, fb, kb * BK, brow);
                    }
                    issued |= 1u << stage;
                    last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Our own copies must have landed before the CTA may exit.
            for (int s = 0; s < STAGES; ++s)
                if ((issued >> s) & 1u)
                    mbar_wait(bar_full + 8 * s, (last_phase >> s) & 1u, nullptr, a.dev_status, lim);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, aphase = 0;
            bool ok = true;
            constexpr uint32_t idesc = idesc_bf16(BM, BN);
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (!mbar_wait(bar_tempty + 8 * acc, aphase ^ 1u, s_abort, a.dev_status, lim)) break;
                tc_fence_after();
                const uint32_t dt = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(bar_full + 8 * stage, phase, s_abort, a.dev_status, lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_k_sw128(sA + stage * A_STAGE);
                    const uint64_t bd = sdesc_k_sw128(sB + stage * B_STAGE);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16(dt, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
                    umma_commit(bar_empty + 8 * stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(bar_tfull + 8 * acc);
                acc ^= 1;
                if (acc == 0) aphase ^= 1u;
            }
            // Every MMA this thread issued has completed once the drain barrier fires.
            umma_commit(bar_drain);
            mbar_wait(bar_drain, 0, nullptr, a.dev_status, lim);
        }
    } else {
        const int q = warp & 3;           // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;  // which half of the tile's columns it converts
        const int r = q * 32 + lane;
        int acc = 0, eh = 0;
        uint32_t aphase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const Tile ti = decode_tile(t, eh, s_cum, s_off, a.n_tiles);
            int ok = 1;
            if (lane == 0) ok = mbar_wait(bar_tfull + 8 * acc, aphase, s_abort, a.dev_status, lim);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            __syncwarp();
            tc_fence_after();
            const bool valid = r < ti.rows;
            const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            __nv_bfloat16 *orow = a.out + (int64_t)(ti.row0 + r) * a.N;
            if (a.epi == EPI_SWIGLU) {
#pragma unroll 1
                for (int c = half * (BN / 4); c < (half + 1) * (BN / 4); c += 32) {
                    float x1[32], x3[32];
                    tmem_ld32x2(trow + c, trow + BN / 2 + c, x1, x3);
                    const int col = ti.n * (BN / 2) + c;
                    if (valid && col < a.N) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack_bf16(silu_fast(x1[2 * i]) * x3[2 * i],
                                              silu_fast(x1[2 * i + 1]) * x3[2 * i + 1]);
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + col);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
            } else {
#pragma unroll 1
                for (int c = half * (BN / 2); c < (half + 1) * (BN / 2); c += 32) {
                    const int col = ti.n * BN + c;
                    if (col >= a.N) break;  // warp-uniform
                    float v[32];
                    tmem_ld32(trow + c, v);
                    if (a.bias) {
                        const float *bp = a.bias + (int64_t)ti.e * a.N + col;
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] += __ldg(bp + i);
                    }
                    if (a.epi == EPI_GELU) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = gelu_tanh_fast(v[i]);
                    }
                    if (valid) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + col);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pack_bf16(v[8 * i], v[8 * i + 1]),
                                                pack_bf16(v[8 * i + 2], v[8 * i + 3]),
                                                pack_bf16(v[8 * i + 4], v[8 * i + 5]),
                                                pack_bf16(v[8 * i + 6], v[8 * i + 7]));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar_tempty + 8 * acc);
            acc ^= 1;
            if (acc == 0) aphase ^= 1u;
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------------------------
// host side

cudaError_t launch_gemm(const void *A, const void *B, const void *B3, int64_t P, int E, int K,
                        int N, int epi, const int32_t *offsets, const float *bias, void *out,
                        uint32_t *dev_status, const FaultHook &hook, cudaStream_t s) {
    const int b_rows = epi == EPI_SWIGLU ? BN / 2 : BN;
    CUtensorMap mA, mB, mB3;
    if (!make_map(&mA, A, P, K, BM)) return cudaErrorInvalidValue;
    if (!make_map(&mB, B, (int64_t)E * N, K, b_rows)) return cudaErrorInvalidValue;
    if (!make_map(&mB3, epi == EPI_SWIGLU ? B3 : B, (int64_t)E * N, K, b_rows))
        return cudaErrorInvalidValue;
    TcArgs a;
    a.offsets = offsets;
    a.bias = bias;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.dev_status = dev_status;
    a.P = P;
    a.E = E;
    a.K = K;
    a.N = N;
    a.n_tiles = (N + b_rows - 1) / b_rows;
    a.epi = epi;
    a.spin_limit_ns = hook.spin_limit_ns;
    a.withhold_loads = hook.withhold;
    const int64_t upper = ((P + BM - 1) / BM + E) * (int64_t)a.n_tiles;
    int64_t grid = num_sms();
    if (grid > upper) grid = upper;
    cudaError_t err = set_max_dynamic_smem((const void *)grouped_gemm_tc_kernel, TC_SMEM);
    if (err != cudaSuccess) return err;
    grouped_gemm_tc_kernel<<<(unsigned)grid, TC_THREADS, TC_SMEM, s>>>(mA, mB, mB3, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffn_tc(const moe_config_t &c, const FfnBufs &b, cudaStream_t s,
                          const FaultHook &hook) {
    const int64_t P = c.T * c.k;
    if (P == 0) return cudaSuccess;
    const bool swiglu = c.act == MOE_ACT_SWIGLU;
    cudaError_t err = launch_gemm(b.x_perm, b.W1, b.W3, P, c.E, c.d, c.f,
                                  swiglu ? EPI_SWIGLU : EPI_GELU, b.offsets,
                                  c.has_bias ? b.b1 : nullptr, b.H, b.dev_status, hook, s);
    if (err != cudaSuccess) return err;
    return launch_gemm(b.H, b.W2, nullptr, P, c.E, c.f, c.d, EPI_STORE, b.offsets,
                       c.has_bias ? b.b2 : nullptr, b.y_perm, b.dev_status, hook, s);
}

}  // namespace moe
