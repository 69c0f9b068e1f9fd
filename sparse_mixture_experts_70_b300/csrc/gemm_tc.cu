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
// Two kernels share this design. grouped_gemm_tc_kernel: one persistent CTA per SM, 320 threads,
// static round-robin tile schedule over 128 x 256 output tiles. grouped_gemm_pair_kernel (experts
// of at least four M tiles on average): 2-CTA clusters computing 256 x 256 tiles with
// tcgen05.mma.cta_group::2, each CTA holding half of A and half of B, a 6-stage ring. In both:
//   warp 0      TMA producer: 2-D tiled bulk copies (128-byte swizzle) of a 128 x 64 A tile and
//               a 256 x 64 B tile (SwiGLU: 128 rows of W1 stacked on 128 rows of W3; a pair CTA
//               copies its halves) into the shared-memory ring, signalling mbarriers with
//               transaction counts (the opt-in fused gather reads A rows of h with
//               tile::gather4 instead).
//   warp 1      MMA issuer (one thread; in a pair, the leader CTA's, with cta_group::2 and
//               M = 256): tcgen05.mma.cta_group::1.kind::f16, M = 128, N = 256,
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
// A dropless top-1 GEMM2 may scatter g * row straight into y[token] (fused combine).
// Every mbarrier wait is bounded by %globaltimer: on expiry the CTA records DEV_ERR_TIMEOUT,
// stops issuing, waits (bounded) for its own copies and MMAs, frees TMEM and returns.
#include <atomic>

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
// Output staging of the TMA-store epilogue: one 32-row x 32-column bf16 box (2 KiB) per epilogue
// warp, after the control block.
#ifndef MOE_GEMM_TMA_STORE
#define MOE_GEMM_TMA_STORE 1
#endif
constexpr int EPI_WARPS = 8;
constexpr int EPI_BOX = 32 * 64;
constexpr size_t TC_SMEM =
    1024 + (size_t)STAGES * (A_STAGE + B_STAGE) + CTL_BYTES + (size_t)EPI_WARPS * EPI_BOX;

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
    int tma_out;  // 1: 32-row groups that lie wholly inside a tile's valid rows leave through
                  // shared-memory staging and TMA stores -- 4-row scatters to the rows' tokens
                  // with out_token -- (the other rows: per-thread stores)
    // fused gather (GEMM1): A row r is row a_rows[r] of a [a_src_rows, K] tensor, read with
    // 4-row TMA gathers, instead of row r of a permuted copy
    const int32_t *a_rows;
    int64_t a_src_rows;
    // fused scatter (GEMM2, one expert per token): sorted row r goes to output row
    // out_token[r], scaled by out_gate[out_token[r]]
    const int32_t *out_token;
    const float *out_gate;
    // K-grouped mode (the weight gradients of the backward): unit (e, n, m) is the 128 x 256
    // tile (m, n) of expert e's [M, N] output, rows e M + m 128 of out [E M, N]; it sums A and B
    // columns [offsets[e], offsets[e+1]) -- multiples of 64, zero-padded -- of A [M, K] and
    // B [N, K] (K: the padded width). m_tiles = ceil(M / 128).
    int M, m_tiles;
    // training forward (GEMM1): the pre-activations also go to pre1 (x . W1_e + b1) and, for
    // SwiGLU, pre3 (x . W3_e), [P, N] bf16 each (null: not saved)
    __nv_bfloat16 *pre1, *pre3;
    // MN-major B (kernels instantiated with MN): B is read from a [rows, N] tensor whose rows are
    // the K index, as 64 x 64 boxes; expert e's k-block kb is rows e b_krows + 64 kb of tmB, or,
    // from k-block b_ksplit on (when > 0), rows e b_krows + 64 (kb - b_ksplit) of tmB3 (B is the
    // two tensors stacked along K). In K-grouped mode, rows kseg[e] + 64 kb.
    int b_mn, b_ksplit, b_krows;
    // MN-major A (K-grouped mode with MN): A is [K rows, M] (rows = the K index), read as two
    // 64 x 64 boxes at columns m 128 and m 128 + 64, rows kseg[e] + 64 kb
    int a_mn;
    // f32 output (plain store, no bias or activation): out_f32 [rows, N] instead of out
    float *out_f32;
};

// The 4 source rows this lane gathers for tile ti (rows 4 lane .. 4 lane + 3 of the tile);
// rows past the tile's valid rows read a real row (token 0), computed and never stored.
__device__ __forceinline__ int4 gather_rows(const TcArgs &a, int row0, int rows, int lane) {
    int r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int i = 4 * lane + j;
        int tok = 0;
        if (i < rows) {
            tok = __ldg(a.a_rows + row0 + i);
            if (tok < 0 || (int64_t)tok >= a.a_src_rows) tok = 0;
        }
        r[j] = tok;
    }
    return make_int4(r[0], r[1], r[2], r[3]);
}

struct Tile {
    int e, n, row0, rows;  // rows <= 0: nothing to compute (the idle half of a CTA pair)
};
// Unit t of the K-grouped schedule of a CTA pair: the experts in `order` (longest K segment
// first, so that the units of long experts do not pile up in the last waves when the experts'
// row counts are skewed), then N tile, then pairs of M tiles, of which CTA `rank` takes the first
// or the second (rows <= 0: past M, an idle half).
__device__ __forceinline__ Tile decode_tile_kg_pair(int t, const TcArgs &a, int rank,
                                                    const int32_t *order) {
    const int mp_n = (a.m_tiles + 1) / 2;
    const int per = mp_n * a.n_tiles;
    Tile ti;
    const int q = t / per;
    ti.e = order[q];
    const int local = t - q * per;
    ti.n = local / mp_n;
    const int m = 2 * (local - ti.n * mp_n) + rank;
    ti.row0 = ti.e * a.M + m * BM;
    ti.rows = min(BM, a.M - m * BM);
    return ti;
}
// The experts by K segment length (s_off [E+1]), longest first, ties by index: thread-parallel
// ranks into order [E], the same permutation in every CTA.
__device__ __forceinline__ void kg_order(const int32_t *s_off, int E, int32_t *order) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int len = s_off[e + 1] - s_off[e];
        int r = 0;
        for (int j = 0; j < E; ++j) {
            const int lj = s_off[j + 1] - s_off[j];
            r += (lj > len || (lj == len && j < e)) ? 1 : 0;
        }
        order[r] = e;
    }
}
// Unit t of the K-grouped schedule of one CTA (experts averaging under 512 rows, each unit a few
// K blocks: the longest-first order measured slower here): expert-major, then N tile, then M
// tile; row0 is the output row (e M + m 128), rows the valid rows of the tile.
__device__ __forceinline__ Tile decode_tile_kg(int t, const TcArgs &a) {
    const int per = a.m_tiles * a.n_tiles;
    Tile ti;
    ti.e = t / per;
    const int local = t - ti.e * per;
    ti.n = local / a.m_tiles;
    const int m = local - ti.n * a.m_tiles;
    ti.row0 = ti.e * a.M + m * BM;
    ti.rows = min(BM, a.M - m * BM);
    return ti;
}
// Unit t of the schedule. s_cum[e] is the first unit of expert e (E+1 entries); within an
// expert, units run N-major, M-minor. A unit is one 128-row M tile, or -- for a CTA pair -- two
// adjacent M tiles, of which CTA `rank` takes the first or the second. eh only moves forward.
template <bool PAIR>
__device__ __forceinline__ Tile decode_tile(int t, int &eh, const int32_t *s_cum,
                                            const int32_t *s_off, int n_tiles, int rank) {
    while (s_cum[eh + 1] <= t) ++eh;
    const int e = eh;
    const int local = t - s_cum[e];
    const int mu = (s_cum[e + 1] - s_cum[e]) / n_tiles;
    const int n = local / mu;
    const int m = PAIR ? 2 * (local - n * mu) + rank : local - n * mu;
    Tile ti;
    ti.e = e;
    ti.n = n;
    ti.row0 = s_off[e] + m * BM;
    ti.rows = min(BM, s_off[e + 1] - ti.row0);
    return ti;
}

// 32 f32 values as bf16 at dst (64 bytes, 16-byte aligned).
__device__ __forceinline__ void store_row32(__nv_bfloat16 *dst, const float (&v)[32]) {
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        d[i] = make_uint4(pack_bf16(v[8 * i], v[8 * i + 1]), pack_bf16(v[8 * i + 2], v[8 * i + 3]),
                          pack_bf16(v[8 * i + 4], v[8 * i + 5]),
                          pack_bf16(v[8 * i + 6], v[8 * i + 7]));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// One 32 x 32 output box through this warp's staging buffer `stg`: wait until the previous TMA
// store has read the buffer, write this lane's row (32 bf16 in pk) with the 64-byte swizzle,
// make the writes visible to the async proxy, and let lane 0 issue the store at (col, row0).
__device__ __forceinline__ void stage_and_store(const CUtensorMap *tmO, uint32_t stg,
                                                const uint32_t (&pk)[16], int col, int row0,
                                                int lane) {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
    const uint32_t rowaddr = stg + (uint32_t)lane * 64u;
    const uint32_t sw = (uint32_t)(lane >> 1) & 3u;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        st_shared_v4(rowaddr + (((uint32_t)j ^ sw) << 4), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                     pk[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tmO, stg, col, row0);
        bulk_commit();
    }
}

// The same for the scattering GEMM2: the warp's 32 rows go to output rows tok (one per lane, the
// lane's token), as eight 4-row scatters of the staged box through the one-row-box map tmO.
__device__ __forceinline__ void stage_and_scatter(const CUtensorMap *tmO, uint32_t stg,
                                                  const uint32_t (&pk)[16], int col, int tok,
                                                  int lane) {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
    const uint32_t rowaddr = stg + (uint32_t)lane * 64u;
    const uint32_t sw = (uint32_t)(lane >> 1) & 3u;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        st_shared_v4(rowaddr + (((uint32_t)j ^ sw) << 4), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                     pk[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r0 = __shfl_sync(0xffffffffu, tok, 4 * i);
        const int r1 = __shfl_sync(0xffffffffu, tok, 4 * i + 1);
        const int r2 = __shfl_sync(0xffffffffu, tok, 4 * i + 2);
        const int r3 = __shfl_sync(0xffffffffu, tok, 4 * i + 3);
        if (lane == 0) tma_scatter4(tmO, stg + (uint32_t)i * 256u, col, r0, r1, r2, r3);
    }
    if (lane == 0) bulk_commit();
}

// Convert this thread's accumulator row (TMEM lane q*32+lane of accumulator `acc_col`) of tile
// ti into bf16 outputs: half the tile's columns per thread (`half`), bias / GELU / SwiGLU in f32.
// Every tcgen05.ld here is executed by the whole warp; only the stores depend on the row. A warp
// whose 32 rows are all valid stores through its staging buffer `stg` with TMA (when a.tma_out;
// the scattering GEMM2 as eight 4-row scatters to the rows' tokens).
// zero: the tile summed nothing (an expert with no slots in K-grouped mode) and stores zeros
// without reading the accumulator.
__device__ __forceinline__ void epilogue_tile(const TcArgs &a, const Tile &ti, uint32_t tmem_base,
                                              uint32_t acc_col, int q, int lane, int half,
                                              const CUtensorMap *tmO, uint32_t stg,
                                              bool zero = false) {
    const int r = q * 32 + lane;
    bool valid = r < ti.rows;
    const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + acc_col;
    __nv_bfloat16 *orow = a.out + (int64_t)(ti.row0 + r) * a.N;
    float gscale = 1.f;
    int tok = 0;
    bool tok_ok = true;
    if (a.out_token && valid) {  // fused combine of a top-1 layer: y[token] = g * (H W2^T + b2)
        tok = __ldg(a.out_token + ti.row0 + r);
        tok_ok = tok >= 0 && (int64_t)tok < a.P;  // y has P = T rows
        if (!tok_ok) {
            report(a.dev_status, DEV_ERR_INDEX);
            tok = 0;
        }
        gscale = __ldg(a.out_gate + tok);
        orow = a.out + (int64_t)tok * a.N;
    }
    // warp-uniform; a group with a token out of range takes the per-thread path, which skips it
    const bool boxed = a.tma_out && q * 32 + 32 <= ti.rows &&
                       (!a.out_token || __all_sync(0xffffffffu, tok_ok));
    valid = valid && tok_ok;
    if (a.epi == EPI_SWIGLU) {
#pragma unroll 1
        for (int c = half * (BN / 4); c < (half + 1) * (BN / 4); c += 32) {
            float x1[32], x3[32];
            tmem_ld32x2(trow + c, trow + BN / 2 + c, x1, x3);
            const int col = ti.n * (BN / 2) + c;
            if (a.pre1 && valid && col < a.N) {
                const int64_t off = (int64_t)(ti.row0 + r) * a.N + col;
                store_row32(a.pre1 + off, x1);
                store_row32(a.pre3 + off, x3);
            }
            if (boxed && col < a.N) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16(silu_fast(x1[2 * i]) * x3[2 * i],
                                      silu_fast(x1[2 * i + 1]) * x3[2 * i + 1]);
                stage_and_store(tmO, stg, pk, col, ti.row0 + q * 32, lane);
            } else if (valid && col < a.N) {
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
            if (zero) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.f;
            } else {
                tmem_ld32(trow + c, v);
            }
            if (a.bias) {
                const float *bp = a.bias + (int64_t)ti.e * a.N + col;
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] += __ldg(bp + i);
            }
            if (a.pre1 && valid) store_row32(a.pre1 + (int64_t)(ti.row0 + r) * a.N + col, v);
            if (a.epi == EPI_GELU) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = gelu_tanh_fast(v[i]);
            }
            if (a.out_token) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= gscale;
            }
            if (a.out_f32) {
                if (valid) {
                    float4 *dst = reinterpret_cast<float4 *>(a.out_f32 +
                                                             (int64_t)(ti.row0 + r) * a.N + col);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                }
                continue;
            }
            if (boxed) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
                if (a.out_token)
                    stage_and_scatter(tmO, stg, pk, col, tok, lane);
                else
                    stage_and_store(tmO, stg, pk, col, ti.row0 + q * 32, lane);
            } else if (valid) {
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
}

// One CTA per SM; see the file comment. KG: the K-grouped schedule; MN: MN-major B allowed
// (TcArgs).
template <bool KG, bool MN>
__global__ void __launch_bounds__(TC_THREADS, 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmB3,
                           const __grid_constant__ CUtensorMap tmO, const TcArgs a) {
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
    pdl_wait();  // offsets and A come from earlier kernels on the stream
    const int E = a.E;
    constexpr bool PAIR = false;
    const int rank = 0;
    const int unit0 = (int)blockIdx.x;
    const int ustep = (int)gridDim.x;

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
        if (KG) {
            // K segments: multiples of BK, ascending, within the operands' width
            bool bad = a.offsets[0] != 0;
            for (int e = 0; e <= E; ++e) {
                const int v = a.offsets[e];
                if (v < 0 || v % BK != 0 || (int64_t)v > (int64_t)a.K ||
                    (e > 0 && v < s_off[e - 1]))
                    bad = true;
                s_off[e] = v;
            }
            s_cum[E] = bad ? 0 : E * a.m_tiles * a.n_tiles;
            if (bad) report(a.dev_status, DEV_ERR_INDEX);
        } else {
            int cum = 0;
            bool bad = false;
            for (int e = 0; e < E; ++e) {
                const int lo = a.offsets[e], hi = a.offsets[e + 1];
                if (lo < 0 || hi < lo || (int64_t)hi > a.P) bad = true;
                s_off[e] = lo;
                s_cum[e] = cum;
                const int mt = (hi - lo + BM - 1) / BM;
                if (!bad) cum += mt * a.n_tiles;
            }
            s_off[E] = a.offsets[E];
            s_cum[E] = cum;
            if (bad) {
                report(a.dev_status, DEV_ERR_INDEX);
                for (int e = 0; e <= E; ++e) s_cum[e] = 0;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = s_cum[E];
    const int nk = a.K / BK;
    const unsigned long long lim = a.spin_limit_ns;

    if (warp == 0 && a.a_rows == nullptr) {
        // Producer: lane 0 waits for free slots and issues the A and B copies.
        if (lane == 0) {
            int stage = 0, eh = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, last_phase = 0;  // per-stage bits
            bool ok = !a.withhold_loads;
            for (int t = unit0; t < total && ok; t += ustep) {
                const Tile ti = KG ? decode_tile_kg(t, a)
                                   : decode_tile<PAIR>(t, eh, s_cum, s_off, a.n_tiles, rank);
                // B rows of this N tile: SwiGLU stacks 128 rows of W1 over 128 rows of W3
                const int brow = KG ? ti.n * BN
                                    : (a.epi == EPI_SWIGLU ? ti.e * a.N + ti.n * (BN / 2)
                                                           : ti.e * a.N + ti.n * BN);
                const int arow = KG ? ti.row0 - ti.e * a.M : ti.row0;
                const int kx0 = KG ? s_off[ti.e] : 0;
                const int nkt = KG ? (s_off[ti.e + 1] - s_off[ti.e]) / BK : nk;
                for (int kb = 0; kb < nkt; ++kb) {
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, s_abort, a.dev_status, lim)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar_full + 8 * stage;
                    const uint32_t sb = sB + stage * B_STAGE;
                    mbar_expect_tx(fb, A_STAGE + B_STAGE);
                    const int kx = kx0 + kb * BK;
                    if (MN && a.a_mn) {
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            tma_load_2d(sA + stage * A_STAGE + q * (A_STAGE / 2), &tmA, fb,
                                        arow + q * 64, kx);
                    } else {
                        tma_load_2d(sA + stage * A_STAGE, &tmA, fb, kx, arow);
                    }
                    if (MN && a.b_mn) {
                        // four 64 x 64 boxes along N, rows = this k-block of the expert's B
                        const bool second = a.b_ksplit > 0 && kb >= a.b_ksplit;
                        const int krow = KG ? kx
                                            : ti.e * a.b_krows + (second ? kb - a.b_ksplit : kb) * BK;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            tma_load_2d(sb + q * (B_STAGE / 4), second ? &tmB3 : &tmB, fb,
                                        ti.n * BN + q * 64, krow);
                    } else if (a.epi == EPI_SWIGLU) {
                        tma_load_2d(sb, &tmB, fb, kx, brow);
                        tma_load_2d(sb + B_STAGE / 2, &tmB3, fb, kx, brow);
                    } else {
                        tma_load_2d(sb, &tmB, fb, kx, brow);
                        tma_load_2d(sb + B_STAGE / 2, &tmB, fb, kx, brow + BN / 2);
                    }
                    issued |= 1u << stage;
                    last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Every copy into this CTA's ring must have landed before it may exit.
            for (int s = 0; s < STAGES; ++s)
                if ((issued >> s) & 1u)
                    mbar_wait(bar_full + 8 * s, (last_phase >> s) & 1u, nullptr, a.dev_status, lim);
        }
    } else if (warp == 0) {
        // Producer with a fused gather: the whole warp runs the loop; lane 0 waits for free
        // slots and issues the B copies, and every lane copies 4 of the tile's 128 A rows.
        const bool gather = a.a_rows != nullptr;
        int stage = 0, eh = 0;
        uint32_t phase = 0;
        uint32_t issued = 0, last_phase = 0;  // per-stage bits
        bool ok = !a.withhold_loads;
        for (int t = unit0; t < total && ok; t += ustep) {
            const Tile ti = decode_tile<PAIR>(t, eh, s_cum, s_off, a.n_tiles, rank);
            const int brow = a.epi == EPI_SWIGLU ? ti.e * a.N + ti.n * (BN / 2)
                                                 : ti.e * a.N + ti.n * BN;
            const int4 gr = gather ? gather_rows(a, ti.row0, ti.rows, lane) : make_int4(0, 0, 0, 0);
            for (int kb = 0; kb < nk; ++kb) {
                int go = 1;
                if (lane == 0)
                    go = mbar_wait(bar_empty + 8 * stage, phase ^ 1u, s_abort, a.dev_status, lim);
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) {
                    ok = false;
                    break;
                }
                const uint32_t fb = bar_full + 8 * stage;
                const uint32_t sb = sB + stage * B_STAGE;
                if (lane == 0) {
                    mbar_expect_tx(fb, A_STAGE + B_STAGE);
                    if (!gather) tma_load_2d(sA + stage * A_STAGE, &tmA, fb, kb * BK, ti.row0);
                    if (a.epi == EPI_SWIGLU) {
                        tma_load_2d(sb, &tmB, fb, kb * BK, brow);
                        tma_load_2d(sb + B_STAGE / 2, &tmB3, fb, kb * BK, brow);
                    } else {
                        tma_load_2d(sb, &tmB, fb, kb * BK, brow);
                        tma_load_2d(sb + B_STAGE / 2, &tmB, fb, kb * BK, brow + BN / 2);
                    }
                }
                if (gather) {
                    __syncwarp();
                    tma_gather4(sA + stage * A_STAGE + lane * 512, &tmA, fb, kb * BK, gr.x, gr.y,
                                gr.z, gr.w);
                }
                issued |= 1u << stage;
                last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // Every copy into this CTA's ring must have landed before it may exit.
        if (lane == 0)
            for (int s = 0; s < STAGES; ++s)
                if ((issued >> s) & 1u)
                    mbar_wait(bar_full + 8 * s, (last_phase >> s) & 1u, nullptr, a.dev_status, lim);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, acc = 0, eh = 0;
            uint32_t phase = 0, aphase = 0;
            bool ok = true;
            const bool bmn = MN && a.b_mn, amn = MN && a.a_mn;
            const uint32_t idesc =
                idesc_bf16(BM, BN) | (bmn ? IDESC_B_MN : 0u) | (amn ? IDESC_A_MN : 0u);
            for (int t = unit0; t < total && ok; t += ustep) {
                const Tile ti = KG ? decode_tile_kg(t, a)
                                   : decode_tile<PAIR>(t, eh, s_cum, s_off, a.n_tiles, rank);
                const bool idle = ti.rows <= 0;
                const int nkt = KG ? (s_off[ti.e + 1] - s_off[ti.e]) / BK : nk;
                if (!mbar_wait(bar_tempty + 8 * acc, aphase ^ 1u, s_abort, a.dev_status, lim)) break;
                tc_fence_after();
                const uint32_t dt = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < nkt; ++kb) {
                    if (!mbar_wait(bar_full + 8 * stage, phase, s_abort, a.dev_status, lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (!idle) {
                        const uint64_t ad = amn ? sdesc_mn_sw128(sA + stage * A_STAGE, A_STAGE / 2)
                                                : sdesc_k_sw128(sA + stage * A_STAGE);
                        const uint64_t bd = bmn ? sdesc_mn_sw128(sB + stage * B_STAGE, B_STAGE / 4)
                                                : sdesc_k_sw128(sB + stage * B_STAGE);
                        // one K = 16 step: 32 bytes along a K-major row, 16 rows of an MN-major box
                        const uint64_t astep = amn ? 2048 >> 4 : 2, bstep = bmn ? 2048 >> 4 : 2;
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            umma_bf16(dt, ad + astep * kk, bd + bstep * kk, idesc,
                                      (kb | kk) != 0 ? 1u : 0u);
                    }
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
        const uint32_t stg = smem_u32(ctl + CTL_BYTES) + (uint32_t)(warp - 2) * EPI_BOX;
        int acc = 0, eh = 0;
        uint32_t aphase = 0;
        for (int t = unit0; t < total; t += ustep) {
            const Tile ti = KG ? decode_tile_kg(t, a)
                               : decode_tile<PAIR>(t, eh, s_cum, s_off, a.n_tiles, rank);
            int ok = 1;
            if (lane == 0) ok = mbar_wait(bar_tfull + 8 * acc, aphase, s_abort, a.dev_status, lim);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            __syncwarp();
            tc_fence_after();
            const bool zero = KG && s_off[ti.e + 1] == s_off[ti.e];
            epilogue_tile(a, ti, tmem_base, (uint32_t)(acc * BN), q, lane, half, &tmO, stg, zero);
            tc_fence_before();
            mbar_arrive(bar_tempty + 8 * acc);
            acc ^= 1;
            if (acc == 0) aphase ^= 1u;
        }
        if (lane == 0) bulk_wait_all();  // this warp's TMA stores have completed
        __syncwarp();
    }

    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------------------------
// CTA-pair kernel: a 2-CTA cluster computes 256 x 256 tiles with tcgen05.mma.cta_group::2.
//
// One MMA of M = 256 drives both SMs' tensor cores and reads each operand byte from shared
// memory once: CTA r holds rows 128r..128r+127 of the A tile and rows 128r..128r+127 of the
// 256-row B tile, at the same shared-memory offsets, and receives D rows 128r..128r+127 in its
// own tensor memory. Per SM and per 64-wide k-step that is 32 KiB of TMA writes and operand reads
// instead of 48 KiB for the single-CTA 128 x 256 tile, whose tensor pipe measured near two thirds
// busy on large experts: with the same shared memory the ring holds 6 stages, so more copies are
// in flight per SM for each flop.
//   - Both CTAs' producers load their own halves; the copies complete on the first (leader)
//     CTA's full barrier, which expects the bytes of both (TMA .cta_group::2 lets the barrier
//     live in the peer CTA).
//   - The leader's single MMA thread issues the MMAs; its commits arrive on the empty and
//     accumulator-full barriers of both CTAs (multicast).
//   - Both CTAs' epilogues read their own accumulator rows and arrive on the leader's
//     accumulator-empty barrier (one arrival per warp, 16 in all).
// The tile table counts units of two adjacent 128-row M tiles; on an expert's odd last tile the
// second CTA computes rows past the expert's end, which its epilogue masks.
constexpr int STAGES2 = 6;
// The pair kernel runs when experts average at least this many 128-row M tiles.
#ifndef PAIR_MIN_TILES
#define PAIR_MIN_TILES 4
#endif
constexpr int A_HALF = BM * BK * 2;          // 16 KiB: this CTA's A rows
constexpr int B_HALF = (BN / 2) * BK * 2;    // 16 KiB: this CTA's half of the B tile
constexpr size_t TC_SMEM_PAIR =
    1024 + (size_t)STAGES2 * (A_HALF + B_HALF) + CTL_BYTES + (size_t)EPI_WARPS * EPI_BOX;

// KG: the K-grouped schedule (MN-major A and B only); MN: MN-major B allowed.
template <bool KG, bool MN>
__global__ void __launch_bounds__(TC_THREADS, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmB3,
                             const __grid_constant__ CUtensorMap tmO, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + STAGES2 * A_HALF;
    uint8_t *ctl = gbase + STAGES2 * (A_HALF + B_HALF);
    const uint32_t bar0 = smem_u32(ctl);
    const uint32_t bar_full = bar0, bar_empty = bar0 + 8 * STAGES2;
    const uint32_t bar_tfull = bar0 + 16 * STAGES2, bar_tempty = bar_tfull + 16;
    const uint32_t bar_drain = bar_tempty + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctl + 256);
    volatile int *s_abort = reinterpret_cast<volatile int *>(ctl + 260);
    int32_t *s_cum = reinterpret_cast<int32_t *>(ctl + 512);   // [E+1]
    int32_t *s_off = s_cum + 260;                             // [E+1]
    int32_t *s_order = s_off + 260;                           // [E] (K-grouped)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();  // offsets and A come from earlier kernels on the stream
    const int E = a.E;
    const int rank = (int)cluster_ctarank();
    const bool leader = rank == 0;
    const int unit0 = (int)(blockIdx.x >> 1);
    const int ustep = (int)(gridDim.x >> 1);
    constexpr uint16_t BOTH = 0x3;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES2; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(bar_tfull + 8 * q, 1);
            mbar_init(bar_tempty + 8 * q, 16);
        }
        mbar_init(bar_drain, 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);  // collective: the same columns in both
        tmem_relinquish_pair();
    }
    if (warp == 2 && lane == 0 && KG) {
        // K segments: multiples of BK, ascending, within the operands' rows
        bool bad = a.offsets[0] != 0;
        for (int e = 0; e <= E; ++e) {
            const int v = a.offsets[e];
            if (v < 0 || v % BK != 0 || (int64_t)v > (int64_t)a.K || (e > 0 && v < s_off[e - 1]))
                bad = true;
            s_off[e] = v;
        }
        s_cum[E] = bad ? 0 : E * ((a.m_tiles + 1) / 2) * a.n_tiles;
        if (bad) report(a.dev_status, DEV_ERR_INDEX);
    } else if (warp == 2 && lane == 0) {
        int cum = 0;
        bool bad = false;
        for (int e = 0; e < E; ++e) {
            const int lo = a.offsets[e], hi = a.offsets[e + 1];
            if (lo < 0 || hi < lo || (int64_t)hi > a.P) bad = true;
            s_off[e] = lo;
            s_cum[e] = cum;
            const int mt = (hi - lo + BM - 1) / BM;
            if (!bad) cum += (mt + 1) / 2 * a.n_tiles;
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
    if (KG) {
        kg_order(s_off, E, s_order);
        __syncthreads();
    }
    cluster_sync();  // both CTAs' barriers exist before any remote arrive or copy completes
    const uint32_t tmem_base = *tmem_slot;
    const int total = s_cum[E];
    const int nk = a.K / BK;
    const unsigned long long lim = a.spin_limit_ns;

    if (warp == 0 && a.a_rows == nullptr) {
        // Producer: lane 0 waits for free slots and issues this CTA's A and B copies, which
        // complete on the leader's barrier.
        if (lane == 0) {
            int stage = 0, eh = 0;
            uint32_t phase = 0;
            bool ok = !a.withhold_loads;
            for (int t = unit0; t < total && ok; t += ustep) {
                const Tile ti = KG ? decode_tile_kg_pair(t, a, rank, s_order)
                                   : decode_tile<true>(t, eh, s_cum, s_off, a.n_tiles, rank);
                // this CTA's half of the B tile: SwiGLU W1 (CTA 0) / W3 (CTA 1) rows, else rows
                // 128 r.. of the 256-row W tile
                const CUtensorMap *bm = (a.epi == EPI_SWIGLU && rank == 1) ? &tmB3 : &tmB;
                const int brow = a.epi == EPI_SWIGLU ? ti.e * a.N + ti.n * (BN / 2)
                                                     : ti.e * a.N + ti.n * BN + rank * (BN / 2);
                const int nkt = KG ? (s_off[ti.e + 1] - s_off[ti.e]) / BK : nk;
                for (int kb = 0; kb < nkt; ++kb) {
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, s_abort, a.dev_status, lim)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = mapa_shared(bar_full + 8 * stage, 0);  // leader's barrier
                    if (leader) mbar_expect_tx(bar_full + 8 * stage, 2 * (A_HALF + B_HALF));
                    if (KG) {
                        // this CTA's 128 columns of the MN-major A: two 64 x 64 boxes
                        const int kx = s_off[ti.e] + kb * BK;
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            tma_load_2d_pair(sA + stage * A_HALF + q * (A_HALF / 2), &tmA, fb,
                                             ti.row0 - ti.e * a.M + q * 64, kx);
                    } else {
                        // an idle half (past its expert's rows) reads rows past the end of A,
                        // which TMA fills with zeros: its masked MMA rows then multiply zeros
                        // (less switching power under the power cap) instead of the next
                        // expert's rows
                        tma_load_2d_pair(sA + stage * A_HALF, &tmA, fb, kb * BK,
                                         ti.rows > 0 ? ti.row0 : (int)a.P);
                    }
                    if (MN && a.b_mn) {
                        // this CTA's 128 columns of B: two 64 x 64 boxes
                        const bool second = a.b_ksplit > 0 && kb >= a.b_ksplit;
                        const int krow = KG ? s_off[ti.e] + kb * BK
                                            : ti.e * a.b_krows + (second ? kb - a.b_ksplit : kb) * BK;
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            tma_load_2d_pair(sB + stage * B_HALF + q * (B_HALF / 2),
                                             second ? &tmB3 : &tmB, fb,
                                             ti.n * BN + rank * (BN / 2) + q * 64, krow);
                    } else {
                        tma_load_2d_pair(sB + stage * B_HALF, bm, fb, kb * BK, brow);
                    }
                    if (++stage == STAGES2) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // A slot is released only after the leader's MMAs consumed it, hence after every copy
            // into it (this CTA's included) landed: wait for all slots once more before exiting.
            if (ok) {
                for (int i = 0; i < STAGES2; ++i) {
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, s_abort, a.dev_status, lim))
                        break;
                    if (++stage == STAGES2) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 0) {
        // Producer with a fused gather: the whole warp runs the loop (see the single-CTA
        // kernel).
        const bool gather = a.a_rows != nullptr;
        int stage = 0, eh = 0;
        uint32_t phase = 0;
        bool ok = !a.withhold_loads;
        for (int t = unit0; t < total && ok; t += ustep) {
            const Tile ti = decode_tile<true>(t, eh, s_cum, s_off, a.n_tiles, rank);
            // this CTA's half of the B tile: SwiGLU W1 (CTA 0) / W3 (CTA 1) rows, else rows
            // 128 r.. of the 256-row W tile
            const CUtensorMap *bm = (a.epi == EPI_SWIGLU && rank == 1) ? &tmB3 : &tmB;
            const int brow = a.epi == EPI_SWIGLU ? ti.e * a.N + ti.n * (BN / 2)
                                                 : ti.e * a.N + ti.n * BN + rank * (BN / 2);
            const int4 gr = gather ? gather_rows(a, ti.row0, ti.rows, lane) : make_int4(0, 0, 0, 0);
            for (int kb = 0; kb < nk; ++kb) {
                int go = 1;
                if (lane == 0)
                    go = mbar_wait(bar_empty + 8 * stage, phase ^ 1u, s_abort, a.dev_status, lim);
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) {
                    ok = false;
                    break;
                }
                const uint32_t fb = mapa_shared(bar_full + 8 * stage, 0);  // leader's barrier
                if (lane == 0) {
                    if (leader) mbar_expect_tx(bar_full + 8 * stage, 2 * (A_HALF + B_HALF));
                    if (!gather) tma_load_2d_pair(sA + stage * A_HALF, &tmA, fb, kb * BK, ti.row0);
                    tma_load_2d_pair(sB + stage * B_HALF, bm, fb, kb * BK, brow);
                }
                if (gather) {
                    __syncwarp();
                    tma_gather4_pair(sA + stage * A_HALF + lane * 512, &tmA, fb, kb * BK, gr.x,
                                     gr.y, gr.z, gr.w);
                }
                if (++stage == STAGES2) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // A slot is released only after the leader's MMAs consumed it, hence after every copy
        // into it (this CTA's included) landed: wait for all slots once more before exiting.
        if (ok && lane == 0) {
            for (int i = 0; i < STAGES2; ++i) {
                if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, s_abort, a.dev_status, lim))
                    break;
                if (++stage == STAGES2) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, aphase = 0;
            bool ok = true;
            const bool bmn = MN && a.b_mn, amn = KG;
            const uint32_t idesc =
                idesc_bf16(2 * BM, BN) | (bmn ? IDESC_B_MN : 0u) | (amn ? IDESC_A_MN : 0u);
            for (int t = unit0; t < total && ok; t += ustep) {
                if (!mbar_wait(bar_tempty + 8 * acc, aphase ^ 1u, s_abort, a.dev_status, lim)) break;
                tc_fence_after();
                const uint32_t dt = tmem_base + (uint32_t)(acc * BN);
                int nkt = nk;
                if (KG) {
                    const Tile ti = decode_tile_kg_pair(t, a, 0, s_order);
                    nkt = (s_off[ti.e + 1] - s_off[ti.e]) / BK;
                }
                for (int kb = 0; kb < nkt; ++kb) {
                    if (!mbar_wait(bar_full + 8 * stage, phase, s_abort, a.dev_status, lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = amn ? sdesc_mn_sw128(sA + stage * A_HALF, A_HALF / 2)
                                            : sdesc_k_sw128(sA + stage * A_HALF);
                    const uint64_t bd = bmn ? sdesc_mn_sw128(sB + stage * B_HALF, B_HALF / 2)
                                            : sdesc_k_sw128(sB + stage * B_HALF);
                    // one K = 16 step: 32 bytes along a K-major row, 16 rows of an MN-major box
                    const uint64_t astep = amn ? 2048 >> 4 : 2, bstep = bmn ? 2048 >> 4 : 2;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16_pair(dt, ad + astep * kk, bd + bstep * kk, idesc,
                                       (kb | kk) != 0 ? 1u : 0u);
                    umma_commit_pair_multicast(bar_empty + 8 * stage, BOTH);
                    if (++stage == STAGES2) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair_multicast(bar_tfull + 8 * acc, BOTH);
                acc ^= 1;
                if (acc == 0) aphase ^= 1u;
            }
            umma_commit_pair(bar_drain);
            mbar_wait(bar_drain, 0, nullptr, a.dev_status, lim);
        }
    } else {
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const uint32_t stg = smem_u32(ctl + CTL_BYTES) + (uint32_t)(warp - 2) * EPI_BOX;
        int acc = 0, eh = 0;
        uint32_t aphase = 0;
        for (int t = unit0; t < total; t += ustep) {
            const Tile ti = KG ? decode_tile_kg_pair(t, a, rank, s_order)
                               : decode_tile<true>(t, eh, s_cum, s_off, a.n_tiles, rank);
            int ok = 1;
            if (lane == 0) ok = mbar_wait(bar_tfull + 8 * acc, aphase, s_abort, a.dev_status, lim);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            __syncwarp();
            tc_fence_after();
            const bool zero = KG && s_off[ti.e + 1] == s_off[ti.e];
            epilogue_tile(a, ti, tmem_base, (uint32_t)(acc * BN), q, lane, half, &tmO, stg, zero);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(bar_tempty + 8 * acc, 0));
            acc ^= 1;
            if (acc == 0) aphase ^= 1u;
        }
        if (lane == 0) bulk_wait_all();  // this warp's TMA stores have completed
        __syncwarp();
    }

    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no copy, commit or remote arrive targets either CTA any more
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------------------------
// host side

// Resident 2-CTA clusters of the pair kernel on this device (0: cannot launch it).
int pair_clusters() {
    // per-device cache (done: queried); several host threads may fill it at once
    static std::atomic<int> cache[64] = {};
    static std::atomic<bool> done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!done[dev].load(std::memory_order_acquire)) {
        int n = 0;
        if (set_max_dynamic_smem((const void *)grouped_gemm_pair_kernel<false, false>, TC_SMEM_PAIR) ==
            cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * 74);
            cfg.blockDim = dim3(TC_THREADS);
            cfg.dynamicSmemBytes = TC_SMEM_PAIR;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<false, false>, &cfg) != cudaSuccess)
                n = 0;
        }
        cudaGetLastError();
        cache[dev].store(n, std::memory_order_relaxed);
        done[dev].store(true, std::memory_order_release);
    }
    return cache[dev].load(std::memory_order_relaxed);
}

// The optional parts of a row-grouped GEMM launch (all off by default).
struct GemmOpts {
    const int32_t *A_rows = nullptr;  // fused gather: A row r is row A_rows[r] of [A_src_rows, K]
    int64_t A_src_rows = 0;
    const int32_t *out_token = nullptr;  // fused scatter (top-1 GEMM2): row r to out[out_token[r]]
    const float *out_gate = nullptr;     //   scaled by out_gate[out_token[r]]
    void *pre1 = nullptr, *pre3 = nullptr;  // training forward: GEMM1's pre-activations
    int b_mn = 0, b_ksplit = 0, b_krows = 0;  // MN-major B (see TcArgs)
    float *out_f32 = nullptr;                 // f32 output instead of out
};

cudaError_t launch_gemm(const void *A, const void *B, const void *B3, int64_t P, int E, int K,
                        int N, int epi, const int32_t *offsets, const float *bias, void *out,
                        uint32_t *dev_status, const FaultHook &hook, cudaStream_t s,
                        const GemmOpts &o = GemmOpts()) {
    const int32_t *A_rows = o.A_rows, *out_token = o.out_token;
    const int64_t A_src_rows = o.A_src_rows;
    const float *out_gate = o.out_gate;
    void *pre1 = o.pre1, *pre3 = o.pre3;
    const int b_mn = o.b_mn, b_ksplit = o.b_ksplit, b_krows = o.b_krows;
    float *out_f32 = o.out_f32;
    if (out_f32 && (epi != EPI_STORE || out_token)) return cudaErrorInvalidValue;
    if (out_token && epi == EPI_SWIGLU) return cudaErrorInvalidValue;  // the scatter is GEMM2's
    // the f32 output leaves through per-thread stores; the store map only has to encode
    if (out_f32) out = out_f32;
    // every B box is 128 rows: one half of the 256-row B tile; a gathered A reads one-row boxes
    CUtensorMap mA, mB, mB3, mO;
    if (A_rows ? !make_map(&mA, A, A_src_rows, K, 1) : !make_map(&mA, A, P, K, BM))
        return cudaErrorInvalidValue;
    // the output of the TMA-store epilogue: [P, N] rows in sorted order, or for the scattering
    // top-1 GEMM2 the token rows of y [P = T, N], written four rows at a time (one-row boxes)
    if (!make_store_map(&mO, out, P, N, out_token ? 1 : 32)) return cudaErrorInvalidValue;
    if (b_mn) {
        // B as [E b_krows, N] row-major (rows = K index), read in 64 x 64 boxes; B3 likewise
        if (A_rows || epi != EPI_STORE || b_krows <= 0 || b_krows % BK != 0)
            return cudaErrorInvalidValue;
        if (!make_map(&mB, B, (int64_t)E * b_krows, N, 64)) return cudaErrorInvalidValue;
        if (!make_map(&mB3, b_ksplit > 0 ? B3 : B, (int64_t)E * b_krows, N, 64))
            return cudaErrorInvalidValue;
    } else {
        if (!make_map(&mB, B, (int64_t)E * N, K, BN / 2)) return cudaErrorInvalidValue;
        if (!make_map(&mB3, epi == EPI_SWIGLU ? B3 : B, (int64_t)E * N, K, BN / 2))
            return cudaErrorInvalidValue;
    }
    TcArgs a;
    a.offsets = offsets;
    a.bias = bias;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.dev_status = dev_status;
    a.P = P;
    a.E = E;
    a.K = K;
    a.N = N;
    const int b_rows = epi == EPI_SWIGLU ? BN / 2 : BN;  // output columns per N tile
    a.n_tiles = (N + b_rows - 1) / b_rows;
    a.epi = epi;
    a.spin_limit_ns = hook.spin_limit_ns;
    a.withhold_loads = hook.withhold;
    a.tma_out = (MOE_GEMM_TMA_STORE && out_f32 == nullptr) ? 1 : 0;
    a.out_f32 = out_f32;
    a.a_rows = A_rows;
    a.a_src_rows = A_src_rows;
    a.out_token = out_token;
    a.out_gate = out_gate;
    a.M = 0;
    a.m_tiles = 0;
    a.pre1 = static_cast<__nv_bfloat16 *>(pre1);
    a.pre3 = static_cast<__nv_bfloat16 *>(pre3);
    a.b_mn = b_mn;
    a.b_ksplit = b_ksplit;
    a.b_krows = b_krows;
    a.a_mn = 0;
    // The CTA-pair kernel when experts average at least four M tiles (on an expert's odd last
    // tile the second CTA computes masked rows, a small loss there).
    const int clusters = pair_clusters();
    const bool pair = clusters > 0 && P >= (int64_t)PAIR_MIN_TILES * BM * E;
    if (pair) {
        const int64_t units = ((P + 2 * BM - 1) / (2 * BM) + E) * (int64_t)a.n_tiles;
        const int64_t ncl = clusters < units ? clusters : units;
        if (b_mn) {
            cudaError_t err = set_max_dynamic_smem(
                (const void *)grouped_gemm_pair_kernel<false, true>, TC_SMEM_PAIR);
            if (err != cudaSuccess) return err;
            return launch_pdl(grouped_gemm_pair_kernel<false, true>, dim3((unsigned)(2 * ncl)),
                              dim3(TC_THREADS), TC_SMEM_PAIR, s, 2, mA, mB, mB3, mO, a);
        }
        return launch_pdl(grouped_gemm_pair_kernel<false, false>, dim3((unsigned)(2 * ncl)),
                          dim3(TC_THREADS), TC_SMEM_PAIR, s, 2, mA, mB, mB3, mO, a);
    }
    const int64_t upper = ((P + BM - 1) / BM + E) * (int64_t)a.n_tiles;
    int64_t grid = num_sms();
    if (grid > upper) grid = upper;
    if (b_mn) {
        cudaError_t err =
            set_max_dynamic_smem((const void *)grouped_gemm_tc_kernel<false, true>, TC_SMEM);
        if (err != cudaSuccess) return err;
        return launch_pdl(grouped_gemm_tc_kernel<false, true>, dim3((unsigned)grid),
                          dim3(TC_THREADS), TC_SMEM, s, 1, mA, mB, mB3, mO, a);
    }
    cudaError_t err = set_max_dynamic_smem((const void *)grouped_gemm_tc_kernel<false, false>, TC_SMEM);
    if (err != cudaSuccess) return err;
    return launch_pdl(grouped_gemm_tc_kernel<false, false>, dim3((unsigned)grid), dim3(TC_THREADS),
                      TC_SMEM, s, 1, mA, mB, mB3, mO, a);
}

// The K-grouped GEMM runs on CTA pairs when its groups average at least this many rows of K.
constexpr int KG_PAIR_MIN_K = 512;

// K-grouped GEMM: out[e M + m, n] = sum over k in [kseg[e], kseg[e+1]) of A(m, k) B(n, k) for
// every expert e (zeros where the segment is empty); kseg [E+1] device int32, multiples of 64.
// A [kwidth, M] and B [kwidth, N] MN-major (the K index is the row) with row strides lda and
// ldb, zero pad rows; rows at or past map_rows (when > 0) read as zeros. out [E M, N] bf16, or
// out_f32 [E M, N] f32.
cudaError_t launch_gemm_kg(const void *A, const void *B, const int32_t *kseg, int E, int M, int N,
                           int64_t kwidth, void *out, uint32_t *dev_status, cudaStream_t s,
                           int64_t lda, int64_t ldb, int64_t map_rows = 0,
                           float *out_f32 = nullptr) {
    if (E <= 0 || E > 256 || M <= 0 || N <= 0 || kwidth <= 0 || kwidth % BK != 0 ||
        kwidth >= (1ll << 31))
        return cudaErrorInvalidValue;
    if (out_f32) out = out_f32;  // the store map only has to encode
    CUtensorMap mA, mB, mO;
    const int64_t rows = map_rows > 0 ? map_rows : kwidth;
    if (M % 64 != 0 || N % 64 != 0 || lda < M || ldb < N || rows > kwidth)
        return cudaErrorInvalidValue;
    if (!make_map_ld(&mA, A, rows, M, lda, 64)) return cudaErrorInvalidValue;
    if (!make_map_ld(&mB, B, rows, N, ldb, 64)) return cudaErrorInvalidValue;
    if (!make_store_map(&mO, out, (int64_t)E * M, N)) return cudaErrorInvalidValue;
    TcArgs a = {};
    a.offsets = kseg;
    a.bias = nullptr;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.dev_status = dev_status;
    a.P = (int64_t)E * M;
    a.E = E;
    a.K = (int)kwidth;
    a.N = N;
    a.n_tiles = (N + BN - 1) / BN;
    a.epi = EPI_STORE;
    a.spin_limit_ns = SPIN_LIMIT_NS;
    a.withhold_loads = 0;
    a.tma_out = out_f32 ? 0 : MOE_GEMM_TMA_STORE;
    a.out_f32 = out_f32;
    a.a_rows = nullptr;
    a.a_src_rows = 0;
    a.out_token = nullptr;
    a.out_gate = nullptr;
    a.M = M;
    a.m_tiles = (M + BM - 1) / BM;
    a.pre1 = a.pre3 = nullptr;
    a.b_mn = a.a_mn = 1;
    a.b_ksplit = a.b_krows = 0;
    const int64_t units = (int64_t)E * a.m_tiles * a.n_tiles;
    if (units >= (1ll << 31)) return cudaErrorInvalidValue;
    const int clusters = pair_clusters();
    if (clusters > 0 && kwidth >= (int64_t)KG_PAIR_MIN_K * E) {
        // 256 x 256 tiles on CTA pairs (each CTA loads half of A and half of B), when the groups
        // average KG_PAIR_MIN_K rows of K: with shorter sums the pair's per-tile handshake costs
        // more than its halved operand traffic saves
        const int64_t punits = (int64_t)E * ((a.m_tiles + 1) / 2) * a.n_tiles;
        const int64_t ncl = clusters < punits ? clusters : punits;
        cudaError_t err =
            set_max_dynamic_smem((const void *)grouped_gemm_pair_kernel<true, true>, TC_SMEM_PAIR);
        if (err != cudaSuccess) return err;
        return launch_pdl(grouped_gemm_pair_kernel<true, true>, dim3((unsigned)(2 * ncl)),
                          dim3(TC_THREADS), TC_SMEM_PAIR, s, 2, mA, mB, mB, mO, a);
    }
    int64_t grid = num_sms();
    if (grid > units) grid = units;
    cudaError_t err =
        set_max_dynamic_smem((const void *)grouped_gemm_tc_kernel<true, true>, TC_SMEM);
    if (err != cudaSuccess) return err;
    return launch_pdl(grouped_gemm_tc_kernel<true, true>, dim3((unsigned)grid), dim3(TC_THREADS),
                      TC_SMEM, s, 1, mA, mB, mB, mO, a);
}

}  // namespace

cudaError_t launch_gemm_rows(const void *A, const int32_t *A_rows, int64_t A_src_rows,
                             const void *B, int64_t P, int E, int K, int N,
                             const int32_t *offsets, const float *bias, void *out,
                             uint32_t *dev_status, cudaStream_t s) {
    if (P == 0) return cudaSuccess;
    GemmOpts o;
    o.A_rows = A_rows;
    o.A_src_rows = A_rows ? A_src_rows : 0;
    return launch_gemm(A, B, nullptr, P, E, K, N, EPI_STORE, offsets, bias, out, dev_status,
                       FaultHook(), s, o);
}

cudaError_t launch_gemm_rows_bmn(const void *A, const void *B, const void *B3, int b_krows,
                                 int b_ksplit, int64_t P, int E, int K, int N,
                                 const int32_t *offsets, void *out, uint32_t *dev_status,
                                 cudaStream_t s) {
    if (P == 0) return cudaSuccess;
    if (K != (b_ksplit > 0 ? 2 * b_krows : b_krows) || (b_ksplit > 0 && b_ksplit * BK != b_krows))
        return cudaErrorInvalidValue;
    GemmOpts o;
    o.b_mn = 1;
    o.b_ksplit = b_ksplit;
    o.b_krows = b_krows;
    return launch_gemm(A, B, B3, P, E, K, N, EPI_STORE, offsets, nullptr, out, dev_status,
                       FaultHook(), s, o);
}

cudaError_t launch_gemm_kgroup_mn(const void *A, int64_t lda, const void *B, int64_t ldb,
                                  const int32_t *kseg, int E, int M, int N, int64_t rows,
                                  void *out, uint32_t *dev_status, cudaStream_t s,
                                  int64_t map_rows, float *out_f32) {
    return launch_gemm_kg(A, B, kseg, E, M, N, rows, out, dev_status, s, lda, ldb, map_rows,
                          out_f32);
}

cudaError_t launch_gemm_rows_f32(const void *A, const void *B, int64_t P, int E, int K, int N,
                                 const int32_t *offsets, float *out, uint32_t *dev_status,
                                 cudaStream_t s) {
    if (P == 0) return cudaSuccess;
    GemmOpts o;
    o.out_f32 = out;
    return launch_gemm(A, B, nullptr, P, E, K, N, EPI_STORE, offsets, nullptr, nullptr, dev_status,
                       FaultHook(), s, o);
}

cudaError_t launch_ffn_tc(const moe_config_t &c, const FfnBufs &b, cudaStream_t s,
                          const FaultHook &hook) {
    const int64_t P = c.T * c.k;
    if (P == 0) return cudaSuccess;
    const bool swiglu = c.act == MOE_ACT_SWIGLU;
    const bool gather = b.gather_h != nullptr;
    const bool scatter = b.scatter_y != nullptr;
    if ((gather || scatter) && (b.sorted_token == nullptr || (scatter && b.gates == nullptr)))
        return cudaErrorInvalidValue;
    GemmOpts o1;
    o1.A_rows = gather ? b.sorted_token : nullptr;
    o1.A_src_rows = gather ? c.T : 0;
    o1.pre1 = b.pre1;
    o1.pre3 = swiglu ? b.pre3 : nullptr;
    cudaError_t err = launch_gemm(gather ? b.gather_h : b.x_perm, b.W1, b.W3, P, c.E, c.d, c.f,
                                  swiglu ? EPI_SWIGLU : EPI_GELU, b.offsets,
                                  c.has_bias ? b.b1 : nullptr, b.H, b.dev_status, hook, s, o1);
    if (err != cudaSuccess) return err;
    GemmOpts o2;
    o2.out_token = scatter ? b.sorted_token : nullptr;
    o2.out_gate = scatter ? b.gates : nullptr;
    return launch_gemm(b.H, b.W2, nullptr, P, c.E, c.f, c.d, EPI_STORE, b.offsets,
                       c.has_bias ? b.b2 : nullptr, scatter ? b.scatter_y : b.y_perm,
                       b.dev_status, hook, s, o2);
}

}  // namespace moe
