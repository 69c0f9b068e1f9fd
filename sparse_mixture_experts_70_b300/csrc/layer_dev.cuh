// layer_dev.cuh -- device-side building blocks shared by several of libmoe's kernels: the
// dispatch pieces (chunk histogram, offsets, the single-block dispatch) and the auxiliary
// reduction. The step kernels (dispatch.cu, combine.cu) and the fused dispatch-and-aux kernel of
// single-chunk layers call the same functions, so both paths compute the same bits.
#pragma once

#include "internal.cuh"

namespace moe {
namespace dev {

constexpr int LB_WINDOW = 8;  // look-back words read per round trip
constexpr uint64_t FLAG_AGG = 1ull << 32;
constexpr uint64_t FLAG_INC = 2ull << 32;

struct DispatchArgs {
    const int32_t *idx;
    int32_t *counts, *offsets, *sorted_token, *slot_of, *excl;
    unsigned long long *words;  // [nchunks][E] look-back words
    uint32_t *done;
    uint32_t *dev_status;
    int64_t P;
    int k, E, nchunks;
    int64_t cap;  // per-expert capacity, -1 when dropless
    unsigned long long spin_limit_ns;
    int withhold;  // test hook: chunk 0 never publishes its look-back word
};

__device__ __forceinline__ void st_release(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// A look-back word carries its flag and its count in one 64-bit store, so a reader needs only
// that word: relaxed loads (at gpu scope, from L2) may be issued several at a time.
__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Chunk histogram: returns this thread's expert (-1 for no slot) and its rank inside the chunk;
// thread e < E receives the chunk's count of expert e in *agg.
__device__ __forceinline__ int chunk_ranks(const DispatchArgs &a, int c, int32_t *cnt, int *lrank,
                                           int *agg) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, E = a.E;
    const int64_t s = (int64_t)c * DISPATCH_THREADS + tid;
    int e = -1;
    if (s < a.P) {
        e = a.idx[s];
        if (e < 0 || e >= E) {
            report(a.dev_status, DEV_ERR_INDEX);
            e = -1;
        }
    }
    for (int q = tid; q < 32 * E; q += DISPATCH_THREADS) cnt[q] = 0;
    __syncthreads();
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) cnt[w * E + e] = __popc(peers);
    __syncthreads();
    int run = 0;
    if (tid < E) {
        for (int ww = 0; ww < 32; ++ww) {
            const int v = cnt[ww * E + tid];
            cnt[ww * E + tid] = run;
            run += v;
        }
    }
    __syncthreads();
    *lrank = e >= 0 ? cnt[w * E + e] + rank : 0;
    *agg = run;
    __syncthreads();
    return e;
}

// counts[e] = tot[e], offsets = exclusive scan over e of the kept rows min(tot[e], cap), and
// s_off[e] = offsets[e], for e < E <= 256, by the block's first 8 warps (warp scans, then a scan
// of the 8 warp totals); the whole block calls it. offsets[E] is the number of kept rows.
__device__ __forceinline__ void publish_offsets(const DispatchArgs &a, const int32_t *tot,
                                                int32_t *s_off, int32_t *s_wsum) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, E = a.E;
    int kept = 0, incl = 0;
    if (tid < 256) {
        if (tid < E) {
            const int c = tot[tid];
            kept = (a.cap >= 0 && c > a.cap) ? (int)a.cap : c;
        }
        incl = kept;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) s_wsum[w] = incl;
    }
    __syncthreads();
    if (tid < 256) {
        int base = 0;
        for (int q = 0; q < w; ++q) base += s_wsum[q];
        const int excl = base + incl - kept;
        if (tid < E) {
            a.counts[tid] = tot[tid];
            a.offsets[tid] = excl;
            s_off[tid] = excl;
        }
        if (tid == E - 1) a.offsets[E] = excl + kept;
    }
    __syncthreads();
}

// All slots fit in one chunk: histogram, scan over experts and scatter in one block, with no
// look-back, flags or workspace.
// All slots fit in one chunk: histogram, scan over experts and scatter in one block of
// DISPATCH_THREADS threads, with no look-back, flags or workspace. Shared memory: cnt[32 * 256],
// s_tot[256], s_off[257], s_wsum[8].
__device__ __forceinline__ void dispatch_single_block(const DispatchArgs &a, int32_t *cnt,
                                                      int32_t *s_tot, int32_t *s_off,
                                                      int32_t *s_wsum) {
    const int tid = threadIdx.x, E = a.E;
    int lrank, agg;
    const int e = chunk_ranks(a, 0, cnt, &lrank, &agg);
    if (tid < E) s_tot[tid] = agg;
    __syncthreads();
    publish_offsets(a, s_tot, s_off, s_wsum);
    if (e >= 0) {
        if (a.cap >= 0 && lrank >= a.cap) {
            a.slot_of[tid] = -1;  // over capacity: dropped
        } else {
            const int pos = s_off[e] + lrank;
            a.sorted_token[pos] = tid / a.k;
            a.slot_of[tid] = pos;
        }
    }
}

// Sum over the 32 lanes of a warp by an xor butterfly: a fixed order, the same result in every
// lane.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// aux = E * sum_e (counts[e] / (T k)) * (sum_b psum_part[b, e] / T) and the router z-loss
// (sum_b psum_part[b, E]) / T, reduced in a fixed order:
//   1. thread (g, c) sums rows g, g + G, g + 2G, ... of column c (G = 1024 / (E + 1) groups)
//      into AUX_ILP running sums (row g + iG goes to sum i mod AUX_ILP, that many loads in
//      flight), added pairwise at the end;
//   2. warp w takes columns w, w + 32, ...: lane l adds group sums l, l + 32, ..., then the warp
//      adds its lanes by a butterfly;
//   3. warp 0 forms the E terms f_e P_e (lane l: experts l, l + 32, ...) and adds them likewise.
// Every step is a tree or a short chain, so the kernel is a few memory latencies long.
constexpr int AUX_ILP = 16;  // a power of two

// The auxiliary value and z-loss reduction above, by one block of 1024 threads. psum_part is read
// with plain (coherent) loads, so the same block may have written it. Shared memory: part[1024],
// colsum[257], s_counts[256].
__device__ __forceinline__ void aux_block(const int32_t *counts, const float *psum, int64_t rows,
                                          int E, int64_t T, int k, float *aux_out,
                                          float *zloss_out, float *part, float *colsum,
                                          int32_t *s_counts) {
    const int C = E + 1;
    const int G = 1024 / C;
    const int g = threadIdx.x / C, col = threadIdx.x % C;
    if ((int)threadIdx.x < E) s_counts[threadIdx.x] = counts[threadIdx.x];
    if (g < G) {
        float r[AUX_ILP];
#pragma unroll
        for (int u = 0; u < AUX_ILP; ++u) r[u] = 0.f;
        int64_t b = g;
        for (; b + (AUX_ILP - 1) * (int64_t)G < rows; b += AUX_ILP * (int64_t)G) {
#pragma unroll
            for (int u = 0; u < AUX_ILP; ++u) r[u] += (psum[(b + u * (int64_t)G) * C + col]);
        }
#pragma unroll
        for (int u = 0; u < AUX_ILP - 1; ++u)
            if (b + u * (int64_t)G < rows) r[u] += (psum[(b + u * (int64_t)G) * C + col]);
#pragma unroll
        for (int w = AUX_ILP / 2; w > 0; w >>= 1)  // pairwise: r[u] += r[u + w]
#pragma unroll
            for (int u = 0; u < w; ++u) r[u] += r[u + w];
        part[g * C + col] = r[0];
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int c = warp; c < C; c += 32) {
        float v = 0.f;
        for (int q = lane; q < G; q += 32) v += part[q * C + c];
        v = warp_sum(v);
        if (lane == 0) colsum[c] = v;
    }
    __syncthreads();
    if (warp == 0) {
        const float fT = (float)T, fTk = (float)T * (float)k;
        float v = 0.f;
        for (int e = lane; e < E; e += 32) v += ((float)s_counts[e] / fTk) * (colsum[e] / fT);
        v = warp_sum(v);
        if (lane == 0) {
            *aux_out = T > 0 ? (float)E * v : 0.f;
            if (zloss_out) *zloss_out = T > 0 ? colsum[E] / fT : 0.f;
        }
    }
}

}  // namespace dev
}  // namespace moe
