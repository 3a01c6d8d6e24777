// Token -> expert bucketing: a stable counting sort of the T*k (token, rank)
// pairs by expert id, in three passes over chunks of 1024 pairs:
//   count   per-chunk histograms (shared-memory atomics),
//   scan    totals, exclusive offsets, and each chunk's starting position
//           for each expert (single CTA),
//   scatter each pair's position = chunk start + pairs of the same expert
//           earlier in the chunk (warp match + per-warp counts), which keeps
//           (token, rank) order within every expert.
#include "internal.h"

namespace moe {

constexpr int kBucketChunk = 1024; // pairs per chunk = threads per CTA

int bucket_chunks(int pairs) { return (pairs + kBucketChunk - 1) / kBucketChunk; }

__global__ void __launch_bounds__(kBucketChunk) bucket_count_kernel(const int32_t *__restrict__ idx,
                                                                    int P, int E,
                                                                    int32_t *__restrict__ chunk_hist)
{
    extern __shared__ int32_t hist[]; // [E]
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        hist[e] = 0;
    __syncthreads();
    const int p = blockIdx.x * kBucketChunk + threadIdx.x;
    if (p < P) {
        const int e = idx[p];
        if (e >= 0 && e < E)
            atomicAdd(&hist[e], 1);
        else
            record_error(MOE_ERR_DEVICE_FAULT);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_hist[(size_t)blockIdx.x * E + e] = hist[e];
}

// One CTA of 1024 threads, E <= 1024: thread e owns expert e.
__global__ void __launch_bounds__(1024) bucket_scan_kernel(int n_chunks, int E,
                                                           int32_t *__restrict__ chunk_hist,
                                                           int32_t *__restrict__ counts,
                                                           int32_t *__restrict__ offsets)
{
    __shared__ int32_t warp_tot[32];
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
    int total = 0;
    if (e < E)
        for (int c = 0; c < n_chunks; ++c)
            total += chunk_hist[(size_t)c * E + e];
    // block-wide exclusive scan of `total` over e
    int incl = total;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int u = __shfl_up_sync(0xFFFFFFFFu, v, o);
            if (lane >= o)
                v += u;
        }
        warp_tot[lane] = v; // inclusive over warps
    }
    __syncthreads();
    const int excl = incl - total + (warp > 0 ? warp_tot[warp - 1] : 0);
    if (e < E) {
        counts[e] = total;
        offsets[e] = excl;
        int run = excl;
        for (int c = 0; c < n_chunks; ++c) {
            const int v = chunk_hist[(size_t)c * E + e];
            chunk_hist[(size_t)c * E + e] = run;
            run += v;
        }
        if (e == E - 1)
            offsets[E] = excl + total;
    }
}

__global__ void __launch_bounds__(kBucketChunk) bucket_scatter_kernel(const int32_t *__restrict__ idx,
                                                                      int P, int k, int E,
                                                                      const int32_t *__restrict__ chunk_base,
                                                                      int32_t *__restrict__ perm_tok,
                                                                      int32_t *__restrict__ perm_rank)
{
    extern __shared__ int32_t cnt[]; // [32 warps][E]
    constexpr int NW = kBucketChunk / 32;
    for (int j = threadIdx.x; j < NW * E; j += blockDim.x)
        cnt[j] = 0;
    __syncthreads();
    const int p = blockIdx.x * kBucketChunk + threadIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int e = -1;
    if (p < P) {
        e = idx[p];
        if (e < 0 || e >= E)
            e = -1;
    }
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank_in_warp == 0)
        cnt[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) { // exclusive prefix over warps
        int run = 0;
        for (int w = 0; w < NW; ++w) {
            const int v = cnt[w * E + x];
            cnt[w * E + x] = run;
            run += v;
        }
    }
    __syncthreads();
    if (e >= 0) {
        const int pos = chunk_base[(size_t)blockIdx.x * E + e] + cnt[warp * E + e] + rank_in_warp;
        perm_tok[pos] = p / k;
        perm_rank[pos] = p - (p / k) * k;
    }
}

cudaError_t launch_bucket(const Shape &s, const int32_t *idx, int T, int32_t *counts,
                          int32_t *offsets, int32_t *perm_tok, int32_t *perm_rank,
                          int32_t *chunk_hist, cudaStream_t st)
{
    const int P = T * s.k;
    const int nc = bucket_chunks(P);
    if (nc == 0) {
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * s.E, st);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (s.E + 1), st);
        return e;
    }
    bucket_count_kernel<<<nc, kBucketChunk, s.E * sizeof(int32_t), st>>>(idx, P, s.E, chunk_hist);
    bucket_scan_kernel<<<1, 1024, 0, st>>>(nc, s.E, chunk_hist, counts, offsets);
    const size_t smem = (size_t)(kBucketChunk / 32) * s.E * sizeof(int32_t);
    static int cur_smem = 0;
    cudaError_t e = ensure_smem(bucket_scatter_kernel, smem, &cur_smem);
    if (e != cudaSuccess)
        return e;
    bucket_scatter_kernel<<<nc, kBucketChunk, smem, st>>>(idx, P, s.k, s.E, chunk_hist, perm_tok, perm_rank);
    return cudaGetLastError();
}

} // namespace moe
