// align.cu -- K2: group the N*k (token, slot) pairs by expert.
//
// The grouping bookkeeping of the M03 "Sparse MoE" drill (step-by-step
// section): flatten the pairs row-major (p = n*k + j), sort them by expert
// with a STABLE order, count the pairs of every expert (bincount) and take
// prefix sums as segment starts; plus FusedMoE's moe_align_block_size step
// (named in the drill's shape-trace section): every expert segment is padded
// to the GEMM row block, padding slots hold the sentinel P = N*k, and every
// row block records its expert.  Experts with no pairs own no block.
//
// Three deterministic passes, none of which uses atomics to order outputs:
//   count:   CTA c histograms pairs [c*chunk, (c+1)*chunk) in shared memory
//   scan:    one CTA: per-expert exclusive scan over chunks (in place),
//            counts, offsets, padded offsets, block owners, sentinels
//   scatter: CTA c ranks each of its pairs among the same-expert pairs before
//            it (warp match + per-warp tallies), so pair p lands at
//            pad_off[e] + #{p' < p : expert(p') = e}: a stable order.
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kAlignThreads = 256;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kAlignThreads)
    align_count_kernel(const int32_t *__restrict__ ids, int64_t P, int E, int chunk,
                       int32_t *__restrict__ chunk_counts, int32_t *status) {
    extern __shared__ int32_t hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int64_t start = static_cast<int64_t>(blockIdx.x) * chunk;
    const int64_t end = min(P, start + chunk);
    bool bad = false;
    for (int64_t p = start + threadIdx.x; p < end; p += blockDim.x) {
        const int e = ids[p];
        if (e < 0 || e >= E) {
            bad = true;
            continue;
        }
        atomicAdd(&hist[e], 1);  // a count: order-free, exact
    }
    if (bad) record_status(status, MOE_ERR_DEVICE_CHECK);
    __syncthreads();
    int32_t *dst = chunk_counts + static_cast<int64_t>(blockIdx.x) * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) dst[e] = hist[e];
}

// Exclusive scan of one value per thread over the whole CTA (blockDim 1024).
__device__ int32_t block_exclusive_scan(int32_t v, int32_t *warp_sums, int32_t *total) {
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    int32_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += t;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t w = lane < (blockDim.x / 32) ? warp_sums[lane] : 0;
        int32_t wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t t = __shfl_up_sync(0xffffffffu, wi, d);
            if (lane >= d) wi += t;
        }
        warp_sums[lane] = wi - w;  // exclusive prefix of the warp totals
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const int32_t r = warp_sums[warp] + incl - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kScanThreads)
    align_scan_kernel(int32_t *__restrict__ chunk_counts, int nchunks, int E, int block_m,
                      int64_t P, int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                      int32_t *__restrict__ pad_offsets, int32_t *__restrict__ num_padded,
                      int32_t *__restrict__ block_expert, int32_t *__restrict__ sorted_pair) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t total;
    const int e = threadIdx.x;
    int32_t cnt = 0;
    if (e < E) {
        // per-expert exclusive scan over chunks, in place: count -> base
        for (int c = 0; c < nchunks; ++c) {
            int32_t *slot = chunk_counts + static_cast<int64_t>(c) * E + e;
            const int32_t v = *slot;
            *slot = cnt;
            cnt += v;
        }
    }
    const int32_t seg = (cnt + block_m - 1) / block_m * block_m;
    const int32_t off = block_exclusive_scan(cnt, warp_sums, &total);
    const int32_t pad = block_exclusive_scan(seg, warp_sums, &total);
    if (e < E) {
        counts[e] = cnt;
        offsets[e] = off;
        pad_offsets[e] = pad;
        if (e == E - 1) {
            offsets[E] = off + cnt;
            pad_offsets[E] = pad + seg;
            *num_padded = pad + seg;
        }
        for (int32_t b = pad / block_m; b < (pad + seg) / block_m; ++b) block_expert[b] = e;
        for (int32_t i = pad + cnt; i < pad + seg; ++i) sorted_pair[i] = static_cast<int32_t>(P);
    }
}

__global__ void __launch_bounds__(kAlignThreads)
    align_scatter_kernel(const int32_t *__restrict__ ids, int64_t P, int E, int chunk,
                         const int32_t *__restrict__ chunk_base,
                         const int32_t *__restrict__ pad_offsets,
                         int32_t *__restrict__ sorted_pair) {
    extern __shared__ int32_t sh[];
    int32_t *running = sh;                 // [E] next destination of each expert
    int32_t *warp_cnt = sh + E;            // [kAlignWarps][E]
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    const int64_t start = static_cast<int64_t>(blockIdx.x) * chunk;
    const int64_t end = min(P, start + chunk);
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        running[e] = pad_offsets[e] + chunk_base[static_cast<int64_t>(blockIdx.x) * E + e];
    for (int i = threadIdx.x; i < kAlignWarps * E; i += blockDim.x) warp_cnt[i] = 0;
    __syncthreads();
    const uint32_t lanes_below = (1u << lane) - 1u;
    for (int64_t base = start; base < end; base += blockDim.x) {
        const int64_t p = base + threadIdx.x;
        int e = p < end ? ids[p] : -1;
        const bool valid = e >= 0 && e < E;
        // lanes that are not real pairs get keys no real expert can match
        const uint32_t peers = __match_any_sync(0xffffffffu, valid ? e : E + lane);
        const int rank_in_warp = __popc(peers & lanes_below);
        if (valid && rank_in_warp == 0) warp_cnt[warp * E + e] = __popc(peers);
        __syncthreads();
        if (valid) {
            int32_t before = 0;
            for (int w = 0; w < warp; ++w) before += warp_cnt[w * E + e];
            sorted_pair[running[e] + before + rank_in_warp] = static_cast<int32_t>(p);
        }
        __syncthreads();
        for (int x = threadIdx.x; x < E; x += blockDim.x) {
            int32_t tot = 0;
            for (int w = 0; w < kAlignWarps; ++w) {
                tot += warp_cnt[w * E + x];
                warp_cnt[w * E + x] = 0;
            }
            running[x] += tot;
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_align(const AlignArgs &a, cudaStream_t s, int *launches) {
    const size_t count_smem = sizeof(int32_t) * a.E;
    align_count_kernel<<<a.nchunks, kAlignThreads, count_smem, s>>>(a.ids, a.P, a.E, a.chunk,
                                                                     a.chunk_counts, a.status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    align_scan_kernel<<<1, kScanThreads, 0, s>>>(a.chunk_counts, a.nchunks, a.E, a.block_m,
                                                 a.P, a.counts, a.offsets, a.pad_offsets,
                                                 a.num_padded, a.block_expert, a.sorted_pair);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const size_t scatter_smem = sizeof(int32_t) * (a.E + kAlignWarps * a.E);
    if (scatter_smem > 48 * 1024) {
        err = cudaFuncSetAttribute(align_scatter_kernel,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(scatter_smem));
        if (err != cudaSuccess) return err;
    }
    align_scatter_kernel<<<a.nchunks, kAlignThreads, scatter_smem, s>>>(
        a.ids, a.P, a.E, a.chunk, a.chunk_counts, a.pad_offsets, a.sorted_pair);
    *launches += 3;
    return cudaGetLastError();
}

}  // namespace moe
