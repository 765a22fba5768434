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
// Large P: three deterministic passes, none of which uses atomics to order
// outputs:
//   count:   CTA c histograms pairs [c*chunk, (c+1)*chunk) in shared memory
//   scan:    one CTA: per-expert exclusive scan over chunks (in place),
//            counts, offsets, padded offsets
//   scatter: CTA c ranks each of its pairs among the same-expert pairs before
//            it (warp match + per-warp tallies), so pair p lands at
//            pad_off[e] + #{p' < p : expert(p') = e}: a stable order; CTA c
//            also writes the sentinel into the padding rows of experts
//            e = c (mod CTAs) and their blocks' owner, spreading that work
//            over all CTAs instead of the scan's single one.
// Small P (decode): the same steps inside one 1024-thread CTA, one launch.
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kAlignThreads = 256;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kScanThreads = 1024;
constexpr int kSmallPairs = 4096;  // single-CTA path up to this many pairs
constexpr int kSmallMaxE = 256;

__global__ void __launch_bounds__(kAlignThreads)
    align_count_kernel(const int32_t *__restrict__ ids, int64_t P, int E, int chunk,
                       int32_t *__restrict__ chunk_counts, int32_t *status) {
    griddep_launch_dependents();
    griddep_wait();
    extern __shared__ int32_t hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int64_t start = static_cast<int64_t>(blockIdx.x) * chunk;
    const int64_t end = min(P, start + chunk);
    bool bad = false;
    constexpr int kPerThread = kAlignChunk / kAlignThreads;
    int my_e[kPerThread];
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {  // every load in flight at once
        const int64_t p = start + threadIdx.x + static_cast<int64_t>(i) * kAlignThreads;
        my_e[i] = p < end ? __ldcg(ids + p) : 0;
    }
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int64_t p = start + threadIdx.x + static_cast<int64_t>(i) * kAlignThreads;
        if (p >= end) continue;
        if (my_e[i] < 0 || my_e[i] >= E) {
            bad = true;
            continue;
        }
        atomicAdd(&hist[my_e[i]], 1);  // a count: order-free, exact
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

// Expert owning padded slot `slot`: the last e with pad_off[e] <= slot
// (experts without pairs share their successor's offset and own nothing).
__device__ __forceinline__ int owner_of(const int32_t *pad_off, int E, int64_t slot) {
    int lo = 0, hi = E;  // answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) / 2;
        if (pad_off[mid] <= slot) lo = mid; else hi = mid;
    }
    return lo;
}

// every padded slot gets the sentinel P, every row block its owner expert
__device__ void fill_padded(const int32_t *pad_off_smem, int E, int block_m, int32_t num_padded,
                            int64_t P, int32_t *sorted_pair, int32_t *block_expert,
                            int32_t *ready) {
    // the GEMMs' hand-off counters (per expert or per block pair) start from
    // zero every call; the previous call's GEMMs are complete, since this
    // kernel follows routing, which followed the previous call's last kernel
    if (ready) {
        const int32_t n = E > num_padded / block_m ? E : num_padded / block_m;
        for (int32_t i = threadIdx.x; i < n; i += blockDim.x) ready[i] = 0;
    }
    for (int32_t i = threadIdx.x; i < num_padded; i += blockDim.x)
        sorted_pair[i] = static_cast<int32_t>(P);
    for (int32_t b = threadIdx.x; b < num_padded / block_m; b += blockDim.x)
        block_expert[b] = owner_of(pad_off_smem, E, static_cast<int64_t>(b) * block_m);
}

__global__ void __launch_bounds__(kScanThreads)
    align_scan_kernel(int32_t *__restrict__ chunk_counts, int nchunks, int E, int block_m,
                      int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                      int32_t *__restrict__ pad_offsets, int32_t *__restrict__ num_padded,
                      int32_t *__restrict__ ready) {
    griddep_launch_dependents();
    griddep_wait();
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t total;
    const int e = threadIdx.x;
    int32_t cnt = 0;
    if (e < E) {
        // per-expert exclusive scan over chunks, in place: count -> base.
        // kBatch independent loads are issued before their stores, so the
        // chunks cost nchunks / kBatch round trips to L2, not nchunks
        constexpr int kBatch = 16;
        for (int c0 = 0; c0 < nchunks; c0 += kBatch) {
            int32_t v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                v[u] = c0 + u < nchunks ? __ldcg(chunk_counts + static_cast<int64_t>(c0 + u) * E + e)
                                        : 0;
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (c0 + u < nchunks) {
                    chunk_counts[static_cast<int64_t>(c0 + u) * E + e] = cnt;
                    cnt += v[u];
                }
        }
    }
    const int32_t seg = (cnt + block_m - 1) / block_m * block_m;
    const int32_t off = block_exclusive_scan(cnt, warp_sums, &total);
    const int32_t pad = block_exclusive_scan(seg, warp_sums, &total);
    __shared__ int32_t npad;
    if (e < E) {
        counts[e] = cnt;
        offsets[e] = off;
        pad_offsets[e] = pad;
        if (e == E - 1) {
            offsets[E] = off + cnt;
            pad_offsets[E] = pad + seg;
            *num_padded = pad + seg;
            npad = pad + seg;
        }
    }
    __syncthreads();
    // the GEMMs' hand-off counters start from zero every call (see
    // fill_padded); the sentinels and block owners are written by the
    // scatter kernel's CTAs, expert by expert, next to the real pairs
    if (ready) {
        const int32_t n = E > npad / block_m ? E : npad / block_m;
        for (int32_t i = threadIdx.x; i < n; i += blockDim.x) ready[i] = 0;
    }
}

__global__ void __launch_bounds__(kAlignThreads)
    align_scatter_kernel(const int32_t *__restrict__ ids, int64_t P, int E, int chunk,
                         const int32_t *__restrict__ chunk_base,
                         const int32_t *__restrict__ pad_offsets,
                         const int32_t *__restrict__ counts, int block_m,
                         int32_t *__restrict__ sorted_pair, int32_t *__restrict__ block_expert) {
    griddep_launch_dependents();
    griddep_wait();
    // experts e = blockIdx.x (mod gridDim.x): the sentinel P in the rows of
    // their blocks past their pairs, and the blocks' owner (positions the
    // real pairs below never take, so no ordering is needed)
    for (int e = blockIdx.x; e < E; e += gridDim.x) {
        const int32_t p0 = __ldcg(pad_offsets + e), p1 = __ldcg(pad_offsets + e + 1);
        const int32_t c = __ldcg(counts + e);
        for (int32_t i = p0 + c + threadIdx.x; i < p1; i += blockDim.x)
            sorted_pair[i] = static_cast<int32_t>(P);
        for (int32_t b = p0 / block_m + threadIdx.x; b < p1 / block_m; b += blockDim.x)
            block_expert[b] = e;
    }
    extern __shared__ int32_t sh[];
    int32_t *running = sh;                 // [E] next destination of each expert
    int32_t *warp_cnt = sh + E;            // [kAlignWarps][E]
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    const int64_t start = static_cast<int64_t>(blockIdx.x) * chunk;
    const int64_t end = min(P, start + chunk);
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        running[e] = __ldcg(pad_offsets + e) +
                     __ldcg(chunk_base + static_cast<int64_t>(blockIdx.x) * E + e);
    for (int i = threadIdx.x; i < kAlignWarps * E; i += blockDim.x) warp_cnt[i] = 0;
    // the chunk's ids, all loaded up front (one round trip to memory)
    constexpr int kPerThread = kAlignChunk / kAlignThreads;
    int my_e[kPerThread];
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int64_t p = start + threadIdx.x + static_cast<int64_t>(i) * kAlignThreads;
        my_e[i] = p < end ? __ldcg(ids + p) : -1;
    }
    __syncthreads();
    const uint32_t lanes_below = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int64_t base = start + static_cast<int64_t>(i) * kAlignThreads;
        if (base >= end) break;  // uniform across the CTA
        const int64_t p = base + threadIdx.x;
        int e = p < end ? my_e[i] : -1;
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

// The whole grouping in one CTA (P <= kSmallPairs, E <= 256).
__global__ void __launch_bounds__(kScanThreads)
    align_small_kernel(const int32_t *__restrict__ ids, int64_t P, int E, int block_m,
                       int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                       int32_t *__restrict__ pad_offsets, int32_t *__restrict__ num_padded,
                       int32_t *__restrict__ sorted_pair, int32_t *__restrict__ block_expert,
                       int32_t *status, int32_t *__restrict__ ready) {
    griddep_launch_dependents();
    griddep_wait();
    __shared__ int32_t hist[kSmallMaxE];
    __shared__ int32_t pad_smem[kSmallMaxE + 1];
    __shared__ int32_t running[kSmallMaxE];
    __shared__ int32_t warp_cnt[kScanThreads / 32][kSmallMaxE];
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t total, npad;
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    for (int i = threadIdx.x; i < kSmallMaxE; i += blockDim.x) hist[i] = 0;
    for (int i = threadIdx.x; i < (kScanThreads / 32) * kSmallMaxE; i += blockDim.x)
        (&warp_cnt[0][0])[i] = 0;
    __syncthreads();
    // each thread keeps its (at most kSmallPairs / kScanThreads) ids in
    // registers for the scatter below: one round trip to memory, not two
    constexpr int kPerThread = kSmallPairs / kScanThreads;
    int my_e[kPerThread];
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int64_t p = threadIdx.x + static_cast<int64_t>(i) * kScanThreads;
        my_e[i] = p < P ? __ldcg(ids + p) : -1;
    }
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int64_t p = threadIdx.x + static_cast<int64_t>(i) * kScanThreads;
        if (p >= P) continue;
        if (my_e[i] < 0 || my_e[i] >= E) {
            bad = true;
            continue;
        }
        atomicAdd(&hist[my_e[i]], 1);
    }
    if (bad) record_status(status, MOE_ERR_DEVICE_CHECK);
    __syncthreads();
    const int e = threadIdx.x;
    const int32_t cnt = e < E ? hist[e] : 0;
    const int32_t seg = (cnt + block_m - 1) / block_m * block_m;
    const int32_t off = block_exclusive_scan(cnt, warp_sums, &total);
    const int32_t pad = block_exclusive_scan(seg, warp_sums, &total);
    if (e < E) {
        counts[e] = cnt;
        offsets[e] = off;
        pad_offsets[e] = pad;
        pad_smem[e] = pad;
        running[e] = pad;
        if (e == E - 1) {
            offsets[E] = off + cnt;
            pad_offsets[E] = pad + seg;
            *num_padded = pad + seg;
            npad = pad + seg;
        }
    }
    __syncthreads();
    fill_padded(pad_smem, E, block_m, npad, P, sorted_pair, block_expert, ready);
    __syncthreads();  // sentinels first, then the real pairs over them
    const uint32_t lanes_below = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int64_t base = static_cast<int64_t>(i) * kScanThreads;
        if (base >= P) break;  // uniform across the CTA
        const int64_t p = base + threadIdx.x;
        const int pe = p < P ? my_e[i] : -1;
        const bool valid = pe >= 0 && pe < E;
        const uint32_t peers = __match_any_sync(0xffffffffu, valid ? pe : E + lane);
        const int rank_in_warp = __popc(peers & lanes_below);
        if (valid && rank_in_warp == 0) warp_cnt[warp][pe] = __popc(peers);
        __syncthreads();
        if (valid) {
            int32_t before = 0;
            for (int w = 0; w < warp; ++w) before += warp_cnt[w][pe];
            sorted_pair[running[pe] + before + rank_in_warp] = static_cast<int32_t>(p);
        }
        __syncthreads();
        if (threadIdx.x < E) {
            int32_t tot = 0;
            for (int w = 0; w < kScanThreads / 32; ++w) {
                tot += warp_cnt[w][threadIdx.x];
                warp_cnt[w][threadIdx.x] = 0;
            }
            running[threadIdx.x] += tot;
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_align(const AlignArgs &a, cudaStream_t s, int *launches) {
    if (a.P <= kSmallPairs && a.E <= kSmallMaxE) {
        *launches += 1;
        return launch_pdl(align_small_kernel, dim3(1), dim3(kScanThreads), 0, s, 1, a.ids, a.P,
                          a.E, a.block_m, a.counts, a.offsets, a.pad_offsets, a.num_padded,
                          a.sorted_pair, a.block_expert, a.status, a.ready);
    }
    // the count and scatter kernels hold a chunk's ids in registers
    if (a.chunk != kAlignChunk) return cudaErrorInvalidValue;
    const size_t count_smem = sizeof(int32_t) * a.E;
    cudaError_t err = launch_pdl(align_count_kernel, dim3(a.nchunks), dim3(kAlignThreads),
                                 count_smem, s, 1, a.ids, a.P, a.E, a.chunk, a.chunk_counts,
                                 a.status);
    if (err != cudaSuccess) return err;
    err = launch_pdl(align_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, 1, a.chunk_counts,
                     a.nchunks, a.E, a.block_m, a.counts, a.offsets, a.pad_offsets,
                     a.num_padded, a.ready);
    if (err != cudaSuccess) return err;
    const size_t scatter_smem = sizeof(int32_t) * (a.E + kAlignWarps * a.E);
    if (scatter_smem > 48 * 1024) {
        err = cudaFuncSetAttribute(align_scatter_kernel,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(scatter_smem));
        if (err != cudaSuccess) return err;
    }
    *launches += 3;
    return launch_pdl(align_scatter_kernel, dim3(a.nchunks), dim3(kAlignThreads), scatter_smem,
                      s, 1, a.ids, a.P, a.E, a.chunk,
                      static_cast<const int32_t *>(a.chunk_counts),
                      static_cast<const int32_t *>(a.pad_offsets),
                      static_cast<const int32_t *>(a.counts), a.block_m, a.sorted_pair,
                      a.block_expert);
}

}  // namespace moe
