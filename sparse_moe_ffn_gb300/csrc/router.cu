// router.cu -- K1: fused router GEMM + fp32 softmax over all experts + top-k
// + optional renormalisation (+ the talker's scalar shared-expert gate).
//
// Follows the routing block of the M03 "Sparse MoE" drill (problem overview):
// logits = x @ router^T, softmax over all E in fp32, top-k in descending
// order, w /= sum(w) when norm_topk_prob; weights are also returned in bf16
// (the pages return them in x's dtype) and ids as int32.  The shared gate is
// sigmoid(x . g), one scalar per token (same page, shared-expert line).
//
// A cluster of `split` CTAs (1, 2, 4 or 8, chosen from H alone) owns 128
// tokens; CTA c of the cluster takes the c-th slice of H.  Each CTA streams x
// [128 x 64] and router [e_pad x 64] slices through a TMA ring into one
// tcgen05 MMA chain (M = 128 tokens, N = e_pad experts, plus g in column
// gamma_col), so its TMEM holds the partial logits of its H slice.  CTA c
// reduces token rows [16c, 16c + 16) (all 128 rows, in 16-row passes, when
// split = 1): every CTA stores its partial rows into the reducing CTA's shared
// memory with distributed-shared-memory stores, and after a cluster barrier
// the reducer sums the `split` partial rows in rank order from local memory.
// 8 lanes per row and 4 rows per warp run the softmax, the k arg-max rounds
// and the renormalisation with shuffle reductions.  Every reduction order depends
// on H and E only, never on N: routing is batch invariant bit for bit.
#include <cuda_bf16.h>
#include <math.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kRouterStages = 3;  // ~99 KB per CTA at E = 128: two CTAs per SM
constexpr int kRouterThreads = 128;
constexpr int kATileBytes = kBlockM * 128;  // 128 tokens x 64 bf16
constexpr int kLanesPerRow = 8;                           // lanes sharing one token row
constexpr int kRowsPerPass = kRouterThreads / kLanesPerRow;  // 16 rows per pass

struct RouterSmem {
    uint64_t full[kRouterStages];
    uint64_t empty[kRouterStages];
    uint64_t acc_full;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ float finite_or_neg_inf(float v) {
    return (v != v) ? -INFINITY : v;  // NaN never wins a comparison
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory address of `local` in cluster CTA `rank`.  The loads below
// are volatile (so they stay after the cluster barrier) but carry no memory
// clobber, so that many of them are in flight at once.
__device__ __forceinline__ uint32_t dsmem_addr(const void *local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    return remote;
}

__device__ __forceinline__ void st_dsmem_f4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// Exclusive scan over the CTA (128 threads) of two consecutive values per
// thread (v0, v1 at positions 2t, 2t+1); returns the prefix of v0 and sets
// *total.  `sums` holds 4 ints of shared memory.
__device__ __forceinline__ int32_t cta_scan2(int32_t v0, int32_t v1, int32_t *sums,
                                             int32_t *total) {
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    const int32_t own = v0 + v1;
    int32_t incl = own;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += t;
    }
    if (lane == 31) sums[warp] = incl;
    __syncthreads();
    int32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kRouterThreads / 32; ++w) {
        if (w < warp) before += sums[w];
        all += sums[w];
    }
    __syncthreads();
    *total = all;
    return before + incl - own;
}

// The grouping of moe_align (block size 128) done by the routing cluster
// when it routes every token (N <= 128), instead of by another launch.
// Definition (M03 "serving way": bincount, prefix offsets, stable order):
// counts[e] = pairs with expert e; offsets = exclusive prefix of counts;
// each expert with pairs owns one 128-row block (counts <= N <= 128), in
// expert order (pad_offsets); its pairs fill the block in ascending
// p = n*k + j, then the sentinel P; block_expert[b] = the block's expert.
// CTA r of the cluster routed tokens [r*rows, (r+1)*rows), i.e. pairs
// [r*rows*k, (r+1)*rows*k) in p order, so a pair's row in its block is
// (its expert's pairs in the CTAs before r) + (those before it in CTA r):
//   1. each CTA counts its pairs per expert and pushes the counts into the
//      table `tbl` [split][E] of every CTA of the cluster (DSMEM stores);
//   2. after a cluster barrier each CTA scans the table itself (no second
//      exchange), and places its own pairs with warp match + per-warp counts;
//   3. CTA r writes the per-expert outputs of experts e = r mod split, CTA 0
//      the totals, and every CTA zeroes its share of the hand-off counters.
// An id outside [0, E) (only a broken routing could write one) is skipped
// and reported as MOE_ERR_DEVICE_CHECK.
// local_ids: this CTA's ids in shared memory (pair i of the CTA at [i]) when
// one 16-row pass routed all its rows, else null (read back from topk_ids).
__device__ __noinline__ void cluster_group(const RouterArgs &a, uint32_t crank, int rows_per_cta,
                                           int32_t *tbl, int32_t *scratch,
                                           const int32_t *local_ids) {
    const int E = a.E;
    const int k = a.k;
    const int tid = threadIdx.x;
    const int lane = tid % 32, warp = tid / 32;
    constexpr int kWarps = kRouterThreads / 32;
    const int64_t P = a.N * k;
    const int64_t row0 = static_cast<int64_t>(crank) * rows_per_cta;
    const int64_t live = a.N > row0 ? min(static_cast<int64_t>(rows_per_cta), a.N - row0) : 0;
    const int64_t p0 = row0 * k;
    const int np = static_cast<int>(live) * k;
    // scratch (this CTA's partial rows are no longer read): per-expert
    // counts, totals, running positions, per-warp counts of a chunk
    int32_t *hist = scratch;                 // [256]
    int32_t *tot = hist + 256;               // [256]
    int32_t *run = tot + 256;                // [256]
    int32_t *padv = run + 256;               // [256]
    int32_t *warp_cnt = padv + 256;          // [kWarps][256]
    int32_t *sums = warp_cnt + kWarps * 256; // [4]
    for (int e = tid; e < 256; e += kRouterThreads) hist[e] = 0;
    for (int i = tid; i < kWarps * 256; i += kRouterThreads) warp_cnt[i] = 0;
    __syncthreads();
    bool bad = false;
    auto id_of = [&](int i) -> int32_t {
        return local_ids ? local_ids[i] : __ldcg(a.topk_ids + p0 + i);
    };
    for (int i = tid; i < np; i += kRouterThreads) {
        const int32_t e = id_of(i);
        if (e < 0 || e >= E) bad = true;
        else atomicAdd(&hist[e], 1);
    }
    if (bad) record_status(a.status, MOE_ERR_DEVICE_CHECK);
    __syncthreads();
    // 1. this CTA's counts into slot [crank] of every CTA's table
    for (int e = tid; e < E; e += kRouterThreads) {
        const int32_t v = hist[e];
        for (int r = 0; r < a.split; ++r)
            asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(
                             dsmem_addr(&tbl[crank * E + e], static_cast<uint32_t>(r))),
                         "r"(v)
                         : "memory");
    }
    cluster_sync();  // every table is complete
    // 2. totals, prefix offsets, padded offsets and this CTA's start rows
    int32_t c2[2], before2[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int e = 2 * tid + u;
        int32_t c = 0, b = 0;
        if (e < E)
            for (int r = 0; r < a.split; ++r) {
                const int32_t v = tbl[r * E + e];
                c += v;
                if (r < static_cast<int>(crank)) b += v;
            }
        c2[u] = c;
        before2[u] = b;
    }
    int32_t total_pairs, total_pad;
    const int32_t off0 = cta_scan2(c2[0], c2[1], sums, &total_pairs);
    const int32_t seg0 = c2[0] > 0 ? kBlockM : 0, seg1 = c2[1] > 0 ? kBlockM : 0;
    const int32_t pad0 = cta_scan2(seg0, seg1, sums, &total_pad);
    const int32_t offs[2] = {off0, off0 + c2[0]};
    const int32_t pads[2] = {pad0, pad0 + seg0};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int e = 2 * tid + u;
        if (e >= E) continue;
        tot[e] = c2[u];
        padv[e] = pads[u];
        run[e] = pads[u] + before2[u];
        // 3. experts of this CTA's share: counts, offsets, blocks, sentinels
        if (e % a.split == static_cast<int>(crank)) {
            a.counts[e] = c2[u];
            a.offsets[e] = offs[u];
            a.pad_offsets[e] = pads[u];
            if (c2[u] > 0) a.block_expert[pads[u] / kBlockM] = e;
        }
    }
    if (crank == 0 && tid == 0) {
        a.offsets[E] = total_pairs;
        a.pad_offsets[E] = total_pad;
        *a.num_padded = total_pad;
    }
    // the hand-off counters start from zero every call (the previous call's
    // GEMMs are complete: routing waited for them)
    for (int i = static_cast<int>(crank) * kRouterThreads + tid; i < a.ready_n;
         i += a.split * kRouterThreads)
        a.ready[i] = 0;
    __syncthreads();
    // sentinels: the rows of each block past its pairs (experts of this
    // CTA's share, 128 rows each, spread over the threads)
    const int share = (E - static_cast<int>(crank) + a.split - 1) / a.split;
    for (int idx = tid; idx < share * kBlockM; idx += kRouterThreads) {
        const int e = static_cast<int>(crank) + a.split * (idx / kBlockM);
        const int r = idx % kBlockM;
        if (tot[e] > 0 && r >= tot[e]) a.sorted_pair[padv[e] + r] = static_cast<int32_t>(P);
    }
    // stable placement of this CTA's pairs, 128 at a time in p order
    const uint32_t lanes_below = (1u << lane) - 1u;
    for (int c0 = 0; c0 < np; c0 += kRouterThreads) {
        const int i = c0 + tid;
        const int32_t e = i < np ? id_of(i) : -1;
        const bool valid = e >= 0 && e < E;
        const uint32_t peers = __match_any_sync(0xffffffffu, valid ? e : E + lane);
        const int rank = __popc(peers & lanes_below);
        if (valid && rank == 0) warp_cnt[warp * 256 + e] = __popc(peers);
        __syncthreads();
        if (valid) {
            int32_t before = 0;
            for (int w = 0; w < warp; ++w) before += warp_cnt[w * 256 + e];
            a.sorted_pair[run[e] + before + rank] = static_cast<int32_t>(p0 + i);
        }
        __syncthreads();
        for (int x = tid; x < E; x += kRouterThreads) {
            int32_t t = 0;
            for (int w = 0; w < kWarps; ++w) {
                t += warp_cnt[w * 256 + x];
                warp_cnt[w * 256 + x] = 0;
            }
            run[x] += t;
        }
        __syncthreads();
    }
}

// PL: logits per lane (e_pad / 8 rounded up to 4, 16 or 32), a compile-time
// bound so that the per-round scans cover only the columns that exist.
template <int PL>
__global__ void __launch_bounds__(kRouterThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap tm_x,
                  const __grid_constant__ CUtensorMap tm_router,
                  const __grid_constant__ CUtensorMap tm_gate, const RouterArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int b_tile_bytes = a.e_pad * 128;
    const int stage_bytes = kATileBytes + b_tile_bytes;
    const int ring_bytes = kRouterStages * stage_bytes;
    const int part_bytes = kBlockM * (a.e_pad + 4) * 4 + kRowsPerPass * a.k * 8;
    // fused grouping: every CTA's expert histogram, pushed into every CTA
    // of the cluster; kept clear of the partial rows, which peers may still
    // be reading while a fast CTA pushes its histogram
    const int tbl_off = (part_bytes + 15) / 16 * 16;
    const int tbl_bytes = a.fuse_align ? a.split * a.E * 4 : 0;
    const int body_bytes = tbl_off + tbl_bytes > ring_bytes ? tbl_off + tbl_bytes : ring_bytes;
    RouterSmem *sm = reinterpret_cast<RouterSmem *>(
        tiles + (body_bytes > part_bytes ? body_bytes : part_bytes));
    float *partial = reinterpret_cast<float *>(tiles);  // reuses the ring once it is idle
    const int ld = a.e_pad + 4;                          // row stride of the partial tile

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t crank = cluster_rank();
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kBlockM;
    const int nk = (a.H + kBlockK - 1) / kBlockK;
    const int kc0 = static_cast<int>(crank) * nk / a.split;
    const int kc1 = static_cast<int>(crank + 1) * nk / a.split;
    const int my_nk = kc1 - kc0;  // >= 1 because split <= nk
    const uint32_t tmem_cols = a.e_pad <= 32 ? 32 : (a.e_pad <= 64 ? 64 : (a.e_pad <= 128 ? 128 : 256));

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRouterStages; ++s) {
            mbar_init(&sm->full[s], 1);
            mbar_init(&sm->empty[s], 1);
        }
        mbar_init(&sm->acc_full, 1);
        mbar_init(&sm->drain, 1);
        sm->abort_flag = 0;
        fence_barrier_init();
        prefetch_tensor_map(&tm_x);
        prefetch_tensor_map(&tm_router);
        if (a.gamma_col >= 0) prefetch_tensor_map(&tm_gate);
    }
    if (warp == 0) {
        tmem_alloc(&sm->tmem_base, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm->tmem_base;
    volatile int *abort_flag = &sm->abort_flag;
    griddep_launch_dependents();
    griddep_wait();  // x may come from the previous kernel in the stream
    if (a.reset_status && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 && a.status)
        *a.status = 0;

    if (warp == 0) {
        // ---------------- TMA producer: this CTA's slice of H
        if (lane == 0) {
            const uint32_t tx = kATileBytes + a.E * 128 + (a.gamma_col >= 0 ? 8 * 128 : 0);
            // the router (and gate) rows are re-read by every layer call: keep them in L2
            const uint64_t keep = l2_policy_evict_last();
            int i = 0;
            for (; i < my_nk; ++i) {
                const int s = i % kRouterStages;
                const uint32_t use = i / kRouterStages;
                if (use > 0 && !mbar_wait(&sm->empty[s], (use - 1) & 1, abort_flag)) {
                    record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                uint8_t *st = tiles + s * stage_bytes;
                const int kcol = (kc0 + i) * kBlockK;
                mbar_arrive_expect_tx(&sm->full[s], tx);
                tma_load_2d(st, &tm_x, &sm->full[s], kcol, static_cast<int>(n0));
                tma_load_2d_hint(st + kATileBytes, &tm_router, &sm->full[s], kcol, 0, keep);
                if (a.gamma_col >= 0)
                    tma_load_2d_hint(st + kATileBytes + a.gamma_col * 128, &tm_gate, &sm->full[s],
                                     kcol, 0, keep);
            }
            for (int j = (i > kRouterStages ? i - kRouterStages : 0); j < i; ++j)
                mbar_wait(&sm->full[j % kRouterStages], (j / kRouterStages) & 1, abort_flag);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kBlockM, a.e_pad);
            for (int i = 0; i < my_nk; ++i) {
                const int s = i % kRouterStages;
                if (!mbar_wait(&sm->full[s], (i / kRouterStages) & 1, abort_flag)) {
                    record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after_sync();
                const uint8_t *st = tiles + s * stage_bytes;
                const uint64_t da = sw128_kmajor_desc(smem_addr(st));
                const uint64_t db = sw128_kmajor_desc(smem_addr(st + kATileBytes));
#pragma unroll
                for (int kk = 0; kk < kBlockK / 16; ++kk)
                    mma_f16kind(tmem, da + 2 * kk, db + 2 * kk, idesc, (i | kk) != 0);
                mma_commit(&sm->empty[s]);
            }
            mma_commit(&sm->acc_full);
            mma_commit(&sm->drain);
            mbar_wait(&sm->drain, 0, abort_flag);
        }
        __syncwarp();
    }

    // ---------------- phase 1: partial logits -> the shared memory of the CTA
    // that reduces them.  Token row r belongs to cluster CTA r / rows_per_cta;
    // each CTA stores its partial row there, into slot [own rank][row], with
    // remote stores (no round trip), so the reduction reads local memory.
    const bool ok = mbar_wait(&sm->acc_full, 0, abort_flag);
    __syncwarp();
    if (!ok) {
        record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
    }
    tc_fence_after_sync();
    const int rows_per_cta = kBlockM / a.split;
    // every ring of the cluster is idle before any CTA writes into a peer's
    cluster_sync();
    // a warp whose 32 token rows are all past N skips the push; inside a
    // warp the TMEM loads stay warp-wide (tcgen05.ld is a .sync.aligned
    // collective) and only the stores of rows past N are dropped
    if (n0 + warp * 32 < a.N) {
        const int row = warp * 32 + lane;  // TMEM lane
        const bool live_row = n0 + row < a.N;
        const uint32_t owner = static_cast<uint32_t>(row / rows_per_cta);
        const int slot = static_cast<int>(crank) * rows_per_cta + row % rows_per_cta;
        const uint32_t dst = dsmem_addr(&partial[slot * ld], owner);
        const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        for (int c = 0; c < (a.e_pad + 31) / 32; ++c) {
            float v[32];
            tmem_load32(trow + c * 32, v);
            tmem_load_wait();
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                if (live_row && c * 32 + i < a.e_pad)
                    st_dsmem_f4(dst + 4 * (c * 32 + i),
                                ok ? make_float4(v[i], v[i + 1], v[i + 2], v[i + 3])
                                   : make_float4(0.f, 0.f, 0.f, 0.f));
        }
    }
    tc_fence_before_sync();
    cluster_sync();  // every partial row has reached its reducer

    // ---------------- phase 2: reduce over the cluster, then route
    // 8 lanes per token row, 4 rows per warp, 16 rows per pass.  Lane `sub`
    // owns the float4 column groups 32i + 4*sub (i < e_pad/32), so each 8-lane
    // group reads 128 contiguous bytes of a partial row per load.  The
    // `split` partials are summed in rank order.
    const int sub = lane % kLanesPerRow;
    const int groups = (a.e_pad + 31) / 32;
    float *slot_w = partial + kBlockM * ld;                              // [16][k]
    int32_t *slot_e = reinterpret_cast<int32_t *>(slot_w + kRowsPerPass * a.k);  // [16][k]
    for (int base = 0; base < rows_per_cta; base += kRowsPerPass) {
        // rows are consecutive tokens: a pass that starts past N has no live row
        if (n0 + static_cast<int>(crank) * rows_per_cta + base >= a.N) break;
        const int rl = warp * (32 / kLanesPerRow) + lane / kLanesPerRow;  // row in pass
        const int row = static_cast<int>(crank) * rows_per_cta + base + rl;
        const int64_t n = n0 + row;
        const bool live = n < a.N;
        float lg[PL];
#pragma unroll
        for (int j = 0; j < PL; ++j) lg[j] = 0.f;
        for (int r = 0; r < a.split; ++r) {
            const float *src = &partial[(r * rows_per_cta + base + rl) * ld + 4 * sub];
            float4 t[PL / 4];
#pragma unroll
            for (int i = 0; i < PL / 4; ++i)
                if (i < groups && 32 * i + 4 * sub < a.e_pad)
                    t[i] = *reinterpret_cast<const float4 *>(src + 32 * i);
#pragma unroll
            for (int i = 0; i < PL / 4; ++i)
                if (i < groups && 32 * i + 4 * sub < a.e_pad) {
                    lg[4 * i + 0] += t[i].x;
                    lg[4 * i + 1] += t[i].y;
                    lg[4 * i + 2] += t[i].z;
                    lg[4 * i + 3] += t[i].w;
                }
        }
        // the shared gate logit lives in one lane's columns
        if (a.gamma_col >= 0 && live && (a.gamma_col % 32) / 4 == sub) {
            const int jg = 4 * (a.gamma_col / 32) + a.gamma_col % 4;
            float lgate = 0.f;
#pragma unroll
            for (int j = 0; j < PL; ++j)
                if (j == jg) lgate = lg[j];
            const float gam = 1.f / (1.f + expf(-lgate));
            a.gamma[n] = gam;
            for (int c = 0; c < a.virt_slots; ++c) {  // the shared expert's chunks
                a.topk_w[n * a.out_ld + a.k + c] = gam;
                a.topk_ids[n * a.out_ld + a.k + c] = a.virt_base + c;
            }
        }
#pragma unroll
        for (int j = 0; j < PL; ++j) {
            const int e = 32 * (j / 4) + 4 * sub + j % 4;
            lg[j] = e < a.E ? finite_or_neg_inf(lg[j]) : -INFINITY;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < PL; ++j) mx = fmaxf(mx, lg[j]);
#pragma unroll
        for (int d = kLanesPerRow / 2; d > 0; d >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d, kLanesPerRow));
        // fast exponentials: their relative error (~1e-6 over the logit
        // range of a softmax) is far below the weights' fp32 budget
        float den = 0.f;
#pragma unroll
        for (int j = 0; j < PL; ++j) {
            const int e = 32 * (j / 4) + 4 * sub + j % 4;
            if (e < a.E) den += __expf(lg[j] - mx);
        }
#pragma unroll
        for (int d = kLanesPerRow / 2; d > 0; d >>= 1)
            den += __shfl_xor_sync(0xffffffffu, den, d, kLanesPerRow);
        const float inv_den = 1.f / den;
        // k arg-max rounds; exp is monotone, so this is the top-k of the
        // probabilities.  A lane's candidates are reduced as a tournament
        // (log2(PL) levels of max instead of a PL-long dependent chain),
        // then across the row's 8 lanes; a selected key becomes 0, so it
        // never wins again.  Each candidate is one 64-bit key: the logit mapped to an unsigned
        // integer of the same order (its sign bit flipped, or all bits for
        // a negative value; -0 first made +0, which compares equal), then
        // 255 - e, so that an equal logit ranks the lower expert first; 0
        // means "none" (past E, or already taken).  The keys order the
        // candidates exactly as (larger logit, then lower expert).
        uint64_t key[PL];
#pragma unroll
        for (int j = 0; j < PL; ++j) {
            const int e = 32 * (j / 4) + 4 * sub + j % 4;
            const uint32_t u = __float_as_uint(lg[j] + 0.f);
            const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
            key[j] = e < a.E ? (static_cast<uint64_t>(ord) << 32) | static_cast<uint32_t>(255 - e)
                             : 0ull;
        }
        float wsum = 0.f;
        for (int r = 0; r < a.k; ++r) {
            uint64_t t[PL];
#pragma unroll
            for (int j = 0; j < PL; ++j) t[j] = key[j];
#pragma unroll
            for (int w = PL / 2; w > 0; w >>= 1)
#pragma unroll
                for (int j = 0; j < w; ++j) t[j] = t[j] > t[j + w] ? t[j] : t[j + w];
            uint64_t best = t[0];
#pragma unroll
            for (int d = kLanesPerRow / 2; d > 0; d >>= 1) {
                const uint64_t o = __shfl_xor_sync(0xffffffffu, best, d, kLanesPerRow);
                best = o > best ? o : best;
            }
#pragma unroll
            for (int j = 0; j < PL; ++j)
                if (key[j] == best) key[j] = 0ull;
            const int be = 255 - static_cast<int>(best & 0xFFu);
            const uint32_t ord = static_cast<uint32_t>(best >> 32);
            const float bv = __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
            const float p = __expf(bv - mx) * inv_den;
            wsum += p;
            if (sub == 0) {
                slot_w[rl * a.k + r] = p;
                slot_e[rl * a.k + r] = be;
            }
        }
        __syncwarp();
        if (live) {
            const float inv = a.norm ? 1.f / wsum : 1.f;
            for (int r = sub; r < a.k; r += kLanesPerRow) {
                const float w = slot_w[rl * a.k + r] * inv;
                a.topk_w[n * a.out_ld + r] = w;
                a.topk_ids[n * a.out_ld + r] = slot_e[rl * a.k + r];
                if (a.topk_w_bf16) {
                    __nv_bfloat16 h = __float2bfloat16_rn(w);
                    a.topk_w_bf16[n * a.out_ld + r] = *reinterpret_cast<uint16_t *>(&h);
                }
            }
        }
        __syncwarp();
    }
    __syncthreads();
    if (a.fuse_align)
        cluster_group(a, crank, rows_per_cta, reinterpret_cast<int32_t *>(tiles + tbl_off),
                      reinterpret_cast<int32_t *>(tiles),
                      rows_per_cta == kRowsPerPass ? slot_e : nullptr);
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, tmem_cols);
    }
}

}  // namespace

int router_split(int H) {
    const int nk = (H + kBlockK - 1) / kBlockK;
    return nk >= 8 ? 8 : (nk >= 4 ? 4 : (nk >= 2 ? 2 : 1));
}

int router_per_lane(int e_pad) {
    const int pl = (e_pad + kLanesPerRow - 1) / kLanesPerRow;
    return pl <= 4 ? 4 : (pl <= 16 ? 16 : 32);
}

size_t router_smem_bytes(int e_pad, int k, int table_bytes) {
    const size_t ring = static_cast<size_t>(kRouterStages) * (kATileBytes + e_pad * 128);
    // the partial tile, then the slot results of one 16-row pass; the fused
    // grouping's table after them (the kernel's layout)
    const size_t part = static_cast<size_t>(kBlockM) * (e_pad + 4) * sizeof(float) +
                        static_cast<size_t>(kRowsPerPass) * k * 8;
    const size_t table_end = (part + 15) / 16 * 16 + static_cast<size_t>(table_bytes);
    const size_t body = table_end > ring ? table_end : ring;
    return 1024 + (body > part ? body : part) + sizeof(RouterSmem);
}

cudaError_t launch_router(const CUtensorMap &tm_x, const CUtensorMap &tm_router,
                          const CUtensorMap &tm_gate, const RouterArgs &a, cudaStream_t s) {
    if (a.fuse_align && (a.N > kBlockM || a.E > 256 || a.virt_slots != 0 || a.out_ld != a.k))
        return cudaErrorInvalidValue;
    const size_t smem = router_smem_bytes(a.e_pad, a.k, a.fuse_align ? a.split * a.E * 4 : 0);
    const int pl = router_per_lane(a.e_pad);
    auto kern = pl == 4 ? router_kernel<4> : (pl == 16 ? router_kernel<16> : router_kernel<32>);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const dim3 grid(static_cast<unsigned>(a.split),
                    static_cast<unsigned>((a.N + kBlockM - 1) / kBlockM), 1);
    return launch_pdl(kern, grid, dim3(kRouterThreads), smem, s,
                      static_cast<unsigned>(a.split), tm_x, tm_router, tm_gate, a);
}

}  // namespace moe
