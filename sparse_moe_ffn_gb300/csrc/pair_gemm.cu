// pair_gemm.cu -- K3 (gate/up) and K4 (down) for workloads whose experts own
// several row blocks each (prefill): the two CTAs of a cluster run one
// tcgen05 MMA of M = 256 rows (cta_group::2) over two row blocks of the same
// expert, so every weight tile they fetch serves 256 rows instead of 128.
// The arithmetic per output element is the one-CTA kernel's (same K order,
// same epilogue, store_tile in gemm_common.cuh); only the tiling differs.
//
// Pair tiles.  Expert e owns row blocks [pad_off[e] / 128, pad_off[e+1] / 128)
// of the grouped layout; they are taken two at a time, so expert e has
// ceil(nb_e / 2) pairs.  An odd block count leaves the last pair with a CTA
// whose rows are all padding: that CTA loads no A rows but still loads its
// weight rows (the pair's MMA reads both CTAs' rows) and stores nothing.  A pair tile is (pair j, N tile nt); cluster c takes pair tiles c,
// c + #clusters, ...
//
// Operand split of a cta_group::2 MMA (M = 256, N columns): A rows 0-127 come
// from the even CTA's shared memory and rows 128-255 from the odd CTA's, at
// the same offset; the N weight rows are split the same way (rows [0, N/2)
// from the even CTA, [N/2, N) from the odd one); each CTA's TMEM receives
// its own 128 rows x N columns.  Every MMA has N = 256, the widest shape (two
// N = 128 MMAs keep the tensor pipe markedly less busy).  Per K slice each
// CTA therefore loads
//   gate/up (BN = 128): 16 KB of x rows + 16 KB of weights, Wg rows in the
//                       even CTA and Wu rows in the odd one, so that N = 256
//                       spans [gate | up] (32 KB, 6 stages);
//   down    (BN = 256): 16 KB of fp16 act rows + 16 KB of fp16 Wd rows
//                       (32 KB, 6 stages), fp16 x fp16 MMAs (kDown); or
//                       16 KB of bf16 act hi rows + 16 KB of their lo halves
//                       + 16 KB of bf16 Wd rows (48 KB, 4 stages), two bf16
//                       MMAs per K step, hi then lo (kDownSplit).
//
// Roles (both CTAs run the same code):
//   warp 0    producer: its CTA's A rows and weight rows, TMA copies whose
//             bytes complete on the even CTA's stage barrier; the even CTA
//             posts the byte count of both halves.
//   warp 1    TMEM allocation (both CTAs, collectively) and, in the even CTA,
//             the MMA issuer; its commits arrive on the stage and
//             accumulator barriers of both CTAs.
//   warps 2-5 epilogue of the CTA's own 128 rows; each warp then arrives on
//             the even CTA's accumulator-empty barrier (8 arrivals a round).
// Hand-off (GemmArgs::act_ready): every gate/up epilogue warp of both CTAs
// publishes its rows of a tile on the block pair's counter, and the down
// GEMM, launched without waiting for the gate/up grid, loads a pair's
// activation rows once all of the pair's arrivals are in.
// Every wait is bounded; a CTA that gives up records MOE_ERR_DEVICE_TIMEOUT.
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kPairThreads = 192;
constexpr int kMaxGroups = MOE_MAX_EXPERTS;

template <int MODE>
struct PairCfg;

// Per CTA and K slice: one 128-row activation tile and B_ROWS weight rows;
// the pair's MMA has N = MMA_N.
template <>
struct PairCfg<kGateUp> {
    static constexpr int BN = 128;     // gate columns per tile (and as many up columns)
    static constexpr int B_ROWS = BN;  // Wg rows (even CTA) or Wu rows (odd CTA)
    static constexpr int MMA_N = 2 * BN;
    static constexpr int A_TILES = 1;
    static constexpr int STAGE_BYTES = kATileBytes + B_ROWS * 128;
    static constexpr int STAGES = 6;
};

template <>
struct PairCfg<kDown> {
    static constexpr int BN = 256;
    static constexpr int B_ROWS = BN / 2;  // this CTA's half of the Wd rows
    static constexpr int MMA_N = BN;
    static constexpr int A_TILES = 1;
    static constexpr int STAGE_BYTES = kATileBytes + B_ROWS * 128;
    static constexpr int STAGES = 6;
};

template <>
struct PairCfg<kDownSplit> {
    static constexpr int BN = 256;
    static constexpr int B_ROWS = BN / 2;
    static constexpr int MMA_N = BN;
    static constexpr int A_TILES = 2;  // act hi rows, then their lo halves
    static constexpr int STAGE_BYTES = 2 * kATileBytes + B_ROWS * 128;
    static constexpr int STAGES = 4;
};

constexpr int kMaxPairStages = 6;

struct PairSmem {
    uint64_t full[kMaxPairStages];   // even CTA: both halves of a stage landed
    uint64_t empty[kMaxPairStages];  // both: the pair's MMAs are done with a stage
    uint64_t acc_full[2];            // both: an accumulator is complete
    uint64_t acc_empty[2];           // even CTA: both epilogues drained an accumulator
    uint64_t drain;                  // even CTA: every MMA it issued has completed
    int pair_prefix[kMaxGroups + 1]; // pairs of the groups before group g
    int block0[kMaxGroups + 1];      // first row block of group g (block0[G] = end)
    int num_groups;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory address of the same variable in cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}

// Arrival on a barrier of a cluster CTA (a shared::cluster address), ordering
// no memory accesses: the accumulator-empty barrier only says that this
// warp's TMEM reads are complete (tcgen05.wait::ld has returned), and a
// release would first drain the epilogue's global stores.
__device__ __forceinline__ void arrive_cluster_relaxed(uint32_t bar_cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                     bar_cluster_addr)
                 : "memory");
}

// 2-D tiled TMA load into this CTA's shared memory whose bytes complete on a
// barrier of the even CTA of the pair (a shared::cluster address).
__device__ __forceinline__ void tma_load_pair(void *dst, const CUtensorMap *map,
                                              uint32_t bar_cluster_addr, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile"
        ".mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
        "l"(map), "r"(bar_cluster_addr), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on the barrier at `bar`'s offset in every CTA of `cta_mask`
// when the MMAs issued so far by this thread have completed.
__device__ __forceinline__ void commit_pair(uint64_t *bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_addr(bar)),
        "h"(cta_mask)
        : "memory");
}

struct PairTile {
    int group;   // expert (0 for a single dense group)
    int block;   // this CTA's row block
    bool rows;   // this CTA's block exists (else its rows are padding)
    bool peer_rows;
};

// Pair tile j of the grouped layout, seen from cluster rank r.
__device__ __forceinline__ PairTile pair_of(const PairSmem *sm, int j, uint32_t r) {
    int lo = 0, hi = sm->num_groups - 1;
    while (lo < hi) {  // last group whose first pair is <= j (skips empty groups)
        const int mid = (lo + hi + 1) / 2;
        if (sm->pair_prefix[mid] <= j) lo = mid;
        else hi = mid - 1;
    }
    const int i = j - sm->pair_prefix[lo];
    const int nb = sm->block0[lo + 1] - sm->block0[lo];
    PairTile t;
    t.group = lo;
    t.block = sm->block0[lo] + 2 * i + static_cast<int>(r);
    t.rows = 2 * i + static_cast<int>(r) < nb;
    t.peer_rows = 2 * i + static_cast<int>(1 - r) < nb;
    return t;
}

template <int MODE>
__global__ void __launch_bounds__(kPairThreads, 1)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                     const __grid_constant__ CUtensorMap tm_b0,
                     const __grid_constant__ CUtensorMap tm_b1,
                     const __grid_constant__ CUtensorMap tm_s0,
                     const __grid_constant__ CUtensorMap tm_s1,
                     const __grid_constant__ CUtensorMap tm_xv, const GemmArgs a) {
    using C = PairCfg<MODE>;
    constexpr int BN = C::BN;
    constexpr int kStages = C::STAGES;
    constexpr int kStageBytes = C::STAGE_BYTES;
    constexpr int kBOffset = C::A_TILES * kATileBytes;
    constexpr int kBBytes = C::B_ROWS * 128;
    constexpr bool kSplit = MODE == kDownSplit;
    constexpr uint32_t kColsPerAcc = C::MMA_N;  // 256 either way
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    PairSmem *sm = reinterpret_cast<PairSmem *>(tiles + kStages * kStageBytes);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm->full[s], 1);
            mbar_init(&sm->empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm->acc_full[i], 1);
            mbar_init(&sm->acc_empty[i], 8);  // 4 epilogue warps x 2 CTAs
        }
        mbar_init(&sm->drain, 1);
        sm->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tensor_map(&tm_a);
        prefetch_tensor_map(&tm_b0);
        if (MODE == kGateUp) prefetch_tensor_map(&tm_b1);
    }
    if (warp == 1) {
        tmem_alloc_pair(&sm->tmem_base, 2 * kColsPerAcc);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // barriers of both CTAs initialised before any remote arrival
    tc_fence_after_sync();
    const uint32_t tmem = sm->tmem_base;
    volatile int *abort_flag = &sm->abort_flag;
    // hand-off (act_ready): down waits per block pair for its A rows, not for
    // the gate/up grid, and reads the block list from the kernels before
    // gate/up; so gate/up lets it launch only after its own dependency wait
    const bool handoff = a.act_ready != nullptr;
    if (!(MODE == kGateUp && handoff)) griddep_launch_dependents();
    // the block list and the A rows come from earlier kernels
    if (!(is_down(MODE) && handoff)) griddep_wait();
    if (MODE == kGateUp && handoff) griddep_launch_dependents();

    // pair prefix over the groups (experts): warp 2 scans, 8 groups per lane
    if (warp == 2) {
        const int G = a.pad_offsets ? a.num_groups : 1;
        int nb[kMaxGroups / 32];
        int b0[kMaxGroups / 32];
        int pairs = 0;
#pragma unroll
        for (int u = 0; u < kMaxGroups / 32; ++u) {
            const int g = lane * (kMaxGroups / 32) + u;
            int first = 0, end = 0;
            if (g < G) {
                if (a.pad_offsets) {
                    first = __ldcg(a.pad_offsets + g) / kBlockM;
                    end = __ldcg(a.pad_offsets + g + 1) / kBlockM;
                } else {
                    end = static_cast<int>((a.num_rows_host + kBlockM - 1) / kBlockM);
                }
            }
            b0[u] = first;
            nb[u] = end - first;
            pairs += (nb[u] + 1) / 2;
        }
        int incl = pairs;  // inclusive scan over lanes
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        int run = incl - pairs;
#pragma unroll
        for (int u = 0; u < kMaxGroups / 32; ++u) {
            const int g = lane * (kMaxGroups / 32) + u;
            if (g < G) {
                sm->pair_prefix[g] = run;
                sm->block0[g] = b0[u];
                if (g == G - 1) {
                    sm->pair_prefix[G] = run + (nb[u] + 1) / 2;
                    sm->block0[G] = b0[u] + nb[u];
                }
            }
            run += (nb[u] + 1) / 2;
        }
        if (lane == 0) sm->num_groups = G;
    }
    __syncthreads();

    const int n_tiles = (a.n_out + BN - 1) / BN;
    const int total_tiles = min(sm->pair_prefix[sm->num_groups] * n_tiles, a.max_tiles);
    const int nk = (a.K + kBlockK - 1) / kBlockK;
    const int pair_id = blockIdx.x / 2;
    const int num_pairs = gridDim.x / 2;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (lane 0)
        if (lane == 0) {
            int g = 0;
            bool failed = false;
            for (int tile = pair_id; tile < total_tiles && !failed; tile += num_pairs) {
                const PairTile pt = pair_of(sm, tile / n_tiles, rank);
                if (is_down(MODE) && handoff && pt.rows) {
                    // this block pair's activation rows are complete once
                    // every gate/up epilogue warp of both CTAs has stored
                    // its rows of every gate/up tile of the pair (bounded)
                    if (!wait_count_ns(a.act_ready + tile / n_tiles, a.act_ready_count,
                                       abort_flag, kWaitTimeoutNs)) {
                        record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                        *abort_flag = 1;
                        failed = true;
                        break;
                    }
                    fence_proxy_async_global();  // the TMA reads below see those rows
                }
                const int nt = tile % n_tiles;
                const uint32_t a_bytes = C::A_TILES * kATileBytes;
                const uint32_t tx = 2 * kBBytes +
                                    a_bytes * ((pt.rows ? 1u : 0u) + (pt.peer_rows ? 1u : 0u));
                const int arow = pt.block * kBlockM;
                // gate/up: Wg rows (even CTA) or Wu rows (odd CTA) of N tile nt;
                // down: this CTA's half of the Wd rows of N tile nt
                const WeightCoord wc = weight_coord<MODE>(
                    a, pt.group, nt * BN, is_down(MODE) ? static_cast<int>(rank) * C::B_ROWS : 0);
                const CUtensorMap *tm_b = (MODE == kGateUp && rank == 1)
                                              ? (wc.shared ? &tm_s1 : &tm_b1)
                                              : (wc.shared ? &tm_s0 : &tm_b0);
                // a shared-expert chunk's block j holds tokens 128 j .. (x
                // itself, rows past N read as zero)
                const bool a_from_x = MODE == kGateUp && a.a_from_x && wc.shared;
                const CUtensorMap *tm_arows = a_from_x ? &tm_xv : &tm_a;
                const int arow_src = a_from_x ? (pt.block - sm->block0[pt.group]) * kBlockM : arow;
                for (int kc = 0; kc < nk; ++kc, ++g) {
                    const int s = g % kStages;
                    const uint32_t use = g / kStages;
                    if (use > 0 && !mbar_wait(&sm->empty[s], (use - 1) & 1, abort_flag)) {
                        record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                        *abort_flag = 1;
                        failed = true;
                        break;
                    }
                    uint8_t *st = tiles + s * kStageBytes;
                    const uint32_t bar = cluster_addr(&sm->full[s], 0);
                    if (leader) mbar_arrive_expect_tx(&sm->full[s], tx);
                    if (pt.rows) {
                        tma_load_pair(st, tm_arows, bar, kc * kBlockK, arow_src);
                        if (kSplit)
                            tma_load_pair(st + kATileBytes, &tm_a, bar, kc * kBlockK,
                                          arow + static_cast<int>(a.lo_rows));
                    }
                    tma_load_pair(st + kBOffset, tm_b, bar, wc.k0 + kc * kBlockK, wc.row);
                }
            }
            // the even CTA's stage barriers count both CTAs' bytes: it waits
            // until the last copy into every stage has landed
            if (leader)
                for (int i = (g > kStages ? g - kStages : 0); i < g; ++i)
                    mbar_wait(&sm->full[i % kStages], (i / kStages) & 1, abort_flag);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA)
        if (leader && lane == 0) {
            // gate/up: bf16 x bf16; kDown: fp16 act x fp16 Wd; kDownSplit:
            // bf16 act hi x bf16 Wd, then act lo x the same Wd, per K step
            constexpr uint32_t idesc = MODE == kDown ? idesc_f16_f32(2 * kBlockM, C::MMA_N)
                                                     : idesc_bf16_f32(2 * kBlockM, C::MMA_N);
            int g = 0, it = 0;
            bool failed = false;
            for (int tile = pair_id; tile < total_tiles && !failed; tile += num_pairs, ++it) {
                const int acc = it & 1;
                const uint32_t use = it >> 1;
                if (use > 0 && !mbar_wait(&sm->acc_empty[acc], (use - 1) & 1, abort_flag)) {
                    failed = true;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d = tmem + acc * kColsPerAcc;
                for (int kc = 0; kc < nk; ++kc, ++g) {
                    const int s = g % kStages;
                    if (!mbar_wait(&sm->full[s], (g / kStages) & 1, abort_flag)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint8_t *st = tiles + s * kStageBytes;
                    const uint64_t da = sw128_kmajor_desc(smem_addr(st));
                    const uint64_t da_lo = sw128_kmajor_desc(smem_addr(st + kATileBytes));
                    const uint64_t db = sw128_kmajor_desc(smem_addr(st + kBOffset));
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk) {
                        const uint32_t accumulate = (kc | kk) != 0;
                        mma_pair(d, da + 2 * kk, db + 2 * kk, idesc, accumulate);
                        if (kSplit) mma_pair(d, da_lo + 2 * kk, db + 2 * kk, idesc, 1);
                    }
                    commit_pair(&sm->empty[s], 3);
                }
                if (!failed) commit_pair(&sm->acc_full[acc], 3);
            }
            if (failed) {
                record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            }
            commit_pair(&sm->drain, 1);
            mbar_wait(&sm->drain, 0, abort_flag);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (4 warps)
        const int quarter = warp % 4;
        const int row = quarter * 32 + lane;
        const uint32_t acc_empty0 = cluster_addr(&sm->acc_empty[0], 0);
        const uint32_t acc_empty1 = cluster_addr(&sm->acc_empty[1], 0);
        int it = 0;
        // row info runs ahead: the pair of a row two tiles ahead and its
        // routing weight one tile ahead, so no L2 round trip delays a tile.
        // grow -1: this CTA's block of the tile holds no rows.
        const int step = num_pairs;
        auto grow_of = [&](int t) -> int64_t {
            if (t >= total_tiles) return -1;
            const PairTile pt = pair_of(sm, t / n_tiles, rank);
            return pt.rows ? static_cast<int64_t>(pt.block) * kBlockM + row : -1;
        };
        int64_t g_cur = grow_of(pair_id);
        TileRow cur = g_cur >= 0 ? tile_row_of<MODE>(a, g_cur, row_pair(a, g_cur)) : no_tile_row();
        int64_t g_next = grow_of(pair_id + step);
        int64_t q_next = g_next >= 0 ? row_pair(a, g_next) : -1;
        for (int tile = pair_id; tile < total_tiles; tile += step, ++it) {
            const int acc = it & 1;
            bool ok = true;
            if (lane == 0) ok = mbar_wait(&sm->acc_full[acc], (it >> 1) & 1, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            tc_fence_after_sync();
            const TileRow nxt = g_next >= 0 ? tile_row_of<MODE>(a, g_next, q_next) : no_tile_row();
            const int64_t g_after = grow_of(tile + 2 * step);
            q_next = g_after >= 0 ? row_pair(a, g_after) : -1;
            if (g_cur >= 0) {  // CTA-uniform: the TMEM loads stay warp-wide
                const uint32_t taddr =
                    tmem + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kColsPerAcc;
                store_tile<MODE, BN>(a, taddr, cur, tile % n_tiles);
            }
            if (MODE == kGateUp && handoff) {
                // publish this warp's rows of the tile (a CTA without rows
                // publishes too: the count is per warp of both CTAs)
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) red_release_gpu(a.act_ready + tile / n_tiles, 1);
            }
            cur = nxt;
            g_cur = g_next;
            g_next = g_after;
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) arrive_cluster_relaxed(acc ? acc_empty1 : acc_empty0);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // both CTAs are done with TMEM and with each other's barriers
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem, 2 * kColsPerAcc);
    }
}

template <int MODE>
cudaError_t launch_pair_one(const CUtensorMap &tm_a, const CUtensorMap &tm_b0,
                            const CUtensorMap &tm_b1, const CUtensorMap &tm_s0,
                            const CUtensorMap &tm_s1, const CUtensorMap &tm_xv, const GemmArgs &a,
                            cudaStream_t s) {
    using C = PairCfg<MODE>;
    const size_t smem = 1024 + static_cast<size_t>(C::STAGES) * C::STAGE_BYTES + sizeof(PairSmem);
    auto kern = pair_gemm_kernel<MODE>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(a.grid), dim3(kPairThreads), smem, s, 2, tm_a, tm_b0, tm_b1,
                      tm_s0, tm_s1, tm_xv, a);
}

}  // namespace

int pair_gemm_block_n(GemmMode mode) { return mode == kGateUp ? PairCfg<kGateUp>::BN
                                                              : PairCfg<kDown>::BN; }
static_assert(PairCfg<kDown>::BN == PairCfg<kDownSplit>::BN, "one down tile width");

cudaError_t launch_pair_gemm(GemmMode mode, const CUtensorMap &tm_a, const CUtensorMap &tm_b0,
                             const CUtensorMap &tm_b1, const GemmArgs &a, cudaStream_t s,
                             const CUtensorMap *tm_s0, const CUtensorMap *tm_s1,
                             const CUtensorMap *tm_xv) {
    if (a.grid < 2 || a.grid % 2) return cudaErrorInvalidValue;
    if (a.pad_offsets && (a.num_groups < 1 || a.num_groups > kMaxGroups))
        return cudaErrorInvalidValue;
    const CUtensorMap &s0 = tm_s0 ? *tm_s0 : tm_b0;
    const CUtensorMap &s1 = tm_s1 ? *tm_s1 : tm_b1;
    if (a.a_from_x && (!tm_xv || mode != kGateUp)) return cudaErrorInvalidValue;
    const CUtensorMap &xv = tm_xv ? *tm_xv : tm_a;
    if (mode == kGateUp) return launch_pair_one<kGateUp>(tm_a, tm_b0, tm_b1, s0, s1, xv, a, s);
    if (mode == kDownSplit)
        return launch_pair_one<kDownSplit>(tm_a, tm_b0, tm_b1, s0, s1, xv, a, s);
    return launch_pair_one<kDown>(tm_a, tm_b0, tm_b1, s0, s1, xv, a, s);
}

}  // namespace moe
