// grouped_gemm.cu -- K3 and K4: the per-expert SwiGLU of the M03 "Sparse
// MoE" drill, Expert(h) = (silu(h Wg^T) * (h Wu^T)) Wd^T, run "the serving
// way" (each expert once over the tokens routed to it) as grouped GEMMs over
// the row blocks that moe_align produced (one group per expert; FusedMoE's
// grouped GEMM as named in the drill's shape-trace section).
//
//   K3 (kGateUp): for the 128 rows of block b (expert e = block_expert[b]),
//       A = x[token(q)] gathered row by row, B0 = Wg[e], B1 = Wu[e];
//       a = silu(A B0^T) * (A B1^T) in fp32 (96- or 128-column tiles),
//       stored as act = fp16(a)
//   K4: A = act rows of block b, B0 = Wd[e];
//       y[q, :] = w[q] * act B0^T in fp32 (256-column tiles), where w[q] is
//       the routing weight of pair q (or the shared gate).  The activation
//       needs more significant bits than bf16's 8 (a bf16 activation costs
//       more relative error per pair than the layer's output tolerance
//       leaves over the final bf16 rounding), so K4 takes it one of two ways:
//         kDownSplit: act as a bf16 pair hi + lo (16 bits) against the
//                     model's bf16 Wd, two MMAs per K step (hi, then lo);
//         kDown:      act in fp16 (11 bits) against an fp16 copy of Wd made
//                     once at load (exact for bf16 weights from 2^-14 up),
//                     one MMA per K step.
//       The per-pair results stay in fp32 until the combine.  A value the
//       stored format cannot hold records MOE_ERR_DEVICE_CHECK.
// Padding rows (q >= q_limit) are computed by the MMA but never loaded from
// memory nor stored.
//
// A rows come in one of two ways, chosen per block:
//   dense  (more than kSparseRows real rows): one tiled 128-row TMA box per A
//          operand per K slice, from rows that are contiguous in memory (x
//          rows copied into expert order by gather_rows_kernel, act rows, or x
//          itself for the shared expert);
//   sparse (at most kSparseRows real rows, e.g. decode): each lane fetches 4
//          rows with one tile::gather4 copy, skipped when all 4 are padding,
//          so padding rows are never read.  A gather4 copy costs the TMA unit
//          far more than a box (32 of them per K slice ran the gate/up GEMM
//          2.6x slower at prefill), hence only for blocks that are mostly
//          padding.
//
// Persistent kernel, one CTA per SM, 6 warps:
//   warp 0    TMA producer: A rows (box or gather4), then lane 0 fetches the
//             weight tile(s) with tiled copies.
//   warp 1    TMEM allocator and MMA issuer (one thread): 4 x K=16 tcgen05
//             MMAs per 64-wide K slice into one of two TMEM accumulators.
//   warps 2-5 epilogue: tcgen05.ld of the 128 x 256 fp32 accumulator (one
//             row per thread), activation or weight scale, 16-byte stores.
// The two accumulators let the epilogue of tile t overlap the mainloop of
// tile t+1.  Every wait is bounded (see ptx.cuh).
#include <cuda_bf16.h>

#include "kernels.cuh"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kMaxStages = 6;
constexpr int kThreads = 192;

struct GemmSmem {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// Tile shape: BN output columns per tile (gate/up: BN gate + BN up
// columns), A_TILES activation tiles (the gathered x, or act; the hi and lo
// halves of a split activation) and B_TILES weight tiles per K slice; as
// many stages as fit in ~200 KB.
template <int MODE, int BN_>
struct Cfg {
    static constexpr int BN = BN_;
    static constexpr int A_TILES = MODE == kDownSplit ? 2 : 1;
    static constexpr int B_TILES = MODE == kGateUp ? 2 : 1;
    static constexpr int B_BYTES = B_TILES * BN * 128;
    static constexpr int STAGE_BYTES = A_TILES * kATileBytes + B_BYTES;
    static constexpr int STAGES = (200 * 1024 / STAGE_BYTES) < kMaxStages
                                      ? (200 * 1024 / STAGE_BYTES) : kMaxStages;
    static_assert(B_TILES * BN <= kAccCols, "accumulator wider than its TMEM slot");
};

template <int MODE, int BN_>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                        const __grid_constant__ CUtensorMap tm_a_box,
                        const __grid_constant__ CUtensorMap tm_b0,
                        const __grid_constant__ CUtensorMap tm_b1,
                        const __grid_constant__ CUtensorMap tm_s0,
                        const __grid_constant__ CUtensorMap tm_s1, const GemmArgs a) {
    using C = Cfg<MODE, BN_>;
    constexpr int BN = C::BN;
    constexpr int kStages = C::STAGES;
    constexpr int kStageBytes = C::STAGE_BYTES;
    constexpr int kBOffset = C::A_TILES * kATileBytes;
    constexpr bool kSplit = MODE == kDownSplit;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    GemmSmem *sm = reinterpret_cast<GemmSmem *>(tiles + kStages * kStageBytes);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm->full[s], 1);
            mbar_init(&sm->empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm->acc_full[i], 1);
            mbar_init(&sm->acc_empty[i], 4);  // one arrival per epilogue warp
        }
        mbar_init(&sm->drain, 1);
        sm->abort_flag = 0;
        fence_barrier_init();
        prefetch_tensor_map(&tm_a);
        prefetch_tensor_map(&tm_b0);
        if (MODE == kGateUp) prefetch_tensor_map(&tm_b1);
        prefetch_tensor_map(&tm_a_box);
    }
    if (warp == 1) {
        tmem_alloc(&sm->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm->tmem_base;
    volatile int *abort_flag = &sm->abort_flag;
    griddep_launch_dependents();
    griddep_wait();  // the block list and A rows come from earlier kernels

    const int64_t rows = a.num_padded ? static_cast<int64_t>(__ldcg(a.num_padded)) : a.num_rows_host;
    const int num_blocks = static_cast<int>((rows + kBlockM - 1) / kBlockM);
    const int n_tiles = (a.n_out + BN - 1) / BN;
    const int total_tiles = min(num_blocks * n_tiles, a.max_tiles);
    const int nk = (a.K + kBlockK - 1) / kBlockK;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (warp)
        // weight tiles used by one row block each (decode) are streamed with
        // evict-first so that they do not push the reused data out of L2
        const uint64_t wpol = a.stream_weights ? l2_policy_evict_first() : 0;
        int g = 0;  // K slices issued by this CTA so far
        bool failed = false;
        for (int tile = blockIdx.x; tile < total_tiles && !failed; tile += gridDim.x) {
            const int blk = tile / n_tiles;
            const int nt = tile % n_tiles;
            const int expert = a.block_expert ? __ldcg(a.block_expert + blk) : 0;
            // dense: the block has more than kSparseRows real rows (real rows
            // come first in a block, so looking at row kSparseRows suffices)
            bool dense = true;
            if (a.sorted_pair) {
                const int64_t probe =
                    __ldcg(a.sorted_pair + static_cast<int64_t>(blk) * kBlockM + kSparseRows);
                dense = probe >= 0 && probe < a.q_limit;
            }
            // sparse: rows 4*lane .. 4*lane+3 of this block
            int src[4];
            bool any = false;
            int first_valid = -1;
            if (!dense) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int64_t row = static_cast<int64_t>(blk) * kBlockM + lane * 4 + i;
                    const int64_t q = __ldcg(a.sorted_pair + row);
                    const bool v = q >= 0 && q < a.q_limit;
                    src[i] = !v ? -1 : (MODE == kGateUp ? static_cast<int>(q / a.k_div)
                                                        : static_cast<int>(row));
                    if (v && first_valid < 0) first_valid = src[i];
                    any |= v;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (src[i] < 0) src[i] = first_valid;  // a real row; its result is dropped
            }
            const uint32_t groups = dense ? 0u : __popc(__ballot_sync(0xffffffffu, any));
            const uint32_t a_bytes = C::A_TILES * (dense ? kATileBytes : groups * 512);
            const int lo = static_cast<int>(a.lo_rows);  // split: rows of the lo half
            const uint32_t tx = a_bytes + C::B_BYTES;
            const int arow = blk * kBlockM;
            const WeightCoord wc = weight_coord<MODE>(a, expert, nt * BN, 0);
            const CUtensorMap *mb0 = wc.shared ? &tm_s0 : &tm_b0;
            const CUtensorMap *mb1 = wc.shared ? &tm_s1 : &tm_b1;
            for (int kc = 0; kc < nk; ++kc, ++g) {
                const int s = g % kStages;
                const uint32_t use = g / kStages;
                bool ok = true;
                if (lane == 0 && use > 0) ok = mbar_wait(&sm->empty[s], (use - 1) & 1, abort_flag);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0) {
                        record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                        *abort_flag = 1;
                    }
                    failed = true;
                    break;
                }
                uint8_t *st = tiles + s * kStageBytes;
                if (lane == 0) mbar_arrive_expect_tx(&sm->full[s], tx);
                __syncwarp();
                if (dense) {
                    if (lane == 0) {
                        tma_load_2d(st, &tm_a_box, &sm->full[s], kc * kBlockK, arow);
                        if (kSplit)
                            tma_load_2d(st + kATileBytes, &tm_a_box, &sm->full[s], kc * kBlockK,
                                        arow + lo);
                    }
                } else if (any) {
                    tma_gather4(st + lane * 512, &tm_a, &sm->full[s], kc * kBlockK, src[0],
                                src[1], src[2], src[3]);
                    if (kSplit)
                        tma_gather4(st + kATileBytes + lane * 512, &tm_a, &sm->full[s],
                                    kc * kBlockK, src[0] + lo, src[1] + lo, src[2] + lo,
                                    src[3] + lo);
                }
                if (lane == 0) {
                    const int kx = wc.k0 + kc * kBlockK;
                    if (a.stream_weights) {
                        tma_load_2d_hint(st + kBOffset, mb0, &sm->full[s], kx, wc.row, wpol);
                        if (MODE == kGateUp)
                            tma_load_2d_hint(st + kBOffset + BN * 128, mb1, &sm->full[s], kx,
                                             wc.row, wpol);
                    } else {
                        tma_load_2d(st + kBOffset, mb0, &sm->full[s], kx, wc.row);
                        if (MODE == kGateUp)
                            tma_load_2d(st + kBOffset + BN * 128, mb1, &sm->full[s], kx, wc.row);
                    }
                }
            }
        }
        // drain: wait until the last copy issued into every stage has landed
        if (lane == 0)
            for (int i = (g > kStages ? g - kStages : 0); i < g; ++i)
                mbar_wait(&sm->full[i % kStages], (i / kStages) & 1, abort_flag);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (1 thread)
        if (lane == 0) {
            // gate/up: the Wg and Wu tiles sit back to back in shared memory,
            // so one MMA of N = 2 BN produces [gate | up] in the accumulator;
            // bf16 x bf16.  kDown: fp16 act x fp16 Wd.  kDownSplit: bf16 act
            // hi x bf16 Wd, then act lo x the same Wd, per K step.
            constexpr uint32_t idesc = MODE == kGateUp ? idesc_bf16_f32(kBlockM, 2 * BN)
                                       : MODE == kDown ? idesc_f16_f32(kBlockM, BN)
                                                       : idesc_bf16_f32(kBlockM, BN);
            int g = 0, it = 0;
            bool failed = false;
            for (int tile = blockIdx.x; tile < total_tiles && !failed; tile += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t use = it >> 1;
                if (use > 0 && !mbar_wait(&sm->acc_empty[acc], (use - 1) & 1, abort_flag)) {
                    failed = true;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d = tmem + acc * kAccCols;
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
                        mma_f16kind(d, da + 2 * kk, db + 2 * kk, idesc, accumulate);
                        if (kSplit) mma_f16kind(d, da_lo + 2 * kk, db + 2 * kk, idesc, 1);
                    }
                    mma_commit(&sm->empty[s]);
                }
                if (!failed) mma_commit(&sm->acc_full[acc]);
            }
            if (failed) {
                record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            }
            mma_commit(&sm->drain);
            mbar_wait(&sm->drain, 0, abort_flag);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (4 warps)
        const int quarter = warp % 4;               // TMEM lanes this warp may read
        const int row = quarter * 32 + lane;        // tile row = TMEM lane
        int it = 0;
        // row info runs ahead: the pair of a row two tiles ahead and its
        // routing weight one tile ahead, so no L2 round trip delays a tile
        const int step = gridDim.x;
        auto grow_of = [&](int t) { return static_cast<int64_t>(t / n_tiles) * kBlockM + row; };
        const int first = blockIdx.x;
        TileRow cur = first < total_tiles ? tile_row<MODE>(a, first / n_tiles, row) : no_tile_row();
        int64_t q_next = first + step < total_tiles ? row_pair(a, grow_of(first + step)) : -1;
        for (int tile = first; tile < total_tiles; tile += step, ++it) {
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
            const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kAccCols;
            const TileRow nxt = tile + step < total_tiles
                                    ? tile_row_of<MODE>(a, grow_of(tile + step), q_next)
                                    : no_tile_row();
            q_next = tile + 2 * step < total_tiles ? row_pair(a, grow_of(tile + 2 * step)) : -1;
            store_tile<MODE, BN>(a, taddr, cur, tile % n_tiles);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm->acc_empty[acc]);
            cur = nxt;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// x_sorted[s, :] = x[sorted_pair[s] / k, :] for the real rows s of dense
// blocks, or of every block when all_blocks is set (the CTA-pair kernel loads
// every block with tiled boxes).  One CTA per row block (grid-stride): a
// broadcast load of the block's row kSparseRows decides whether it is dense,
// so sparse blocks (all of them at decode) cost one load.  Warp w copies rows
// w, w + 8, ..., w + 120: their 16 row-map entries come with one load, then
// two rows at a time are copied with all their 16-byte loads (8 per lane and
// row) in flight before the stores, until the first padding row (real rows
// come first).  The stores
// are streaming (evict-first): the GEMM reads each x_sorted row once, while
// each x row is read k times here and should stay in L2.
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads)
    gather_rows_kernel(const uint16_t *__restrict__ x, int H, int k,
                       const int32_t *__restrict__ sorted_pair,
                       const int32_t *__restrict__ num_padded, int64_t P, int64_t cap,
                       uint16_t *__restrict__ x_sorted, int all_blocks, int skip_slot) {
    griddep_launch_dependents();
    griddep_wait();
    constexpr int kWarps = kGatherThreads / 32;
    constexpr int kRowsPerWarp = kBlockM / kWarps;  // 16
    constexpr int kUnroll = 8;                      // 16-byte pieces per lane per row in flight
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int64_t nblocks = min(static_cast<int64_t>(__ldcg(num_padded)), cap) / kBlockM;
    const int n16 = H / 8;  // 16-byte pieces per row
    for (int64_t b = blockIdx.x; b < nblocks; b += gridDim.x) {
        const int64_t base = b * kBlockM;
        if (!all_blocks) {
            const int32_t probe = __ldcg(sorted_pair + base + kSparseRows);
            if (probe < 0 || probe >= P) continue;  // sparse block: its rows are gathered by TMA
        }
        if (skip_slot < k) {
            // a block of the shared expert's chunks (slots >= skip_slot): its
            // rows are x itself, in token order, loaded from x by the GEMM
            const int32_t first = __ldcg(sorted_pair + base);
            if (first >= 0 && first < P && first % k >= skip_slot) continue;
        }
        const int32_t q_lane =
            lane < kRowsPerWarp ? __ldcg(sorted_pair + base + warp + kWarps * lane) : -1;
        for (int i = 0; i < kRowsPerWarp; i += 2) {
            const int32_t q0 = __shfl_sync(0xffffffffu, q_lane, i);
            const int32_t q1 = __shfl_sync(0xffffffffu, q_lane, i + 1);
            const bool v0 = q0 >= 0 && q0 < P;
            const bool v1 = v0 && q1 >= 0 && q1 < P;  // padding only after the real rows
            if (!v0) break;
            const uint4 *s0 = reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(q0 / k) * H);
            const uint4 *s1 = reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(v1 ? q1 / k : 0) * H);
            uint4 *d0 = reinterpret_cast<uint4 *>(x_sorted + (base + warp + kWarps * i) * H);
            uint4 *d1 = reinterpret_cast<uint4 *>(x_sorted + (base + warp + kWarps * (i + 1)) * H);
            for (int c0 = lane; c0 < n16; c0 += 32 * kUnroll) {
                uint4 a0[kUnroll], a1[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int c = c0 + 32 * u;
                    if (c < n16) a0[u] = __ldcg(s0 + c);
                    if (v1 && c < n16) a1[u] = __ldcg(s1 + c);
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int c = c0 + 32 * u;
                    if (c < n16) __stcs(d0 + c, a0[u]);
                    if (v1 && c < n16) __stcs(d1 + c, a1[u]);
                }
            }
            if (!v1) break;
        }
    }
}

}  // namespace

cudaError_t launch_gather_rows(const uint16_t *x, int H, int k, const int32_t *sorted_pair,
                               const int32_t *num_padded, int64_t P, int64_t cap,
                               uint16_t *x_sorted, int all_blocks, int skip_slot, int num_sms,
                               cudaStream_t s) {
    int64_t blocks = cap / kBlockM;  // one CTA per row block, at most 4 per SM
    const int64_t limit = static_cast<int64_t>(num_sms) * 4;
    if (blocks > limit) blocks = limit;
    if (blocks < 1) blocks = 1;
    return launch_pdl(gather_rows_kernel, dim3(static_cast<unsigned>(blocks)),
                      dim3(kGatherThreads), 0, s, 1,
                      x, H, k, sorted_pair, num_padded, P, cap, x_sorted, all_blocks, skip_slot);
}

template <int MODE, int BN>
cudaError_t launch_one(const CUtensorMap &tm_a, const CUtensorMap &tm_a_box,
                       const CUtensorMap &tm_b0, const CUtensorMap &tm_b1,
                       const CUtensorMap &tm_s0, const CUtensorMap &tm_s1, const GemmArgs &a,
                       cudaStream_t s) {
    using C = Cfg<MODE, BN>;
    const size_t smem = 1024 + static_cast<size_t>(C::STAGES) * C::STAGE_BYTES + sizeof(GemmSmem);
    auto kern = grouped_gemm_kernel<MODE, BN>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(a.grid), dim3(kThreads), smem, s, 1, tm_a, tm_a_box, tm_b0,
                      tm_b1, tm_s0, tm_s1, a);
}

bool gemm_block_n_supported(GemmMode mode, int bn) {
    return mode == kGateUp ? (bn == 96 || bn == 128) : (bn == 256);
}

cudaError_t launch_gemm(GemmMode mode, int bn, const CUtensorMap &tm_a,
                        const CUtensorMap &tm_a_box, const CUtensorMap &tm_b0,
                        const CUtensorMap &tm_b1, const GemmArgs &a, cudaStream_t s,
                        const CUtensorMap *tm_s0, const CUtensorMap *tm_s1) {
    const CUtensorMap &s0 = tm_s0 ? *tm_s0 : tm_b0;
    const CUtensorMap &s1 = tm_s1 ? *tm_s1 : tm_b1;
    if (mode == kGateUp && bn == 96)
        return launch_one<kGateUp, 96>(tm_a, tm_a_box, tm_b0, tm_b1, s0, s1, a, s);
    if (mode == kGateUp && bn == 128)
        return launch_one<kGateUp, 128>(tm_a, tm_a_box, tm_b0, tm_b1, s0, s1, a, s);
    if (mode == kDown && bn == 256)
        return launch_one<kDown, 256>(tm_a, tm_a_box, tm_b0, tm_b1, s0, s1, a, s);
    if (mode == kDownSplit && bn == 256)
        return launch_one<kDownSplit, 256>(tm_a, tm_a_box, tm_b0, tm_b1, s0, s1, a, s);
    return cudaErrorInvalidValue;
}

}  // namespace moe
