// sparse_gemm.cu -- K3 (gate/up) and K4 (down) for batches whose row blocks
// hold only a few real rows each (decode: N·k pairs spread over many
// experts).  Same arithmetic per output element as the other grouped GEMMs
// (same K order, same epilogue: store_tile in gemm_common.cuh); only the
// staging differs.
//
// Such a GEMM streams every weight tile once and is bound by how many weight
// bytes each SM keeps in flight (HBM3e under load answers in ~4 us, so ~190 KB
// per SM is needed to approach the read bandwidth).  The activation rows of a block are loaded
// as 32-row sub-blocks into a 4 KB region (instead of a 16 KB 128-row
// tile), which leaves room for more weight stages:
//   gate/up BN = 96: 4 KB + 24 KB per stage, 8 stages (192 KB of weights);
//   gate/up BN = 128: 4 KB + 32 KB, 6 stages (192 KB);
//   down BN = 256: 4 KB of act + 32 KB of Wd, 6 stages (192 KB; 144 KB
//   with 128-row activation tiles).  The fp16 activation (kDown) fills the
//   4 KB with 32 rows; the bf16 hi/lo activation (kDownSplit) with 16 hi
//   rows followed by the same 16 rows' lo halves, so its passes hold 16 rows
//   and the weight bytes in flight stay the same.
// Gate/up: the MMA is still M = 128: its A operand spans 16 KB from the
// region's start, so the rows past a pass read whatever follows in the
// stage; they only feed accumulator rows that the epilogue never stores
// (and TMEM lanes 0-31 belong to the first epilogue warp alone).
// Down: the operands swap roles, so that the MMA's M side is the weights'
// and its N side the pass's rows: D^T = Wd * act^T as two M = 128 MMAs
// (weight rows 0-127 and 128-255 of the tile) of N = rows per pass (32, or
// 16 for kDownSplit, whose lo MMAs read the lo rows), K = 16 each: no
// padding row is read or multiplied (an M = 128 MMA over 16 real rows does
// 8x the tensor work).  The kernel's time is set by its weight stream either
// way.  Each product and each K step's sum reach an output element in the
// same order as in the other tilings.  The epilogue then holds one output
// column per thread (TMEM lane = weight row) for the pass's rows.
// A block with more real rows than a pass holds is computed as several
// passes over K (rare at decode); real rows come first in a block, so a
// block with n real rows takes ceil(n / rows per pass) passes.
//
// The producer publishes each tile's pass count through a small ring of
// shared-memory words (full/empty barriers per slot), so that the MMA issuer
// and the epilogue never wait on a global load.  The next tile's row map
// and expert are loaded while the current tile's stages are issued.
//
// Hand-off (GemmArgs::act_ready, decode with expert-indexed tiles): each
// gate/up tile publishes itself on its expert's counter once its rows are
// stored, and the down GEMM, launched without waiting for the gate/up grid,
// waits per tile for its expert's count before gathering the activation
// rows; down CTAs thus start on the SMs that gate/up frees first.
//
// Roles: warp 0 TMA producer (gather4 of the sub-block's real rows, lane 0
// the weight tile(s)); warp 1 TMEM allocation and MMA issuer; warps 2-5
// epilogue (gate/up: warp 4, which owns TMEM lanes 0-31, stores and the
// others only release the accumulator; down: each warp stores the output
// columns of its 32 TMEM lanes).  Every wait is bounded.
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kSubTileBytes = kSparseRows * 128;  // A region: 32 rows x 64 16-bit values
constexpr int kSparseMaxStages = 8;
constexpr int kSparseThreads = 192;
constexpr int kInfoSlots = 4;
constexpr int kInfoReaders = 1 + 4;  // MMA warp + four epilogue warps

template <int MODE, int BN_>
struct SparseCfg {
    static constexpr int BN = BN_;
    // rows per pass, and the A copies per row (hi and lo for kDownSplit)
    static constexpr int SUB_ROWS = MODE == kDownSplit ? kSparseRows / 2 : kSparseRows;
    static constexpr int A_COPIES = MODE == kDownSplit ? 2 : 1;
    static constexpr int LO_OFFSET = SUB_ROWS * 128;  // lo rows after the hi rows
    static constexpr int B_BYTES = (MODE == kGateUp ? 2 : 1) * BN * 128;
    static constexpr int STAGE_BYTES = kSubTileBytes + B_BYTES;
    static constexpr int STAGES = (224 * 1024 / STAGE_BYTES) < kSparseMaxStages
                                      ? (224 * 1024 / STAGE_BYTES) : kSparseMaxStages;
    // gate/up's MMA reads a 16 KB (128-row) A operand from the A region's
    // start (down's swapped MMAs read only the pass's rows)
    static_assert(STAGE_BYTES >= (A_COPIES - 1) * LO_OFFSET + kATileBytes,
                  "a 128-row A read would leave the stage");
    static_assert(STAGES * STAGE_BYTES + 1024 + 1024 <= 227 * 1024, "shared memory");
    static_assert((MODE == kGateUp ? 2 : 1) * BN <= kAccCols, "accumulator too wide");
};

constexpr int kMaxExperts = MOE_MAX_EXPERTS;

struct SparseSmem {
    int pad[kMaxExperts + 1];  // expert-indexed tiles: padded row offset of each expert
    uint64_t full[kSparseMaxStages];
    uint64_t empty[kSparseMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t info_full[kInfoSlots];
    uint64_t info_empty[kInfoSlots];
    uint64_t drain;
    int info[kInfoSlots];
    uint32_t tmem_base;
    int abort_flag;
};

// Consumer side of the tile-info ring: the pass count of local tile j
// (warp-wide; -1 when the wait gave up).
__device__ __forceinline__ int read_passes(SparseSmem *sm, int j, int lane,
                                           volatile int *abort_flag) {
    int n = -1;
    if (lane == 0) {
        const int slot = j % kInfoSlots;
        if (mbar_wait(&sm->info_full[slot], (j / kInfoSlots) & 1, abort_flag)) {
            n = *reinterpret_cast<volatile int *>(&sm->info[slot]);
            mbar_arrive(&sm->info_empty[slot]);
        }
    }
    return __shfl_sync(0xffffffffu, n, 0);
}

// Down epilogue of the swapped MMA, for the thread that owns TMEM lane
// (weight row) t of its warp's quarter: taddr = that quarter's lanes and the
// accumulator; h0 = t's output column in the tile's first 128 (the second
// half's is h0 + 128).  Columns [0, ROWS) of the lane hold the first half's
// values for the pass's rows 0 .. ROWS-1, [ROWS, 2 ROWS) the second half's.
// Lane i of the warp holds row i's TileRow (pair q, routing weight w); real
// rows come first.  Per value the arithmetic of store_tile's down branch: y
// = w * acc in fp32, stored as a pair row (bf16 hi at out, int8 residual at
// out_res, row q), so every tiling stores the same bits.
template <int ROWS>
__device__ __forceinline__ void store_tile_swapped(const GemmArgs &a, uint32_t taddr,
                                                   const TileRow &r, int h0, int lane) {
    static_assert(ROWS == 16 || ROWS == 32, "rows per pass");
    float v[2 * ROWS];
    tmem_load32(taddr, *reinterpret_cast<float(*)[32]>(v));
    if (ROWS == 32) tmem_load32(taddr + 32, *reinterpret_cast<float(*)[32]>(v + 32));
    tmem_load_wait();
    const int32_t q_lane = r.valid ? static_cast<int32_t>(r.q) : -1;
    uint16_t *hi_plane = static_cast<uint16_t *>(a.out);
    float vmax = 0.f;
#pragma unroll
    for (int j = 0; j < ROWS; ++j) {
        const int32_t q = __shfl_sync(0xffffffffu, q_lane, j);
        const float w = __shfl_sync(0xffffffffu, r.w, j);
        if (q < 0) break;  // warp-uniform: the rest of the pass is padding
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int h = h0 + half * kBlockM;
            const float y = w * v[half * ROWS + j];
            if (h < a.n_out) {
                vmax = max_abs_nan(vmax, y, y);
                const __nv_bfloat16 hb = __float2bfloat16_rn(y);
                const int64_t o = static_cast<int64_t>(q) * a.out_ld + h;
                hi_plane[o] = __bfloat16_as_ushort(hb);
                a.out_res[o] = static_cast<int8_t>(pair_residual(y, __bfloat162float(hb)));
            }
        }
    }
    if (!(vmax <= kF32Max)) record_status(a.status, MOE_ERR_DEVICE_CHECK);
}

template <int MODE, int BN_>
__global__ void __launch_bounds__(kSparseThreads, 1)
    sparse_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                       const __grid_constant__ CUtensorMap tm_b0,
                       const __grid_constant__ CUtensorMap tm_b1,
                       const __grid_constant__ CUtensorMap tm_s0,
                       const __grid_constant__ CUtensorMap tm_s1, const GemmArgs a) {
    using C = SparseCfg<MODE, BN_>;
    constexpr int BN = C::BN;
    constexpr int kStages = C::STAGES;
    constexpr int kStageBytes = C::STAGE_BYTES;
    constexpr int kBOffset = kSubTileBytes;
    constexpr int kSubRows = C::SUB_ROWS;
    constexpr int kLanesPerPass = kSubRows / 4;  // each lane gathers 4 rows
    constexpr bool kSplit = MODE == kDownSplit;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    SparseSmem *sm = reinterpret_cast<SparseSmem *>(tiles + kStages * kStageBytes);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm->full[s], 1);
            mbar_init(&sm->empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm->acc_full[i], 1);
            mbar_init(&sm->acc_empty[i], 4);
        }
        for (int i = 0; i < kInfoSlots; ++i) {
            mbar_init(&sm->info_full[i], 1);
            mbar_init(&sm->info_empty[i], kInfoReaders);
        }
        mbar_init(&sm->drain, 1);
        sm->abort_flag = 0;
        fence_barrier_init();
        prefetch_tensor_map(&tm_a);
        prefetch_tensor_map(&tm_b0);
        if (MODE == kGateUp) prefetch_tensor_map(&tm_b1);
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
    const int n_tiles = (a.n_out + BN - 1) / BN;
    const bool by_expert = a.expert_tiles != 0;
    // decode hand-off (act_ready): the down GEMM launched after this one does
    // not wait for this grid but for per-expert counts, and it reads the
    // block list from the kernels before this one; so gate/up lets it launch
    // only once every gate/up CTA has seen those kernels complete
    const bool handoff = a.act_ready != nullptr;
    if (!(MODE == kGateUp && handoff)) griddep_launch_dependents();
    // weights are inputs, not results of earlier kernels: with expert-indexed
    // tiles the first tile's weight rows are known now, and L2 fetches them
    // while memory is otherwise idle (routing)
    // (half of the tile's rows: the same gain as the whole tile in a timed
    // decode loop, with half the L2 footprint)
    if (by_expert && threadIdx.x == 0 && static_cast<int>(blockIdx.x) < a.num_groups * n_tiles &&
        static_cast<int>(blockIdx.x) / n_tiles < a.virt_base) {
        const int64_t e = blockIdx.x / n_tiles;
        const int64_t r0 = static_cast<int64_t>(blockIdx.x % n_tiles) * BN;
        const int64_t nrows = min(static_cast<int64_t>(BN), a.w_rows - r0) / 2;
        const int64_t off = (e * a.w_rows + r0) * a.K * 2;
        const uint32_t bytes = static_cast<uint32_t>(nrows * a.K * 2);
        if (bytes > 0) {
            prefetch_l2_bulk(static_cast<const uint8_t *>(a.w0) + off, bytes);
            if (MODE == kGateUp) prefetch_l2_bulk(static_cast<const uint8_t *>(a.w1) + off, bytes);
        }
    }
    // the block list and the A rows come from earlier kernels (with the
    // hand-off, down waits per expert for its A rows instead)
    if (!(is_down(MODE) && handoff)) griddep_wait();
    if (MODE == kGateUp && handoff) griddep_launch_dependents();

    int total_tiles;
    if (by_expert) {
        for (int i = threadIdx.x; i <= a.num_groups; i += blockDim.x)
            sm->pad[i] = __ldcg(a.pad_offsets + i);
        __syncthreads();
        total_tiles = min(a.num_groups * n_tiles, a.max_tiles);
    } else {
        const int64_t rows = static_cast<int64_t>(__ldcg(a.num_padded));
        total_tiles = min(static_cast<int>((rows + kBlockM - 1) / kBlockM) * n_tiles, a.max_tiles);
    }
    // row block of a tile (-1: its expert received no pairs)
    auto block_of = [&](int tile) -> int {
        if (!by_expert) return tile / n_tiles;
        const int e = tile / n_tiles;
        return sm->pad[e + 1] > sm->pad[e] ? sm->pad[e] / kBlockM : -1;
    };
    auto expert_of = [&](int tile) -> int {
        return by_expert ? tile / n_tiles : __ldcg(a.block_expert + tile / n_tiles);
    };
    const int nk = (a.K + kBlockK - 1) / kBlockK;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (warp)
        const uint64_t wpol = a.stream_weights ? l2_policy_evict_first() : 0;
        int g = 0;
        bool failed = false;
        // lane l holds rows 4l .. 4l+3 of a block; the next tile's are loaded
        // while this tile's stages are issued and compared only then
        int32_t q_next[4] = {-1, -1, -1, -1};
        int expert_next = 0;
        if (static_cast<int>(blockIdx.x) < total_tiles) {
            const int b0 = block_of(blockIdx.x);
            if (b0 >= 0) {
                const int64_t base = static_cast<int64_t>(b0) * kBlockM;
#pragma unroll
                for (int i = 0; i < 4; ++i) q_next[i] = __ldcg(a.sorted_pair + base + lane * 4 + i);
            }
            expert_next = expert_of(blockIdx.x);
        }
        for (int tile = blockIdx.x, j = 0; tile < total_tiles && !failed;
             tile += gridDim.x, ++j) {
            const int blk = block_of(tile);
            const int nt = tile % n_tiles;
            int src[4];
            bool any = false;
            int last = 0;  // 1 + highest real row of the block
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int32_t q = q_next[i];
                const bool v = q >= 0 && q < a.q_limit;
                src[i] = !v ? -1 : (MODE == kGateUp ? static_cast<int>(q / a.k_div)
                                                    : blk * kBlockM + lane * 4 + i);
                any |= v;
                if (v) last = lane * 4 + i + 1;
            }
            const int expert = expert_next;
            const int next = tile + static_cast<int>(gridDim.x);
            if (next < total_tiles) {
                const int bn = block_of(next);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    q_next[i] = bn >= 0 ? __ldcg(a.sorted_pair + static_cast<int64_t>(bn) * kBlockM +
                                                 lane * 4 + i)
                                        : -1;
                expert_next = expert_of(next);
            }
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, d));
            const int passes = (last + kSubRows - 1) / kSubRows;
            {
                bool ok = true;
                if (lane == 0) {
                    const int slot = j % kInfoSlots;
                    if (j >= kInfoSlots)
                        ok = mbar_wait(&sm->info_empty[slot], ((j / kInfoSlots) - 1) & 1, abort_flag);
                    if (ok) {
                        sm->info[slot] = passes;
                        mbar_arrive(&sm->info_full[slot]);
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    if (lane == 0) {
                        record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                        *abort_flag = 1;
                    }
                    failed = true;
                    break;
                }
            }
            // a lane's 4 rows sit in pass lane / kLanesPerPass; padding rows
            // copy a real row of the same group (their results are dropped)
            int first_valid = -1;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (src[i] >= 0 && first_valid < 0) first_valid = src[i];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (src[i] < 0) src[i] = first_valid;
            const WeightCoord wc = weight_coord<MODE>(a, expert, nt * BN, 0);
            const CUtensorMap *mb0 = wc.shared ? &tm_s0 : &tm_b0;
            const CUtensorMap *mb1 = wc.shared ? &tm_s1 : &tm_b1;
            if (is_down(MODE) && handoff && passes > 0) {
                // this expert's activation rows are complete once all its
                // gate/up tiles are stored (bounded wait by lane 0; the warp
                // barrier after it orders the other lanes' accesses, and each
                // lane's proxy fence its own TMA copies, after that acquire)
                bool ready = false;
                if (lane == 0)
                    ready = wait_count_ns(a.act_ready + expert, a.act_ready_count, abort_flag,
                                          kWaitTimeoutNs);
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (!ready) {
                    if (lane == 0) {
                        record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                        *abort_flag = 1;
                    }
                    failed = true;
                    break;
                }
                __syncwarp();
                fence_proxy_async_global();  // the TMA reads below see those rows
            }
            for (int p = 0; p < passes && !failed; ++p) {
                // lanes kLanesPerPass * p .. kLanesPerPass * (p + 1) - 1 gather pass p
                const bool mine = lane / kLanesPerPass == p && any;
                const uint32_t groups = __popc(__ballot_sync(0xffffffffu, mine));
                const uint32_t tx = groups * 512 * C::A_COPIES + C::B_BYTES;
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
                    if (mine) {
                        const int slot = lane % kLanesPerPass;
                        tma_gather4(st + slot * 512, &tm_a, &sm->full[s], kc * kBlockK, src[0],
                                    src[1], src[2], src[3]);
                        if (kSplit) {
                            const int lo = static_cast<int>(a.lo_rows);
                            tma_gather4(st + C::LO_OFFSET + slot * 512, &tm_a, &sm->full[s],
                                        kc * kBlockK, src[0] + lo, src[1] + lo, src[2] + lo,
                                        src[3] + lo);
                        }
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
                                tma_load_2d(st + kBOffset + BN * 128, mb1, &sm->full[s], kx,
                                            wc.row);
                        }
                    }
                }
            }
        }
        if (lane == 0)
            for (int i = (g > kStages ? g - kStages : 0); i < g; ++i)
                mbar_wait(&sm->full[i % kStages], (i / kStages) & 1, abort_flag);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (1 thread)
        // gate/up: Wg and Wu tiles are adjacent, one bf16 MMA of N = 2 BN;
        // kDown: fp16 act x fp16 Wd; kDownSplit: bf16 act hi x bf16 Wd, then
        // act lo x the same Wd, per K step
        // down (swapped): A = 128 weight rows, B = the pass's kSubRows rows
        constexpr uint32_t idesc = MODE == kGateUp ? idesc_bf16_f32(kBlockM, 2 * BN)
                                   : MODE == kDown ? idesc_f16_f32(kBlockM, kSubRows)
                                                   : idesc_bf16_f32(kBlockM, kSubRows);
        static_assert(!is_down(MODE) || BN == 2 * kBlockM, "down tiles: two 128-row halves");
        int g = 0, it = 0;
        bool failed = false;
        for (int tile = blockIdx.x, j = 0; tile < total_tiles && !failed; tile += gridDim.x, ++j) {
            const int passes = read_passes(sm, j, lane, abort_flag);
            if (passes < 0) {
                failed = true;
                break;
            }
            for (int p = 0; p < passes && !failed; ++p, ++it) {
                if (lane == 0) {
                    const int acc = it & 1;
                    const uint32_t use = it >> 1;
                    if (use > 0 && !mbar_wait(&sm->acc_empty[acc], (use - 1) & 1, abort_flag)) {
                        failed = true;
                    } else {
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
                            const uint64_t da_lo = sw128_kmajor_desc(smem_addr(st + C::LO_OFFSET));
                            const uint64_t db = sw128_kmajor_desc(smem_addr(st + kBOffset));
                            const uint64_t db1 =
                                sw128_kmajor_desc(smem_addr(st + kBOffset + kATileBytes));
#pragma unroll
                            for (int kk = 0; kk < kBlockK / 16; ++kk) {
                                const uint32_t acc_on = (kc | kk) != 0;
                                if (MODE == kGateUp) {
                                    mma_f16kind(d, da + 2 * kk, db + 2 * kk, idesc, acc_on);
                                } else {
                                    // columns [0, kSubRows): weight rows 0-127;
                                    // [kSubRows, 2 kSubRows): rows 128-255
                                    mma_f16kind(d, db + 2 * kk, da + 2 * kk, idesc, acc_on);
                                    mma_f16kind(d + kSubRows, db1 + 2 * kk, da + 2 * kk, idesc,
                                                acc_on);
                                    if (kSplit) {
                                        mma_f16kind(d, db + 2 * kk, da_lo + 2 * kk, idesc, 1);
                                        mma_f16kind(d + kSubRows, db1 + 2 * kk, da_lo + 2 * kk,
                                                    idesc, 1);
                                    }
                                }
                            }
                            mma_commit(&sm->empty[s]);
                        }
                        if (!failed) mma_commit(&sm->acc_full[acc]);
                    }
                }
                failed = __shfl_sync(0xffffffffu, failed, 0);
            }
        }
        if (lane == 0) {
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
        const int quarter = warp % 4;  // warp 4 owns TMEM lanes 0-31
        int it = 0;
        bool failed = false;
        for (int tile = blockIdx.x, j = 0; tile < total_tiles && !failed; tile += gridDim.x, ++j) {
            const int passes = read_passes(sm, j, lane, abort_flag);
            if (passes < 0) {
                if (lane == 0) {
                    record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            for (int p = 0; p < passes; ++p, ++it) {
                const int acc = it & 1;
                TileRow r = no_tile_row();
                // gate/up: lane i of warp 4 holds row i; down: lane i of every
                // epilogue warp holds row i (column i of the swapped result)
                if ((is_down(MODE) || quarter == 0) && lane < kSubRows)
                    r = tile_row<MODE>(a, block_of(tile), p * kSubRows + lane);
                bool ok = true;
                if (lane == 0) ok = mbar_wait(&sm->acc_full[acc], (it >> 1) & 1, abort_flag);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0) {
                        record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                        *abort_flag = 1;
                    }
                    failed = true;
                    break;
                }
                tc_fence_after_sync();
                if (MODE == kGateUp) {
                    if (quarter == 0) store_tile<MODE, BN>(a, tmem + acc * kAccCols, r, tile % n_tiles);
                } else {
                    store_tile_swapped<kSubRows>(
                        a, tmem + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kAccCols, r,
                        (tile % n_tiles) * BN + quarter * 32 + lane, lane);
                }
                if (MODE == kGateUp && handoff && quarter == 0 && p == passes - 1) {
                    // publish the tile: its rows' stores, then the count
                    fence_proxy_async_global();
                    __syncwarp();
                    if (lane == 0) red_release_gpu(a.act_ready + expert_of(tile), 1);
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm->acc_empty[acc]);
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int MODE, int BN>
cudaError_t launch_sparse_one(const CUtensorMap &tm_a, const CUtensorMap &tm_b0,
                              const CUtensorMap &tm_b1, const CUtensorMap &tm_s0,
                              const CUtensorMap &tm_s1, const GemmArgs &a, cudaStream_t s) {
    using C = SparseCfg<MODE, BN>;
    const size_t smem = 1024 + static_cast<size_t>(C::STAGES) * C::STAGE_BYTES + sizeof(SparseSmem);
    auto kern = sparse_gemm_kernel<MODE, BN>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(a.grid), dim3(kSparseThreads), smem, s, 1, tm_a, tm_b0, tm_b1,
                      tm_s0, tm_s1, a);
}

}  // namespace

cudaError_t launch_sparse_gemm(GemmMode mode, int bn, const CUtensorMap &tm_a,
                               const CUtensorMap &tm_b0, const CUtensorMap &tm_b1,
                               const GemmArgs &a, cudaStream_t s, const CUtensorMap *tm_s0,
                               const CUtensorMap *tm_s1) {
    if (!a.sorted_pair || !a.block_expert || !a.num_padded) return cudaErrorInvalidValue;
    const CUtensorMap &s0 = tm_s0 ? *tm_s0 : tm_b0;
    const CUtensorMap &s1 = tm_s1 ? *tm_s1 : tm_b1;
    if (mode == kGateUp && bn == 96)
        return launch_sparse_one<kGateUp, 96>(tm_a, tm_b0, tm_b1, s0, s1, a, s);
    if (mode == kGateUp && bn == 128)
        return launch_sparse_one<kGateUp, 128>(tm_a, tm_b0, tm_b1, s0, s1, a, s);
    if (mode == kDown && bn == 256)
        return launch_sparse_one<kDown, 256>(tm_a, tm_b0, tm_b1, s0, s1, a, s);
    if (mode == kDownSplit && bn == 256)
        return launch_sparse_one<kDownSplit, 256>(tm_a, tm_b0, tm_b1, s0, s1, a, s);
    return cudaErrorInvalidValue;
}

}  // namespace moe
