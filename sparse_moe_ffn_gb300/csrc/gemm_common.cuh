// gemm_common.cuh -- pieces shared by the grouped GEMM kernels (one-CTA,
// 32-row sparse and CTA-pair): tile constants, the SwiGLU helper and the
// epilogue that turns one TMEM accumulator row into stored outputs.
#pragma once

#include <cuda_bf16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kATileBytes = kBlockM * 128;  // 128 rows x 64 bf16
constexpr int kAccCols = 256;               // fp32 columns per accumulator
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr float kF16Max = 65504.f;
constexpr int kSparseRows = 32;             // blocks with at most this many real rows gather

__device__ __forceinline__ float silu_times(float g, float u) {
    return g / (1.f + __expf(-g)) * u;
}

// One row of a tile: grouped row `grow`, the pair (or token) q it holds,
// whether it is real, and the down projection's scale.  Loaded before the
// tile's accumulator is ready, so that the two dependent L2 reads overlap
// the MMAs instead of delaying the epilogue.
struct TileRow {
    int64_t grow;
    int64_t q;
    float w;
    bool valid;
};

template <int MODE>
__device__ __forceinline__ TileRow tile_row(const GemmArgs &a, int blk, int row) {
    TileRow r;
    r.grow = static_cast<int64_t>(blk) * kBlockM + row;
    r.q = a.sorted_pair ? __ldcg(a.sorted_pair + r.grow) : r.grow;
    r.valid = r.q >= 0 && r.q < a.q_limit;
    r.w = (MODE == kDown && r.valid) ? (a.scale ? __ldcg(a.scale + r.q) : 1.f) : 0.f;
    return r;
}

// Epilogue of one tile for the thread that owns TMEM lane r.grow % 128:
// output columns [nt * BN, nt * BN + BN) (gate/up: the accumulator holds BN
// gate columns, then BN up columns).  taddr = this warp's TMEM lane quarter
// and the tile's accumulator.
//   gate/up: act = fp16(silu(g) * u), the down projection's A operand;
//   down:    y[q] = fp16(w[q] * acc), the pair's weighted result.
// fp16 keeps 11 significant bits; a value past its range (65504) is
// reported as MOE_ERR_DEVICE_CHECK rather than silently turned into
// infinity.
template <int MODE, int BN>
__device__ __forceinline__ void store_tile(const GemmArgs &a, uint32_t taddr, const TileRow &r,
                                           int nt) {
    const int64_t grow = r.grow;
    const int64_t q = r.q;
    const bool valid = r.valid;
    const int col0 = nt * BN;
    float vmax = 0.f;
    if (MODE == kGateUp) {
        uint16_t *dst = a.out + grow * a.out_ld + col0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float gv[32], uv[32];
            tmem_load32(taddr + c * 32, gv);
            tmem_load32(taddr + BN + c * 32, uv);
            tmem_load_wait();
            if (valid) {
#pragma unroll
                for (int v8 = 0; v8 < 4; ++v8) {
                    const int col = col0 + c * 32 + v8 * 8;
                    if (col + 8 <= a.n_out) {
                        uint32_t pk[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float a0 = silu_times(gv[v8 * 8 + 2 * i], uv[v8 * 8 + 2 * i]);
                            const float a1 = silu_times(gv[v8 * 8 + 2 * i + 1],
                                                        uv[v8 * 8 + 2 * i + 1]);
                            vmax = fmaxf(vmax, fmaxf(fabsf(a0), fabsf(a1)));
                            pk[i] = pack_f16x2(a0, a1);
                        }
                        *reinterpret_cast<uint4 *>(dst + c * 32 + v8 * 8) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
            }
        }
    } else {
        const float w = r.w;
        uint16_t *dst = a.out + (valid ? q : 0) * a.out_ld + col0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float yv[32];
            tmem_load32(taddr + c * 32, yv);
            tmem_load_wait();
            if (valid) {
#pragma unroll
                for (int v8 = 0; v8 < 4; ++v8) {
                    const int col = col0 + c * 32 + v8 * 8;
                    if (col + 8 <= a.n_out) {
                        float t[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            t[i] = w * yv[v8 * 8 + i];
                            vmax = fmaxf(vmax, fabsf(t[i]));
                        }
                        uint4 pk;
                        pk.x = pack_f16x2(t[0], t[1]);
                        pk.y = pack_f16x2(t[2], t[3]);
                        pk.z = pack_f16x2(t[4], t[5]);
                        pk.w = pack_f16x2(t[6], t[7]);
                        *reinterpret_cast<uint4 *>(dst + c * 32 + v8 * 8) = pk;
                    }
                }
            }
        }
    }
    if (!(vmax <= kF16Max)) record_status(a.status, MOE_ERR_DEVICE_CHECK);
}

}  // namespace moe
