// gemm_common.cuh -- pieces shared by the grouped GEMM kernels (one-CTA,
// 32-row sparse and CTA-pair): tile constants, the SwiGLU helper and the
// epilogue that turns one TMEM accumulator row into stored outputs.
#pragma once

#include <cuda_bf16.h>

#include "kernels.cuh"
#include "pair_rows.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kATileBytes = kBlockM * 128;  // 128 rows x 64 bf16
constexpr int kAccCols = 256;               // fp32 columns per accumulator
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr float kF16Max = 65504.f;
constexpr float kF32Max = 3.402823466e38f;
constexpr int kSparseRows = 32;             // blocks with at most this many real rows gather

// silu(g) * u = g / (1 + e^-g) * u, with the fast division (a reciprocal
// and a multiply, ~2 ulp; the activation is rounded to 11 or 16 bits after
// it).  The exponent is capped at 80 so that the divisor stays below 2^126,
// the fast division's range; for g < -80 silu is below 1e-33 in magnitude
// either way.
__device__ __forceinline__ float silu_times(float g, float u) {
    return __fdividef(g, 1.f + __expf(fminf(-g, 80.f))) * u;
}

// max(a, |b|, |c|) that returns NaN when any operand is NaN (fmaxf drops a
// NaN operand), so that the stored-range checks below see NaN outputs too
__device__ __forceinline__ float max_abs_nan(float a, float b, float c) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(fabsf(b)), "f"(fabsf(c)));
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(r), "f"(a));
    return r;
}

// Where the weight rows of N tile nt of group (expert) `expert` are: the
// routed weights (row expert * w_rows + n0 + extra, K from 0), or, for a
// virtual expert of the folded shared expert, the shared weights (gate/up:
// row v * virt_chunk + n0; down: row n0 + extra, K from v * virt_chunk).
struct WeightCoord {
    bool shared;
    int row;
    int k0;
};

template <int MODE>
__device__ __forceinline__ WeightCoord weight_coord(const GemmArgs &a, int expert, int n0,
                                                    int extra) {
    WeightCoord c;
    c.shared = expert >= a.virt_base;
    if (!c.shared) {
        c.row = static_cast<int>(static_cast<int64_t>(expert) * a.w_rows) + n0 + extra;
        c.k0 = 0;
    } else if (MODE == kGateUp) {
        c.row = (expert - a.virt_base) * a.virt_chunk + n0 + extra;
        c.k0 = 0;
    } else {
        c.row = n0 + extra;
        c.k0 = (expert - a.virt_base) * a.virt_chunk;
    }
    return c;
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

// The pair (or token) held by grouped row grow: one load, issued early.
__device__ __forceinline__ int64_t row_pair(const GemmArgs &a, int64_t grow) {
    return a.sorted_pair ? __ldcg(a.sorted_pair + grow) : grow;
}

// The TileRow of grouped row grow, whose pair q is already known; issues the
// routing-weight load (down) without waiting for it.
template <int MODE>
__device__ __forceinline__ TileRow tile_row_of(const GemmArgs &a, int64_t grow, int64_t q) {
    TileRow r;
    r.grow = grow;
    r.q = q;
    r.valid = q >= 0 && q < a.q_limit;
    r.w = (is_down(MODE) && r.valid) ? (a.scale ? __ldcg(a.scale + q) : 1.f) : 0.f;
    return r;
}

template <int MODE>
__device__ __forceinline__ TileRow tile_row(const GemmArgs &a, int blk, int row) {
    const int64_t grow = static_cast<int64_t>(blk) * kBlockM + row;
    return tile_row_of<MODE>(a, grow, row_pair(a, grow));
}

// A tile row that stores nothing (its block holds no rows).
__device__ __forceinline__ TileRow no_tile_row() {
    TileRow r;
    r.grow = 0;
    r.q = -1;
    r.w = 0.f;
    r.valid = false;
    return r;
}

// Epilogue of one tile for the thread that owns TMEM lane r.grow % 128:
// output columns [nt * BN, nt * BN + BN) (gate/up: the accumulator holds BN
// gate columns, then BN up columns).  taddr = this warp's TMEM lane quarter
// and the tile's accumulator.
//   gate/up: a = silu(g) * u in fp32, stored as the down projection's A
//            operand: fp16(a) (a.lo_rows == 0), or the bf16 pair
//            hi = bf16(a) at row grow and lo = bf16(a - hi) at row
//            grow + a.lo_rows (hi + lo carries 16 significant bits);
//   down:    y[q] = w[q] * acc in fp32, the pair's weighted result, stored
//            as a pair row (pair_rows.cuh: bf16 hi + int8 residual, 16
//            significant bits) until the combine rounds the token's sum to
//            bf16 once.
// A value the stored format cannot hold (an fp16 activation past 65504, or
// anything non-finite) is reported as MOE_ERR_DEVICE_CHECK.
template <int MODE, int BN>
__device__ __forceinline__ void store_tile(const GemmArgs &a, uint32_t taddr, const TileRow &r,
                                           int nt) {
    static_assert(MODE == kGateUp || BN % 64 == 0, "down tiles are read 64 columns at a time");
    const int64_t grow = r.grow;
    const int64_t q = r.q;
    const bool valid = r.valid;
    const int col0 = nt * BN;
    float vmax = 0.f;
    // 32 bytes per store when every output row starts on a 32-byte boundary,
    // else 16; stores never pass n_out (a multiple of 8)
    const int esize = 2;  // bf16 / fp16 outputs
    const bool wide = (a.out_ld * esize) % 32 == 0 && (reinterpret_cast<uintptr_t>(a.out) % 32) == 0;
    // 32 bytes (pk) to dst, which holds elements [col, col + 32 / esize)
    auto store32 = [&](void *dst, int col, const uint32_t (&pk)[8]) {
        const int per16 = 16 / esize;
        if (wide && col + 2 * per16 <= a.n_out) {
            st_global_v8(dst, pk);
        } else {
            if (col + per16 <= a.n_out)
                *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            if (col + 2 * per16 <= a.n_out)
                *reinterpret_cast<uint4 *>(static_cast<uint8_t *>(dst) + 16) =
                    make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
    };
    if (MODE == kGateUp) {
        uint16_t *dst = static_cast<uint16_t *>(a.out) + grow * a.out_ld + col0;
        const bool split = a.lo_rows != 0;
        uint16_t *dst_lo = dst + a.lo_rows * a.out_ld;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float gv[32], uv[32];
            tmem_load32(taddr + c * 32, gv);
            tmem_load32(taddr + BN + c * 32, uv);
            tmem_load_wait();
            if (valid) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[8], pl[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int j = h * 16 + 2 * i;
                        const float a0 = silu_times(gv[j], uv[j]);
                        const float a1 = silu_times(gv[j + 1], uv[j + 1]);
                        vmax = max_abs_nan(vmax, a0, a1);
                        if (split) {
                            pk[i] = pack_bf16x2(a0, a1);
                            const float2 hi = unpack_bf16x2(pk[i]);
                            pl[i] = pack_bf16x2(a0 - hi.x, a1 - hi.y);
                        } else {
                            pk[i] = pack_f16x2(a0, a1);
                        }
                    }
                    const int cc = c * 32 + h * 16;
                    store32(dst + cc, col0 + cc, pk);
                    if (split) store32(dst_lo + cc, col0 + cc, pl);
                }
            }
        }
        if (!(vmax <= (split ? kF32Max : kF16Max))) record_status(a.status, MOE_ERR_DEVICE_CHECK);
    } else {
        const float w = r.w;
        const int64_t row = (valid ? q : 0) * a.out_ld + col0;
        uint16_t *dst = static_cast<uint16_t *>(a.out) + row;
        int8_t *dst_res = a.out_res + row;
        // residual plane: 16 bytes per 16 columns when its rows start on
        // 16-byte boundaries, else 8
        const bool res16 = a.out_ld % 16 == 0;
        // 64 columns per TMEM round trip: two loads in flight, one wait
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
            float yv[64];
            tmem_load32(taddr + c * 64, *reinterpret_cast<float(*)[32]>(yv));
            tmem_load32(taddr + c * 64 + 32, *reinterpret_cast<float(*)[32]>(yv + 32));
            tmem_load_wait();
            if (valid) {
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t pk[8], pr[4];
                    float tv[16], hv[16];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        tv[2 * i] = w * yv[h * 16 + 2 * i];
                        tv[2 * i + 1] = w * yv[h * 16 + 2 * i + 1];
                        vmax = max_abs_nan(vmax, tv[2 * i], tv[2 * i + 1]);
                        pk[i] = pack_bf16x2(tv[2 * i], tv[2 * i + 1]);
                        const float2 hi = unpack_bf16x2(pk[i]);
                        hv[2 * i] = hi.x;
                        hv[2 * i + 1] = hi.y;
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        pr[i] = pair_residual4(tv[4 * i], hv[4 * i], tv[4 * i + 1], hv[4 * i + 1],
                                               tv[4 * i + 2], hv[4 * i + 2], tv[4 * i + 3],
                                               hv[4 * i + 3]);
                    const int cc = c * 64 + h * 16;
                    store32(dst + cc, col0 + cc, pk);
                    if (col0 + cc + 16 <= a.n_out && res16) {
                        *reinterpret_cast<uint4 *>(dst_res + cc) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
                    } else {
                        if (col0 + cc + 8 <= a.n_out)
                            *reinterpret_cast<uint2 *>(dst_res + cc) = make_uint2(pr[0], pr[1]);
                        if (col0 + cc + 16 <= a.n_out)
                            *reinterpret_cast<uint2 *>(dst_res + cc + 8) = make_uint2(pr[2], pr[3]);
                    }
                }
            }
        }
        if (!(vmax <= kF32Max)) record_status(a.status, MOE_ERR_DEVICE_CHECK);
    }
}

}  // namespace moe
