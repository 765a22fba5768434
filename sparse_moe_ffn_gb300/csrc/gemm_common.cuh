// gemm_common.cuh -- pieces shared by the one-CTA and the CTA-pair grouped
// GEMM kernels: tile constants, the SwiGLU and hi/lo helpers and the epilogue
// that turns one TMEM accumulator row into stored outputs.
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

// a -> (hi, lo) with hi = bf16(a) and lo = bf16(a - hi), two values at a time
__device__ __forceinline__ void split_bf16x2(float a0, float a1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a0, a1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a0 - hf.x, a1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Epilogue of one tile for the thread that owns TMEM lane `row`: row `row`
// of row block `blk`, output columns [nt * BN, nt * BN + BN) (gate/up: the
// accumulator holds BN gate columns, then BN up columns).  taddr = this
// warp's TMEM lane quarter and the tile's accumulator.
template <int MODE, int BN>
__device__ __forceinline__ void store_tile(const GemmArgs &a, uint32_t taddr, int blk, int nt,
                                           int row) {
    const int64_t grow = static_cast<int64_t>(blk) * kBlockM + row;
    const int64_t q = a.sorted_pair ? __ldcg(a.sorted_pair + grow) : grow;
    const bool valid = q >= 0 && q < a.q_limit;
    const int col0 = nt * BN;
    if (MODE == kGateUp) {
        uint16_t *dst = a.out + grow * a.out_ld + col0;
        uint16_t *dst_lo = a.out_lo + grow * a.out_ld + col0;
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
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float a0 = silu_times(gv[v8 * 8 + 2 * i], uv[v8 * 8 + 2 * i]);
                            const float a1 = silu_times(gv[v8 * 8 + 2 * i + 1],
                                                        uv[v8 * 8 + 2 * i + 1]);
                            split_bf16x2(a0, a1, hi[i], lo[i]);
                        }
                        *reinterpret_cast<uint4 *>(dst + c * 32 + v8 * 8) =
                            make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4 *>(dst_lo + c * 32 + v8 * 8) =
                            make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
            }
        }
    } else {
        const float w = !valid ? 0.f : (a.scale ? __ldcg(a.scale + q) : 1.f);
        uint16_t *dst = a.out + (valid ? q : 0) * a.out_ld + col0;
        float vmax = 0.f;
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
        // fp16 keeps 11 significant bits; a value past its range is
        // reported rather than silently turned into infinity
        if (!(vmax <= kF16Max)) record_status(a.status, MOE_ERR_DEVICE_CHECK);
    }
}

}  // namespace moe
