// combine.cu -- K5: weighted accumulate of every token's k expert outputs.
//
// The scatter-add of the M03 "Sparse MoE" drill (each token receives the sum
// of all k weighted expert outputs, an accumulation and never an assignment)
// done without atomics: the down-projection epilogue stored w * Expert(x) of
// pair p = n*k + j at row p of ypair, so token n's k contributions are the k
// consecutive rows n*k .. n*k+k-1.  They are decoded (pair_rows.cuh: bf16 hi
// + int8 residual, 16 significant bits), summed in slot order in fp32, the
// shared-expert term gamma * SharedMLP(x) (same page, talker line), given as
// shared_slots partial rows per token (its chunks of intermediate rows), is
// added last in chunk order, and the result is rounded to bf16 once.  The contributions need
// those 16 bits: the bf16 rounding of the exact result already uses ~97% of
// the layer's max-error bound at prefill size, and an fp16 rounding of each
// contribution (11 bits) pushed the largest outputs past it.
// Bandwidth bound: one thread per 8 output columns, a 16-byte and an 8-byte
// load per contribution and one 16-byte store.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "pair_rows.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kCombineThreads = 256;

// acc[0..7] += the 8 pair-row values held in h (16 bytes of the bf16
// plane) and r (8 bytes of the residual plane)
__device__ __forceinline__ void add_loaded8(float (&acc)[8], uint4 h, uint2 r) {
    const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
    const uint32_t rw[2] = {r.x, r.y};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 hv = unpack_bf16x2(hw[i]);
        const uint32_t rr = rw[i / 2] >> (16 * (i % 2));
        const int r0 = static_cast<int8_t>(rr & 0xFFu);
        const int r1 = static_cast<int8_t>((rr >> 8) & 0xFFu);
        acc[2 * i] += pair_decode(hv.x, r0);
        acc[2 * i + 1] += pair_decode(hv.y, r1);
    }
}

// acc[0..7] += the 8 pair-row values of row offset o, read through L2
__device__ __forceinline__ void add_pair8(float (&acc)[8], const uint16_t *hi_plane,
                                          const int8_t *res_plane, int64_t o) {
    const uint4 h = __ldcg(reinterpret_cast<const uint4 *>(hi_plane + o));
    const uint2 r = __ldcg(reinterpret_cast<const uint2 *>(res_plane + o));
    add_loaded8(acc, h, r);
}

// 32 bytes of the bf16 plane in one load, through L2
__device__ __forceinline__ void ld_cg_v8(const void *p, uint32_t (&v)[8]) {
    asm volatile("ld.global.cg.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7])
                 : "l"(p));
}

// acc[0..15] += the 16 pair-row values of row offset o (32 bytes of the bf16
// plane, 16 of the residual plane)
__device__ __forceinline__ void add_pair16(float (&acc)[16], const uint16_t *hi_plane,
                                           const int8_t *res_plane, int64_t o) {
    uint32_t h[8];
    ld_cg_v8(hi_plane + o, h);
    const uint4 r = __ldcg(reinterpret_cast<const uint4 *>(res_plane + o));
    float a0[8], a1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        a0[i] = acc[i];
        a1[i] = acc[8 + i];
    }
    add_loaded8(a0, make_uint4(h[0], h[1], h[2], h[3]), make_uint2(r.x, r.y));
    add_loaded8(a1, make_uint4(h[4], h[5], h[6], h[7]), make_uint2(r.z, r.w));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        acc[i] = a0[i];
        acc[8 + i] = a1[i];
    }
}

// 16 output columns per thread (H % 16 == 0, large batches): one 32-byte and
// one 16-byte load per slot; the same adds in the same order as the 8-column
// form, so the same bits.
__global__ void __launch_bounds__(kCombineThreads)
    combine16_kernel(const uint16_t *__restrict__ ypair_hi, const int8_t *__restrict__ ypair_res,
                     const int32_t *__restrict__ row_index, int64_t rows,
                     const uint16_t *__restrict__ yshared_hi,
                     const int8_t *__restrict__ yshared_res, int shared_slots, int64_t N,
                     int H, int k, uint16_t *__restrict__ out);

// The row of slot j of token n (-1: a pair that was never sent).
__device__ __forceinline__ int64_t slot_row(const int32_t *row_index, int64_t rows, int64_t n,
                                            int k, int j) {
    const int64_t p = n * k + j;
    const int64_t row = row_index ? static_cast<int64_t>(__ldcg(row_index + p)) : p;
    return row < 0 || row >= rows ? -1 : row;
}

// HOIST (k <= kHoistSlots, small batches): every slot's loads are issued
// before the first add, one round trip to memory instead of k; the adds
// run in the same slot order either way, so both forms give the same bits.
constexpr int kHoistSlots = 8;

template <bool HOIST>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const uint16_t *__restrict__ ypair_hi, const int8_t *__restrict__ ypair_res,
                   const int32_t *__restrict__ row_index, int64_t rows,
                   const uint16_t *__restrict__ yshared_hi,
                   const int8_t *__restrict__ yshared_res, int shared_slots, int64_t N,
                   int H, int k, uint16_t *__restrict__ out) {
    griddep_launch_dependents();
    griddep_wait();
    const int groups = H / 8;
    const int64_t total = N * groups;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = idx / groups;
        const int col = static_cast<int>(idx % groups) * 8;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (HOIST) {
            uint4 h[kHoistSlots];
            uint2 r[kHoistSlots];
            bool live[kHoistSlots];
#pragma unroll
            for (int j = 0; j < kHoistSlots; ++j) {
                const int64_t row = j < k ? slot_row(row_index, rows, n, k, j) : -1;
                live[j] = row >= 0;
                if (live[j]) {
                    h[j] = __ldcg(reinterpret_cast<const uint4 *>(ypair_hi + row * H + col));
                    r[j] = __ldcg(reinterpret_cast<const uint2 *>(ypair_res + row * H + col));
                }
            }
#pragma unroll
            for (int j = 0; j < kHoistSlots; ++j)
                if (live[j]) add_loaded8(acc, h[j], r[j]);
        } else {
            for (int j = 0; j < k; ++j) {
                const int64_t row = slot_row(row_index, rows, n, k, j);
                if (row < 0) continue;  // a pair that was never sent
                add_pair8(acc, ypair_hi, ypair_res, row * H + col);
            }
        }
        for (int c = 0; c < shared_slots; ++c)
            add_pair8(acc, yshared_hi, yshared_res, (n * shared_slots + c) * H + col);
        uint4 pk;
        pk.x = pack_bf16x2(acc[0], acc[1]);
        pk.y = pack_bf16x2(acc[2], acc[3]);
        pk.z = pack_bf16x2(acc[4], acc[5]);
        pk.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4 *>(out + n * H + col) = pk;
    }
}

__global__ void __launch_bounds__(kCombineThreads)
    combine16_kernel(const uint16_t *__restrict__ ypair_hi, const int8_t *__restrict__ ypair_res,
                     const int32_t *__restrict__ row_index, int64_t rows,
                     const uint16_t *__restrict__ yshared_hi,
                     const int8_t *__restrict__ yshared_res, int shared_slots, int64_t N,
                     int H, int k, uint16_t *__restrict__ out) {
    griddep_launch_dependents();
    griddep_wait();
    const int groups = H / 16;
    const int64_t total = N * groups;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = idx / groups;
        const int col = static_cast<int>(idx % groups) * 16;
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
        for (int j = 0; j < k; ++j) {
            const int64_t row = slot_row(row_index, rows, n, k, j);
            if (row < 0) continue;  // a pair that was never sent
            add_pair16(acc, ypair_hi, ypair_res, row * H + col);
        }
        for (int c = 0; c < shared_slots; ++c)
            add_pair16(acc, yshared_hi, yshared_res, (n * shared_slots + c) * H + col);
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
        st_global_v8(out + n * H + col, pk);
    }
}

}  // namespace

cudaError_t launch_combine(const uint16_t *ypair_hi, const int8_t *ypair_res,
                           const int32_t *row_index, int64_t rows, const uint16_t *yshared_hi,
                           const int8_t *yshared_res, int shared_slots, int64_t N, int H, int k,
                           uint16_t *out, int num_sms, cudaStream_t s) {
    const int64_t total = N * (H / 8);
    int64_t blocks = (total + kCombineThreads - 1) / kCombineThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    // few tokens: latency-bound, so every slot's loads go out at once; many
    // tokens: bandwidth-bound, where the hoisted form's registers would cost
    // occupancy
    const bool hoist = k <= kHoistSlots && N <= 256;
    // 32-byte accesses need 32-byte aligned planes and output
    const bool al32 = ((reinterpret_cast<uintptr_t>(ypair_hi) |
                        reinterpret_cast<uintptr_t>(yshared_hi) |
                        reinterpret_cast<uintptr_t>(out)) & 31u) == 0;
    if (!hoist && H % 16 == 0 && al32) {
        const int64_t total16 = N * (H / 16);
        int64_t b16 = (total16 + kCombineThreads - 1) / kCombineThreads;
        if (b16 > cap) b16 = cap;
        return launch_pdl(combine16_kernel, dim3(static_cast<unsigned>(b16)),
                          dim3(kCombineThreads), 0, s, 1, ypair_hi, ypair_res, row_index, rows,
                          yshared_hi, yshared_res, yshared_hi ? shared_slots : 0, N, H, k, out);
    }
    return launch_pdl(hoist ? combine_kernel<true> : combine_kernel<false>,
                      dim3(static_cast<unsigned>(blocks)), dim3(kCombineThreads), 0, s, 1,
                      ypair_hi, ypair_res, row_index, rows, yshared_hi, yshared_res,
                      yshared_hi ? shared_slots : 0, N, H, k, out);
}

}  // namespace moe
