// combine.cu -- K5: weighted accumulate of every token's k expert outputs.
//
// The scatter-add of the M03 "Sparse MoE" drill (each token receives the sum
// of all k weighted expert outputs, an accumulation and never an assignment)
// done without atomics: the down-projection epilogue stored w * Expert(x) of
// pair p = n*k + j at row p of ypair in fp32, so token n's k contributions
// are the k consecutive rows n*k .. n*k+k-1.  They are summed in slot order
// in fp32, the shared-expert term gamma * SharedMLP(x) (same page, talker
// line) is added last, and the result is rounded to bf16 once.  Keeping the
// contributions in fp32 matters: the bf16 rounding of the exact result
// already uses ~97% of the layer's max-error bound at prefill size, and an
// fp16 rounding of each contribution pushed the largest outputs past it.
// Bandwidth bound: one thread per 8 output columns, two 16-byte loads per
// contribution and one 16-byte store.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kCombineThreads = 256;

// acc[0..7] += the 8 floats at p (32-byte aligned), read through L2
__device__ __forceinline__ void add_f32x8(float (&acc)[8], const float *p) {
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldcg(reinterpret_cast<const float4 *>(p + 4));
    acc[0] += a.x;
    acc[1] += a.y;
    acc[2] += a.z;
    acc[3] += a.w;
    acc[4] += b.x;
    acc[5] += b.y;
    acc[6] += b.z;
    acc[7] += b.w;
}

__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float *__restrict__ ypair, const float *__restrict__ yshared,
                   int64_t N, int H, int k, uint16_t *__restrict__ out) {
    griddep_launch_dependents();
    griddep_wait();
    const int groups = H / 8;
    const int64_t total = N * groups;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = idx / groups;
        const int col = static_cast<int>(idx % groups) * 8;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const float *src = ypair + n * k * static_cast<int64_t>(H) + col;
        for (int j = 0; j < k; ++j) add_f32x8(acc, src + static_cast<int64_t>(j) * H);
        if (yshared) add_f32x8(acc, yshared + n * H + col);
        uint4 pk;
        pk.x = pack_bf16x2(acc[0], acc[1]);
        pk.y = pack_bf16x2(acc[2], acc[3]);
        pk.z = pack_bf16x2(acc[4], acc[5]);
        pk.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4 *>(out + n * H + col) = pk;
    }
}

}  // namespace

cudaError_t launch_combine(const float *ypair, const float *yshared, int64_t N, int H, int k,
                           uint16_t *out, int num_sms, cudaStream_t s) {
    const int64_t total = N * (H / 8);
    int64_t blocks = (total + kCombineThreads - 1) / kCombineThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    return launch_pdl(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kCombineThreads),
                      0, s, 1, ypair, yshared, N, H, k, out);
}

}  // namespace moe
