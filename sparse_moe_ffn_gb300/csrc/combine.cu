// combine.cu -- K5: weighted accumulate of every token's k expert outputs.
//
// The scatter-add of the M03 "Sparse MoE" drill ("out.index_add_(0, toks,
// y * w)": each token receives the sum of all k contributions, never just the
// last one written) done without atomics: the down-projection epilogue stored
// w * Expert(x) of pair p = n*k + j at row p of ypair, so token n's k
// contributions are the k consecutive fp16 rows n*k .. n*k+k-1.  They are
// summed in slot order in fp32, the shared-expert term gamma * SharedMLP(x) (same
// page, talker line) is added last, and the result is rounded to bf16 once.
// Bandwidth bound: one thread per 8 output columns, 16-byte loads and stores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kCombineThreads = 256;

__device__ __forceinline__ void add_f16x8(float (&acc)[8], const uint4 &v) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h[i]);
        acc[2 * i] += f.x;
        acc[2 * i + 1] += f.y;
    }
}

__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const uint16_t *__restrict__ ypair, const uint16_t *__restrict__ yshared,
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
        const uint16_t *src = ypair + n * k * static_cast<int64_t>(H) + col;
        for (int j = 0; j < k; ++j)
            add_f16x8(acc, __ldcg(reinterpret_cast<const uint4 *>(src + static_cast<int64_t>(j) * H)));
        if (yshared)
            add_f16x8(acc, __ldcg(reinterpret_cast<const uint4 *>(yshared + n * H + col)));
        uint4 pk;
        pk.x = pack_bf16x2(acc[0], acc[1]);
        pk.y = pack_bf16x2(acc[2], acc[3]);
        pk.z = pack_bf16x2(acc[4], acc[5]);
        pk.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4 *>(out + n * H + col) = pk;
    }
}

}  // namespace

cudaError_t launch_combine(const uint16_t *ypair, const uint16_t *yshared, int64_t N, int H,
                           int k, uint16_t *out, int num_sms, cudaStream_t s) {
    const int64_t total = N * (H / 8);
    int64_t blocks = (total + kCombineThreads - 1) / kCombineThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    return launch_pdl(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kCombineThreads),
                      0, s, 1, ypair, yshared, N, H, k, out);
}

}  // namespace moe
