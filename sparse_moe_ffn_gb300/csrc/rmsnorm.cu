// rmsnorm.cu -- the decoder layer's step before the MoE, in one kernel:
// residual-add then RMSNorm (Nano-vLLM notes, question 4 on the decoder
// layer: "x += residual; residual = x; return norm(x)", done in one GPU
// kernel; Qwen3.5 walkthrough section 2.1, fused add + norm).
//
//   r        = bf16(x + residual)         (the add in the model's dtype)
//   residual = r
//   normed   = bf16(r / sqrt(mean(r^2) + eps) * w)      or * (1 + w) (Gemma)
//
// One warp per token row, 16-byte loads and stores, the sum of squares in
// fp32 (per lane, then a shuffle tree).  Bandwidth bound: 8 bytes read and 4
// written per element (plus the weight, read from L2).
#include <cuda_bf16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads)
    add_rmsnorm_kernel(const uint16_t *__restrict__ x, uint16_t *__restrict__ residual,
                       const uint16_t *__restrict__ w, int64_t N, int H, float eps, int gemma,
                       uint16_t *__restrict__ normed) {
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x % 32;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
    const int groups = H / 8;
    for (int64_t n = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32; n < N;
         n += warps) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(x + n * H);
        uint4 *rr = reinterpret_cast<uint4 *>(residual + n * H);
        float ss = 0.f;
        for (int g = lane; g < groups; g += 32) {
            const uint4 a = __ldcg(xr + g), b = __ldcg(rr + g);
            const __nv_bfloat162 *ah = reinterpret_cast<const __nv_bfloat162 *>(&a);
            const __nv_bfloat162 *bh = reinterpret_cast<const __nv_bfloat162 *>(&b);
            uint4 o;
            uint32_t *op = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 fa = __bfloat1622float2(ah[i]), fb = __bfloat1622float2(bh[i]);
                const __nv_bfloat162 s = __floats2bfloat162_rn(fa.x + fb.x, fa.y + fb.y);
                const float2 fs = __bfloat1622float2(s);
                ss += fs.x * fs.x + fs.y * fs.y;
                op[i] = *reinterpret_cast<const uint32_t *>(&s);
            }
            rr[g] = o;
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
        const float inv = 1.f / sqrtf(ss / static_cast<float>(H) + eps);
        const uint4 *wr = reinterpret_cast<const uint4 *>(w);
        uint4 *nr = reinterpret_cast<uint4 *>(normed + n * H);
        for (int g = lane; g < groups; g += 32) {
            const uint4 r = rr[g], wv = __ldg(wr + g);  // r: this thread's own store above
            const __nv_bfloat162 *rh = reinterpret_cast<const __nv_bfloat162 *>(&r);
            const __nv_bfloat162 *wh = reinterpret_cast<const __nv_bfloat162 *>(&wv);
            uint4 o;
            uint32_t *op = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 fr = __bfloat1622float2(rh[i]);
                float2 fw = __bfloat1622float2(wh[i]);
                if (gemma) {
                    fw.x += 1.f;
                    fw.y += 1.f;
                }
                op[i] = pack_bf16x2(fr.x * inv * fw.x, fr.y * inv * fw.y);
            }
            nr[g] = o;
        }
    }
}

}  // namespace

cudaError_t launch_add_rmsnorm(const uint16_t *x, uint16_t *residual, const uint16_t *w,
                               int64_t N, int H, float eps, int gemma, uint16_t *normed,
                               int num_sms, cudaStream_t s) {
    int64_t blocks = (N * 32 + kNormThreads - 1) / kNormThreads;
    const int64_t limit = static_cast<int64_t>(num_sms) * 16;
    if (blocks > limit) blocks = limit;
    return launch_pdl(add_rmsnorm_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kNormThreads),
                      0, s, 1, x, residual, w, N, H, eps, gemma, normed);
}

}  // namespace moe
