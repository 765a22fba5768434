// convert.cu -- data movement around the layer: the load-time conversion of
// the down-projection weights from the model's bf16 to the fp16 operand
// format of the down GEMM, and the copies between pinned host buffers and
// the device for moe_forward_host.
//
// bf16 -> fp32 is exact, and fp32 -> fp16 rounds to nearest even: a bf16
// value carries 8 significant bits and fp16 11, so every value from 2^-14
// (fp16's smallest normal) to 65504 converts exactly; smaller magnitudes land
// on fp16's subnormal grid (spacing 2^-24).  A magnitude above 65504, or a
// NaN, records MOE_ERR_DEVICE_CHECK.  Bandwidth bound: 8 values per thread
// with 16-byte loads and stores, the last n % 8 values one at a time.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kConvertThreads = 256;
constexpr float kHalfMax = 65504.f;

__device__ __forceinline__ uint16_t bf16_to_f16(uint16_t b, bool &bad) {
    const float f = __uint_as_float(static_cast<uint32_t>(b) << 16);
    bad |= !(fabsf(f) <= kHalfMax);
    return __half_as_ushort(__float2half_rn(f));
}

__global__ void __launch_bounds__(kConvertThreads)
    convert_kernel(const uint16_t *__restrict__ src, uint16_t *__restrict__ dst, int64_t n,
                   int32_t *status) {
    const int64_t groups = n / 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    bool bad = false;
    for (int64_t i = tid; i < groups; i += stride) {
        const uint4 v = reinterpret_cast<const uint4 *>(src)[i];
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = bf16_to_f16(static_cast<uint16_t>(in[j] & 0xffffu), bad);
            const uint32_t hi = bf16_to_f16(static_cast<uint16_t>(in[j] >> 16), bad);
            out[j] = lo | (hi << 16);
        }
        reinterpret_cast<uint4 *>(dst)[i] = make_uint4(out[0], out[1], out[2], out[3]);
    }
    for (int64_t i = groups * 8 + tid; i < n; i += stride) dst[i] = bf16_to_f16(src[i], bad);
    if (bad) record_status(status, MOE_ERR_DEVICE_CHECK);
}

// dst[i] = src[i] over n16 16-byte words, one side being pinned host memory
// mapped into the device's address space: all SMs read or write it over the
// CPU-GPU link directly, four words per thread in flight.
__global__ void __launch_bounds__(kConvertThreads)
    copy16_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int64_t n16) {
    griddep_launch_dependents();
    griddep_wait();  // the source may be the previous kernel's output
    constexpr int kUnroll = 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t i0 = tid; i0 < n16; i0 += stride * kUnroll) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (i0 + u * stride < n16) v[u] = src[i0 + u * stride];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (i0 + u * stride < n16) dst[i0 + u * stride] = v[u];
    }
}

}  // namespace

cudaError_t launch_copy16(const void *src, void *dst, size_t bytes, int num_sms, cudaStream_t s) {
    const int64_t n16 = static_cast<int64_t>(bytes / 16);
    int64_t blocks = (n16 + kConvertThreads - 1) / kConvertThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(copy16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kConvertThreads), 0,
                      s, 1, static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n16);
}

cudaError_t launch_convert_bf16_to_f16(const uint16_t *src, uint16_t *dst, int64_t n,
                                       int32_t *status, int num_sms, cudaStream_t s) {
    int64_t blocks = (n / 8 + kConvertThreads - 1) / kConvertThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    convert_kernel<<<static_cast<unsigned>(blocks), kConvertThreads, 0, s>>>(src, dst, n, status);
    return cudaGetLastError();
}

}  // namespace moe
