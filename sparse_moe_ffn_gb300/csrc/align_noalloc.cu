// align_noalloc.cu -- moe_align_noalloc: moe_align for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain scratch memory at the point where they
// group the routed pairs: code that is being captured into a CUDA graph may
// not call cudaMalloc, plugin-style hosts hand a kernel only its input and
// output buffers, and latency-critical paths must not take an allocator's
// locks or its implicit device synchronisation.  This entry point keeps its
// scratch (status word, padded offsets, per-chunk counts) in a file-scope
// device array instead, so the caller passes only inputs and outputs.
//
// The array is kNoallocScratchBytes (1 MiB) on every GPU that loads the
// library, held until the process exits.  Host code cannot use the array's
// name as a device address, so the first call on each device looks the
// address up with cudaGetSymbolAddress (with that device current) and caches
// it; that first call should therefore come before any stream capture.  The
// cache remembers the CUDA context the address belongs to, and looks it up
// again when the device's current context has changed (after a
// cudaDeviceReset the runtime makes a new one).  All
// calls share the one array: calls whose work overlaps on the GPU (other
// streams, other host threads) race with each other.  The scratch needs no
// clearing between calls: moe_align resets the status word and writes every
// chunk count before reading it.
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.cuh"
#include "moe.h"

namespace {

constexpr size_t kNoallocScratchBytes = MOE_ALIGN_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_address[kMaxDevices] = {nullptr};
CUcontext g_scratch_context[kMaxDevices] = {nullptr};

// The driver's cuCtxGetCurrent (looked up once through the runtime).
PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    });
    return fn;
}

// Device address of g_noalloc_scratch on the current device: looked up once
// per device and context, with that device current.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    CUcontext ctx = nullptr;
    auto get_ctx = ctx_get_current();
    if (get_ctx && get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_address[dev] == nullptr || ctx == nullptr || g_scratch_context[dev] != ctx) {
        // (this also makes the device's primary context current if no
        // context was yet)
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (get_ctx && get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
        g_scratch_address[dev] = p;
        g_scratch_context[dev] = ctx;
    }
    *out = g_scratch_address[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" moe_status_t moe_align_noalloc(const int32_t *topk_ids, int64_t N, int k, int E,
                                          int block_m, int32_t *sorted_pair,
                                          int32_t *block_expert, int32_t *counts,
                                          int32_t *offsets, int32_t *num_padded,
                                          int32_t *device_status, cudaStream_t stream) {
    if (N < 0 || k < 1 || E < 1 || block_m < 1) return moe_align(topk_ids, N, k, E, block_m,
                                                                  sorted_pair, block_expert,
                                                                  counts, offsets, num_padded,
                                                                  nullptr, 0, stream);
    const size_t need = moe_align_workspace_bytes(N, k, E, block_m);
    if (need > kNoallocScratchBytes) {
        moe::set_last_error("moe_align_noalloc: this size needs more scratch than the library's "
                            "static MOE_ALIGN_NOALLOC_SCRATCH_BYTES; use moe_align");
        return MOE_ERR_UNSUPPORTED;
    }
    if (N == 0) {  // nothing to group: the status word still reports the call
        if (device_status &&
            cudaMemsetAsync(device_status, 0, sizeof(int32_t), stream) != cudaSuccess) {
            moe::set_last_error("moe_align_noalloc: status reset failed");
            return MOE_ERR_CUDA;
        }
        return MOE_OK;
    }
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) {
        moe::set_last_error("moe_align_noalloc: cudaGetSymbolAddress of the static scratch failed");
        return MOE_ERR_CUDA;
    }
    moe_status_t st = moe_align(topk_ids, N, k, E, block_m, sorted_pair, block_expert, counts,
                                offsets, num_padded, scratch, kNoallocScratchBytes, stream);
    if (st != MOE_OK || device_status == nullptr) return st;
    // the status word sits at the start of the scratch (moe_align's layout)
    if (cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                        stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
