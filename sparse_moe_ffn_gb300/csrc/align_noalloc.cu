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
// it; that first call should therefore come before any stream capture.  All
// calls share the one array: calls whose work overlaps on the GPU (other
// streams, other host threads) race with each other.  The scratch needs no
// clearing between calls: moe_align resets the status word and writes every
// chunk count before reading it.
#include <mutex>

#include "kernels.cuh"
#include "moe.h"

namespace {

constexpr size_t kNoallocScratchBytes = MOE_ALIGN_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_address[kMaxDevices] = {nullptr};

// Device address of g_noalloc_scratch on the current device (looked up once).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_address[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_address[dev] = p;
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
    if (N == 0) return MOE_OK;
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
