// ep.cu -- the sending side of expert-parallel dispatch on the device: the
// (token, slot) pairs grouped by the rank that owns their expert, and the
// rows, local expert ids and weights packed in that order for the
// all-to-all (the M03 drill's level-3 follow-up: the (token, expert) table
// drives the exchange).  Rank r of R owns experts [r E_r, (r + 1) E_r),
// E_r = ceil(E / R).
//
//   1. dest[p] = ids[p] / E_r for every pair p = n k + j, and inv[p] = -1
//      (ep_dest_kernel);
//   2. the pairs grouped by dest, in pair order within a rank: the grouping
//      kernels of moe_align with R groups and blocks of one row, so that
//      order[i] lists the pairs rank by rank and counts[r] is the number
//      sent to rank r;
//   3. send row i = pair order[i]: x[order[i] / k], its local expert id
//      ids - dest E_r and its weight, plus inv[order[i]] = i, the row at
//      which the pair's result will come back (ep_pack_kernel).
// Integer and copy work: one warp per send row copies the token's H bf16
// values with 16-byte accesses.
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kEpThreads = 256;

__global__ void __launch_bounds__(kEpThreads)
    ep_dest_kernel(const int32_t *__restrict__ ids, int64_t P, int E, int e_local,
                   int32_t *__restrict__ dest, int32_t *__restrict__ inv, int32_t *status) {
    griddep_launch_dependents();
    griddep_wait();  // the ids may come from the routing kernel just before
    bool bad = false;
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < P;
         p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t e = __ldcg(ids + p);
        inv[p] = -1;  // no send row yet (stays so for a pair with a bad id)
        // an id outside [0, E) gets no rank (the grouping skips it)
        if (e < 0 || e >= E) {
            bad = true;
            dest[p] = -1;
        } else {
            dest[p] = e / e_local;
        }
    }
    if (bad) record_status(status, MOE_ERR_DEVICE_CHECK);
}

__global__ void __launch_bounds__(kEpThreads)
    ep_pack_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ ids,
                   const float *__restrict__ weights, const int32_t *__restrict__ order,
                   const int32_t *__restrict__ num_rows, int64_t P, int H, int k, int e_local,
                   uint16_t *__restrict__ send_x, int32_t *__restrict__ send_ids,
                   float *__restrict__ send_w, int32_t *__restrict__ inv) {
    griddep_launch_dependents();
    griddep_wait();
    const int warps = blockDim.x / 32;
    const int lane = threadIdx.x % 32;
    // pairs with a bad id were left out of the grouping
    const int64_t rows = min(static_cast<int64_t>(__ldcg(num_rows)), P);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * warps + threadIdx.x / 32; i < rows;
         i += static_cast<int64_t>(gridDim.x) * warps) {
        const int32_t q = __ldcg(order + i);
        if (q < 0 || q >= P) continue;
        if (lane == 0) {
            const int32_t e = __ldcg(ids + q);
            send_ids[i] = e - (e / e_local) * e_local;
            send_w[i] = __ldcg(weights + q);
            inv[q] = static_cast<int32_t>(i);
        }
        const uint4 *src = reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(q / k) * H);
        uint4 *dst = reinterpret_cast<uint4 *>(send_x + i * H);
        for (int c = lane; c < H / 8; c += 32) dst[c] = __ldcg(src + c);
    }
}

// The shared expert run on its own (a rank's local term): every token n
// gets C slots p = n C + c, slot c being chunk c (virtual expert c) with
// the shared gate gamma[n] as its weight.
__global__ void __launch_bounds__(kEpThreads)
    shared_slots_kernel(const float *__restrict__ gamma, int64_t N, int C,
                        int32_t *__restrict__ ids, float *__restrict__ w) {
    griddep_launch_dependents();
    griddep_wait();  // gamma may come from the routing kernel just before
    const int64_t P = N * C;
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < P;
         p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        ids[p] = static_cast<int32_t>(p % C);
        w[p] = __ldcg(gamma + p / C);
    }
}

}  // namespace

cudaError_t launch_ep_dest(const int32_t *ids, int64_t P, int E, int e_local, int32_t *dest,
                           int32_t *inv, int32_t *status, int num_sms, cudaStream_t s) {
    int64_t blocks = (P + kEpThreads - 1) / kEpThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(ep_dest_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kEpThreads), 0,
                      s, 1, ids, P, E, e_local, dest, inv, status);
}

cudaError_t launch_ep_pack(const uint16_t *x, const int32_t *ids, const float *weights,
                           const int32_t *order, const int32_t *num_rows, int64_t P, int H, int k,
                           int e_local, uint16_t *send_x, int32_t *send_ids, float *send_w,
                           int32_t *inv, int num_sms, cudaStream_t s) {
    const int warps = kEpThreads / 32;
    int64_t blocks = (P + warps - 1) / warps;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(ep_pack_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kEpThreads), 0, s,
                      1, x, ids, weights, order, num_rows, P, H, k, e_local, send_x, send_ids,
                      send_w, inv);
}

cudaError_t launch_shared_slots(const float *gamma, int64_t N, int C, int32_t *ids, float *w,
                                int num_sms, cudaStream_t s) {
    int64_t blocks = (N * C + kEpThreads - 1) / kEpThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(shared_slots_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kEpThreads),
                      0, s, 1, gamma, N, C, ids, w);
}

}  // namespace moe
