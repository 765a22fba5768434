// router.cu -- K1: fused router GEMM + fp32 softmax over all experts + top-k
// + optional renormalisation (+ the talker's scalar shared-expert gate).
//
// Follows the routing block of the M03 "Sparse MoE" drill (problem overview):
// logits = x @ router^T, softmax over all E in fp32, top-k in descending
// order, w /= sum(w) when norm_topk_prob; weights are also returned in bf16
// (the pages return them in x's dtype) and ids as int32.  The shared gate is
// sigmoid(x . g), one scalar per token (same page, shared-expert line).
//
// One CTA owns 128 tokens.  The logits tile [128 x e_pad] is one tcgen05 MMA
// chain: x rows are the A operand (M = 128 tokens), router rows are B (N =
// e_pad experts, plus g in column gamma_col), K = H streamed through a 4-stage
// TMA pipeline in 64-wide slices.  The fp32 accumulator sits in TMEM with
// token r in lane r, so the epilogue thread of lane r owns its whole logit
// row: max, sum of exponentials and the k arg-max rounds need no cross-thread
// reduction at all.  The reduction order over H is the same for every token
// and every N, which makes routing batch invariant bit for bit.
#include <cuda_bf16.h>
#include <math.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kRouterStages = 4;
constexpr int kRouterThreads = 128;
constexpr int kATileBytes = kBlockM * 128;  // 128 tokens x 64 bf16

struct RouterSmem {
    uint64_t full[kRouterStages];
    uint64_t empty[kRouterStages];
    uint64_t acc_full;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ float finite_or_neg_inf(float v) {
    return (v != v) ? -INFINITY : v;  // NaN never wins a comparison
}

__global__ void __launch_bounds__(kRouterThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap tm_x,
                  const __grid_constant__ CUtensorMap tm_router,
                  const __grid_constant__ CUtensorMap tm_gate, const RouterArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int b_tile_bytes = a.e_pad * 128;
    const int stage_bytes = kATileBytes + b_tile_bytes;
    RouterSmem *sm = reinterpret_cast<RouterSmem *>(tiles + kRouterStages * stage_bytes);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBlockM;
    const int nk = (a.H + kBlockK - 1) / kBlockK;
    const uint32_t tmem_cols = a.e_pad <= 32 ? 32 : (a.e_pad <= 64 ? 64 : (a.e_pad <= 128 ? 128 : 256));

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRouterStages; ++s) {
            mbar_init(&sm->full[s], 1);
            mbar_init(&sm->empty[s], 1);
        }
        mbar_init(&sm->acc_full, 1);
        mbar_init(&sm->drain, 1);
        sm->abort_flag = 0;
        fence_barrier_init();
        prefetch_tensor_map(&tm_x);
        prefetch_tensor_map(&tm_router);
        if (a.gamma_col >= 0) prefetch_tensor_map(&tm_gate);
    }
    if (warp == 0) {
        tmem_alloc(&sm->tmem_base, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm->tmem_base;
    volatile int *abort_flag = &sm->abort_flag;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            const uint32_t tx = kATileBytes + a.E * 128 + (a.gamma_col >= 0 ? 8 * 128 : 0);
            int kc = 0;
            for (; kc < nk; ++kc) {
                const int s = kc % kRouterStages;
                const uint32_t use = kc / kRouterStages;
                if (use > 0 && !mbar_wait(&sm->empty[s], (use - 1) & 1, abort_flag)) {
                    record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                uint8_t *st = tiles + s * stage_bytes;
                mbar_arrive_expect_tx(&sm->full[s], tx);
                tma_load_2d(st, &tm_x, &sm->full[s], kc * kBlockK, static_cast<int>(n0));
                tma_load_2d(st + kATileBytes, &tm_router, &sm->full[s], kc * kBlockK, 0);
                if (a.gamma_col >= 0)
                    tma_load_2d(st + kATileBytes + a.gamma_col * 128, &tm_gate, &sm->full[s],
                                kc * kBlockK, 0);
            }
            // drain: wait for the last load issued to every stage
            for (int i = (kc > kRouterStages ? kc - kRouterStages : 0); i < kc; ++i)
                mbar_wait(&sm->full[i % kRouterStages], (i / kRouterStages) & 1, abort_flag);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kBlockM, a.e_pad);
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % kRouterStages;
                if (!mbar_wait(&sm->full[s], (kc / kRouterStages) & 1, abort_flag)) {
                    record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after_sync();
                const uint8_t *st = tiles + s * stage_bytes;
                const uint64_t da = sw128_kmajor_desc(smem_addr(st));
                const uint64_t db = sw128_kmajor_desc(smem_addr(st + kATileBytes));
#pragma unroll
                for (int kk = 0; kk < kBlockK / 16; ++kk)
                    mma_bf16(tmem, da + 2 * kk, db + 2 * kk, idesc, (kc | kk) != 0);
                mma_commit(&sm->empty[s]);
            }
            mma_commit(&sm->acc_full);
            mma_commit(&sm->drain);
            mbar_wait(&sm->drain, 0, abort_flag);
        }
        __syncwarp();
    }

    // ---------------- epilogue: every thread owns one token row (TMEM lane)
    const bool ok = mbar_wait(&sm->acc_full, 0, abort_flag);
    __syncwarp();
    if (!ok) {
        record_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
    } else {
        tc_fence_after_sync();
        const int row = warp * 32 + lane;
        const int64_t n = n0 + row;
        const bool live = n < a.N;
        const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const int nchunk = (a.E + 31) / 32;

        float mx = -INFINITY;
        for (int c = 0; c < nchunk; ++c) {
            float v[32];
            tmem_load32(trow + c * 32, v);
            tmem_load_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (c * 32 + i < a.E) mx = fmaxf(mx, finite_or_neg_inf(v[i]));
        }
        float den = 0.f;
        for (int c = 0; c < nchunk; ++c) {
            float v[32];
            tmem_load32(trow + c * 32, v);
            tmem_load_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (c * 32 + i < a.E) den += expf(finite_or_neg_inf(v[i]) - mx);
        }
        // top-k: round j takes the largest (logit, lower index first) key that
        // comes strictly after the key taken in round j-1.  exp is monotone,
        // so this is the top-k of the probabilities.
        float prev_v = INFINITY;
        int prev_i = -1;
        float wsum = 0.f;
        float *w_row = a.topk_w + n * a.k;
        int32_t *id_row = a.topk_ids + n * a.k;
        for (int j = 0; j < a.k; ++j) {
            float best_v = -INFINITY;
            int best_i = -1;
            for (int c = 0; c < nchunk; ++c) {
                float v[32];
                tmem_load32(trow + c * 32, v);
                tmem_load_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int e = c * 32 + i;
                    const float x = finite_or_neg_inf(v[i]);
                    const bool after_prev = (x < prev_v) || (x == prev_v && e > prev_i);
                    if (e < a.E && after_prev && (best_i < 0 || x > best_v)) {
                        best_v = x;
                        best_i = e;
                    }
                }
            }
            const float p = expf(best_v - mx) / den;
            wsum += p;
            if (live) {
                w_row[j] = p;
                id_row[j] = best_i;
            }
            prev_v = best_v;
            prev_i = best_i;
        }
        if (live) {
            const float inv = a.norm ? 1.f / wsum : 1.f;
            for (int j = 0; j < a.k; ++j) {
                const float w = a.norm ? w_row[j] * inv : w_row[j];
                if (a.norm) w_row[j] = w;
                if (a.topk_w_bf16) {
                    __nv_bfloat16 h = __float2bfloat16_rn(w);
                    a.topk_w_bf16[n * a.k + j] = *reinterpret_cast<uint16_t *>(&h);
                }
            }
        }
        if (a.gamma_col >= 0) {
            const float lg = tmem_load1(trow + a.gamma_col);
            tmem_load_wait();
            if (live) a.gamma[n] = 1.f / (1.f + expf(-lg));
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, tmem_cols);
    }
}

}  // namespace

size_t router_smem_bytes(int e_pad) {
    return 1024 + static_cast<size_t>(kRouterStages) * (kATileBytes + e_pad * 128) +
           sizeof(RouterSmem);
}

cudaError_t launch_router(const CUtensorMap &tm_x, const CUtensorMap &tm_router,
                          const CUtensorMap &tm_gate, const RouterArgs &a, cudaStream_t s) {
    const size_t smem = router_smem_bytes(a.e_pad);
    cudaError_t err = cudaFuncSetAttribute(router_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const unsigned grid = static_cast<unsigned>((a.N + kBlockM - 1) / kBlockM);
    router_kernel<<<grid, kRouterThreads, smem, s>>>(tm_x, tm_router, tm_gate, a);
    return cudaGetLastError();
}

}  // namespace moe
