/*
 * moe.h -- C ABI of the GB300 (sm_103a) sparse MoE FFN layer library
 * (libsparse_moe_ffn.so).
 *
 * The layer is the one defined on the page "M03 · Sparse MoE: routing,
 * per-expert grouped compute, shared expert" (nano-vllm-omni drills), problem
 * overview:
 *
 *   logits = x @ router^T                     [N, E]
 *   probs  = softmax(logits) over all E (fp32)
 *   w, ids = topk(probs, k)                   descending
 *   if norm_topk_prob: w = w / sum(w)
 *   out[n] = sum_j w[n,j] * Expert_{ids[n,j]}(x[n]),
 *   Expert(h) = (silu(h Wg^T) * (h Wu^T)) Wd^T
 *   talker only: out += sigmoid(x @ g^T) * SharedMLP(x)   (scalar gate per token)
 *
 * computed the "serving way" of that page: the N*k (token, slot) pairs are
 * grouped by expert (stable order, counts, prefix offsets, padded to the GEMM
 * block as FusedMoE's moe_align_block_size does), each expert runs one
 * grouped SwiGLU over its gathered tokens, and the weighted results are
 * accumulated back to every token.
 *
 * Conventions shared by every entry point
 *   - All tensors are dense, row-major, on the current CUDA device, unless a
 *     parameter says "host".  bf16 data is passed as moe_bf16_t (the raw
 *     IEEE bfloat16 bit pattern), fp16 data as moe_f16_t (IEEE binary16).
 *     Pointers to bf16 / fp16 matrices must be 16-byte aligned; H and I must
 *     be multiples of 8 (16-byte rows for TMA).
 *   - Every weight is taken in the model's bf16, as the pages define the
 *     layer.  Each entry point that takes down-projection weights also has a
 *     *_prepared twin taking an fp16 copy of them instead (w_down_f16,
 *     shared_down_proj_f16), made once at load by moe_convert_bf16_to_f16:
 *     every bf16 value of magnitude 2^-14 or more converts exactly (fp16 has
 *     more significand bits), smaller ones round to fp16's subnormal grid
 *     (absolute error <= 2^-25).  With bf16 down weights the gate/up
 *     activation is kept as a bf16 pair hi + lo and the down GEMM issues two
 *     MMAs per K step; with the fp16 copy it is kept in fp16 and one MMA per
 *     K step suffices, which halves the down GEMM's tensor work.
 *   - The caller owns every buffer, including the workspace.  The library
 *     never allocates, frees or synchronises (except moe_read_device_status),
 *     and keeps no state between calls: calls on different streams with
 *     different workspaces may run concurrently.
 *   - Work is enqueued asynchronously on `stream`.  A call returns MOE_OK once
 *     its kernels are enqueued; device-side failures (a bounded wait that ran
 *     out, an out-of-range expert id given to moe_align) are recorded in the
 *     workspace's status word and read with moe_read_device_status.
 *   - Argument errors return at once and enqueue nothing.  N = 0 is a no-op
 *     that returns MOE_OK.
 *   - Routing ties (equal probabilities) go to the lower expert index; slot j
 *     of a token holds its j-th largest probability.
 */
#ifndef SPARSE_MOE_FFN_MOE_H
#define SPARSE_MOE_FFN_MOE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* IEEE bfloat16 bit pattern. */
typedef uint16_t moe_bf16_t;
/* IEEE binary16 (fp16) bit pattern. */
typedef uint16_t moe_f16_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,          /* null pointer, bad size, k > E, misalignment */
    MOE_ERR_WORKSPACE_TOO_SMALL = 2,  /* workspace_bytes below the *_workspace_bytes value */
    MOE_ERR_UNSUPPORTED = 3,          /* valid but outside the library's limits (E > 256 ...) */
    MOE_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed */
    MOE_ERR_DEVICE_CHECK = 5,         /* a kernel found a bad value (e.g. expert id >= E) */
    MOE_ERR_DEVICE_TIMEOUT = 6        /* a kernel's bounded wait ran out; it stopped early */
} moe_status_t;

/* GEMM row block used by moe_forward: every expert segment is padded to it. */
#define MOE_BLOCK_M 128
/* Largest expert count the fused router supports (its MMA tile is <= 256 wide). */
#define MOE_MAX_EXPERTS 256

/* Static description of a status code.  Never NULL. */
const char *moe_status_string(moe_status_t status);

/* Detail of the last error returned on the calling thread ("" if none). */
const char *moe_last_error(void);

/* -------------------------------------------------------------------------
 * moe_route -- the routing block of the M03 problem overview (logits, fp32
 * softmax over all E experts, top-k, optional norm_topk_prob renorm), plus
 * the talker's scalar shared-expert gate sigmoid(x . g).  Also the router of
 * the Nano-vLLM notes' Qwen3MoeSparseMoeBlock (softmax in fp32, topk, renorm).
 *
 *   x            [N, H] bf16
 *   router       [E, H] bf16
 *   shared_gate  [1, H] bf16 or NULL
 *   topk_w       [N, k] fp32 out: routing weights (renormalised iff
 *                norm_topk_prob != 0)
 *   topk_ids     [N, k] int32 out: expert ids, slot 0 = largest probability
 *   topk_w_bf16  [N, k] bf16 out or NULL: topk_w rounded to nearest even
 *                (the pages return weights in x's dtype)
 *   shared_gamma [N]    fp32 out: sigmoid(x . g); required iff shared_gate
 *   workspace    >= moe_route_workspace_bytes() bytes, or NULL (then device
 *                failures are not recorded)
 * Limits: 1 <= k <= E <= 256 (E <= 248 with a shared gate), H % 8 == 0.
 * ---------------------------------------------------------------------- */
size_t moe_route_workspace_bytes(void);
moe_status_t moe_route(const moe_bf16_t *x, const moe_bf16_t *router,
                       const moe_bf16_t *shared_gate, int64_t N, int H, int E,
                       int k, int norm_topk_prob, float *topk_w,
                       int32_t *topk_ids, moe_bf16_t *topk_w_bf16,
                       float *shared_gamma, void *workspace,
                       size_t workspace_bytes, cudaStream_t stream);

/* -------------------------------------------------------------------------
 * moe_align -- the grouping bookkeeping of the M03 walk-through (flatten the
 * pairs p = n*k + j row-major, stable sort by expert, per-expert counts,
 * prefix-sum segment starts), padded to block_m rows per expert segment as
 * FusedMoE's moe_align_block_size (named in the M03 shape-trace section).
 *
 *   topk_ids     [N, k] int32 in, each in [0, E)
 *   sorted_pair  [cap] int32 out, cap = moe_align_capacity(N, k, E, block_m):
 *                expert e's pairs in ascending p start at
 *                pad_off[e] = sum_{e'<e} round_up(counts[e'], block_m), followed
 *                by the sentinel N*k up to the next multiple of block_m.
 *                Slots >= *num_padded are left unspecified.
 *   block_expert [cap / block_m] int32 out: owner expert of each row block
 *                (entries >= *num_padded / block_m unspecified)
 *   counts       [E] int32 out: pairs per expert (sum = N*k)
 *   offsets      [E+1] int32 out: exclusive prefix sum of counts
 *   num_padded   [1] int32 out: pad_off[E]
 *   workspace    >= moe_align_workspace_bytes(...) bytes (scratch + status)
 * An id outside [0, E) is skipped and records MOE_ERR_DEVICE_CHECK.
 * Limits: 1 <= E <= 1024, 1 <= block_m <= 1024, N*k + E*block_m < 2^31.
 * ---------------------------------------------------------------------- */
int64_t moe_align_capacity(int64_t N, int k, int E, int block_m);
size_t moe_align_workspace_bytes(int64_t N, int k, int E, int block_m);
moe_status_t moe_align(const int32_t *topk_ids, int64_t N, int k, int E,
                       int block_m, int32_t *sorted_pair, int32_t *block_expert,
                       int32_t *counts, int32_t *offsets, int32_t *num_padded,
                       void *workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* -------------------------------------------------------------------------
 * moe_align_noalloc -- moe_align without a caller-provided workspace, for
 * callers that cannot allocate device memory (no counterpart on the pages:
 * it exists for integration, not for the method).  Code being captured into
 * a CUDA graph may not call cudaMalloc, plugin-style hosts give a kernel
 * only its input and output buffers, and latency-critical paths must avoid an
 * allocator's locks and implicit synchronisation; such callers pass only
 * topk_ids and the outputs of moe_align.
 *
 * The scratch lives in a static device array of
 * MOE_ALIGN_NOALLOC_SCRATCH_BYTES (1 MiB) that every GPU loading the library
 * holds until exit.  Sizes whose moe_align_workspace_bytes(N, k, E, block_m)
 * exceed it return MOE_ERR_UNSUPPORTED (for E = 128 that is above ~4M pairs).
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current): make that first call
 * before any stream capture.  The address is kept per device and CUDA
 * context; a call made under a new context (after cudaDeviceReset, say)
 * looks it up again, so that call too belongs before any capture.  Every
 * call shares the array, so calls whose work overlaps on the GPU (other
 * streams, other host threads) race; the array needs no clearing between
 * calls.  device_status (nullable, int32 on the device) receives the call's
 * status word (MOE_ERR_DEVICE_CHECK for an id outside [0, E); 0 for N = 0)
 * by an asynchronous copy or memset on `stream`.
 * Arguments and outputs are those of moe_align.  Allocates nothing.
 * ---------------------------------------------------------------------- */
#define MOE_ALIGN_NOALLOC_SCRATCH_BYTES (1u << 20)
moe_status_t moe_align_noalloc(const int32_t *topk_ids, int64_t N, int k, int E,
                               int block_m, int32_t *sorted_pair,
                               int32_t *block_expert, int32_t *counts,
                               int32_t *offsets, int32_t *num_padded,
                               int32_t *device_status, cudaStream_t stream);

/* -------------------------------------------------------------------------
 * moe_forward -- the whole layer (M03 problem overview and its "serving way";
 * the shared expert of the same page and of the talker MoE block in the
 * vLLM Qwen3.5 walkthrough, section "2.5B Sparse MoE").
 *
 *   x                 [N, H] bf16
 *   router            [E, H] bf16
 *   w_gate, w_up      [E, I, H] bf16
 *   w_down            [E, H, I] bf16
 *   shared_gate_proj  [I_s, H] bf16 \
 *   shared_up_proj    [I_s, H] bf16  | all four NULL: no shared expert
 *   shared_down_proj  [H, I_s] bf16  | (I_s ignored); all four set: shared
 *   shared_gate       [1, H]   bf16 /  expert with I_s >= 8, I_s % 8 == 0
 *   out               [N, H] bf16 out (may not alias any input)
 *   workspace         >= moe_forward_workspace_bytes(...) bytes, 256-byte
 *                     aligned; holds the routing, grouping and intermediate
 *                     activations (layout: moe_forward_layout)
 * Precision: bf16 inputs, fp32 routing and accumulation; the gate/up
 * activation a = silu(g)*u is kept as the bf16 pair hi = bf16(a),
 * lo = bf16(a - hi) (16 significant bits) and both halves are multiplied by
 * the bf16 down weights; each pair's weighted down projection is
 * accumulated in fp32 and kept as a pair row (see "Pair rows" below: 16
 * significant bits in 3 bytes); the k contributions are summed in fp32 in
 * slot order, and out is rounded to bf16 once.
 * The shared expert runs in the same grouped GEMMs as C = ceil(I_s / I)
 * virtual experts of I intermediate rows each (see moe_forward_layout_t):
 * gamma * SharedMLP(x) arrives as C partial sums over disjoint intermediate
 * rows, each a pair row with weight gamma, added after the k routed slots.
 * A non-finite activation or pair output records MOE_ERR_DEVICE_CHECK.
 * The result does not depend on the other tokens of the batch and is
 * bitwise reproducible.
 * Limits: as moe_route, plus I % 8 == 0, E + C <= 256 and
 * N*(k + C) + (E + C)*128 < 2^30 (C = 0 without the shared expert).
 * ---------------------------------------------------------------------- */
size_t moe_forward_workspace_bytes(int64_t N, int H, int E, int I, int k, int I_s);
moe_status_t moe_forward(const moe_bf16_t *x, const moe_bf16_t *router,
                         const moe_bf16_t *w_gate, const moe_bf16_t *w_up,
                         const moe_bf16_t *w_down,
                         const moe_bf16_t *shared_gate_proj,
                         const moe_bf16_t *shared_up_proj,
                         const moe_bf16_t *shared_down_proj,
                         const moe_bf16_t *shared_gate, int64_t N, int H, int E,
                         int I, int I_s, int k, int norm_topk_prob,
                         moe_bf16_t *out, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/* -------------------------------------------------------------------------
 * moe_forward_prepared -- moe_forward with the down projections given as the
 * fp16 copies moe_convert_bf16_to_f16 makes once at load (w_down_f16
 * [E, H, I], shared_down_proj_f16 [H, I_s]; a load-time preparation the pages
 * do not have).  The activation is then kept in fp16 (11 significant bits)
 * and multiplied by the fp16 weights with one MMA per K step instead of two,
 * which halves the down GEMM's tensor work at large N.  Everything else --
 * arguments, workspace, routing, pair rows, slot-order fp32 combine,
 * limits, errors -- is moe_forward's.  The outputs differ from moe_forward's
 * by the activation's rounding (both stay within the layer's tolerance).
 * ---------------------------------------------------------------------- */
moe_status_t moe_forward_prepared(const moe_bf16_t *x, const moe_bf16_t *router,
                                  const moe_bf16_t *w_gate, const moe_bf16_t *w_up,
                                  const moe_f16_t *w_down_f16,
                                  const moe_bf16_t *shared_gate_proj,
                                  const moe_bf16_t *shared_up_proj,
                                  const moe_f16_t *shared_down_proj_f16,
                                  const moe_bf16_t *shared_gate, int64_t N, int H,
                                  int E, int I, int I_s, int k, int norm_topk_prob,
                                  moe_bf16_t *out, void *workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/* -------------------------------------------------------------------------
 * Pair rows -- how the weighted per-pair outputs v = w * Expert(x) are held
 * between the down projection and the combine (moe_experts writes them,
 * moe_combine reads them; the pages have no counterpart).  Two planes of
 * the same [rows, H] shape: hi = bf16(v) (round to nearest even) and an
 * int8 residual r.  With f the 8-bit exponent field of hi (as an IEEE
 * float), clamped to f >= 16:
 *     r = clamp(round_even((v - hi) * 2^(142 - f)), -127, 127)
 *     v' = hi + r * 2^(f - 142)
 * so |v' - v| <= 2^-16 |v| (or <= 2^-127 for |v| < 2^-111).
 * ---------------------------------------------------------------------- */

/* -------------------------------------------------------------------------
 * moe_experts -- the per-expert half of the layer for rows whose expert and
 * weight are already chosen: the receiving side of expert-parallel dispatch
 * (M03 drill, level-3 follow-up on splitting experts across devices: the
 * (token, expert) table drives an all-to-all).  For every row r:
 *   y[r] = weights[r] * Expert_{ids[r]}(x_rows[r])   (as pair rows)
 * with the arithmetic of moe_forward's per-pair outputs (grouping by expert,
 * gate/up with the hi/lo activation, down), so the bits equal the pair rows
 * moe_forward produces for the same (row, expert, weight);
 * moe_experts_prepared does the same with fp16 down weights and equals
 * moe_forward_prepared's pair rows.
 *   x_rows   [R, H] bf16      ids [R] int32 in [0, E)      weights [R] fp32
 *   w_gate, w_up [E, I, H] bf16, w_down [E, H, I] bf16 (w_down_f16: fp16):
 *            the experts this call serves (a rank's slice of the layer's
 *            experts)
 *   y_hi     [R, H] bf16 out, y_res [R, H] int8 out: the pair rows of y
 *            (both 16-byte aligned)
 *   workspace >= moe_experts_workspace_bytes(R, H, E, I) bytes, 256-byte
 *            aligned; its first 4 bytes are the status word
 *            (moe_read_device_status)
 * Errors: argument problems before anything is enqueued; ids outside [0, E)
 * record MOE_ERR_DEVICE_CHECK (their rows are left unwritten).
 * ---------------------------------------------------------------------- */
size_t moe_experts_workspace_bytes(int64_t R, int H, int E, int I);
moe_status_t moe_experts(const moe_bf16_t *x_rows, const int32_t *ids,
                         const float *weights, int64_t R, int H, int E, int I,
                         const moe_bf16_t *w_gate, const moe_bf16_t *w_up,
                         const moe_bf16_t *w_down, moe_bf16_t *y_hi, int8_t *y_res,
                         void *workspace, size_t workspace_bytes, cudaStream_t stream);
moe_status_t moe_experts_prepared(const moe_bf16_t *x_rows, const int32_t *ids,
                                  const float *weights, int64_t R, int H, int E,
                                  int I, const moe_bf16_t *w_gate,
                                  const moe_bf16_t *w_up, const moe_f16_t *w_down_f16,
                                  moe_bf16_t *y_hi, int8_t *y_res, void *workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/* -------------------------------------------------------------------------
 * moe_shared_expert -- the gated shared expert of the talker layer on its own
 * (vLLM Qwen3.5 walkthrough, "2.5B Sparse MoE": gamma * SharedMLP(x) with
 * gamma = sigmoid(x . g)), computed exactly as moe_forward computes it: its
 * I_s intermediate rows cut into C = moe_shared_chunks(I, I_s) = ceil(I_s / I)
 * chunks of I rows (I: the routed experts' intermediate size; the last chunk
 * padded with zero weights), chunk c a virtual expert with weight gamma.
 * For every token n and chunk c (row n*C + c of y):
 *   y[n*C + c] = gamma[n] * Wd[:, chunk c] (silu(Wg[chunk c] x) * (Wu[chunk c] x))
 * as pair rows, bit for bit the rows moe_forward holds in slots k .. k+C-1;
 * moe_combine / moe_combine_indexed add them with shared_slots = C.  This is
 * the expert-parallel layer's local shared term (it needs no exchange).
 *   x [N, H] bf16; shared_gamma [N] fp32 (moe_route's output)
 *   shared_gate_proj, shared_up_proj [I_s, H] bf16; shared_down_proj [H, I_s]
 *     bf16 (moe_shared_expert_prepared: its fp16 copy, as in
 *     moe_forward_prepared)
 *   y_hi [N*C, H] bf16 out, y_res [N*C, H] int8 out (16-byte aligned)
 *   workspace >= moe_shared_expert_workspace_bytes(N, H, I, I_s) bytes,
 *     256-byte aligned; its first 4 bytes are the status word
 * Limits: H, I, I_s positive multiples of 8, C <= 256, N*C + C*128 < 2^30.
 * ---------------------------------------------------------------------- */
int moe_shared_chunks(int I, int I_s);
size_t moe_shared_expert_workspace_bytes(int64_t N, int H, int I, int I_s);
moe_status_t moe_shared_expert(const moe_bf16_t *x, const float *shared_gamma,
                               int64_t N, int H, int I, int I_s,
                               const moe_bf16_t *shared_gate_proj,
                               const moe_bf16_t *shared_up_proj,
                               const moe_bf16_t *shared_down_proj, moe_bf16_t *y_hi,
                               int8_t *y_res, void *workspace, size_t workspace_bytes,
                               cudaStream_t stream);
moe_status_t moe_shared_expert_prepared(const moe_bf16_t *x, const float *shared_gamma,
                                        int64_t N, int H, int I, int I_s,
                                        const moe_bf16_t *shared_gate_proj,
                                        const moe_bf16_t *shared_up_proj,
                                        const moe_f16_t *shared_down_proj_f16,
                                        moe_bf16_t *y_hi, int8_t *y_res,
                                        void *workspace, size_t workspace_bytes,
                                        cudaStream_t stream);

/* -------------------------------------------------------------------------
 * moe_combine -- the weighted accumulation of the layer (M03 drill: each
 * token's outputs summed back, index_add_ in the pages' PyTorch form), done
 * without atomics:
 *   out[n] = bf16(sum_{j<k} ypair[n*k + j] + sum_{c<S} yshared[n*S + c]),
 * the pair rows decoded and summed in fp32 in slot order, then the shared
 * expert's S = shared_slots chunk rows in chunk order.  ypair: pair rows
 * [N*k, H] (ypair_hi bf16, ypair_res int8); yshared: pair rows [N*S, H]
 * (moe_shared_expert's output, S = moe_shared_chunks(I, I_s)) with
 * 1 <= S <= 256, or both planes NULL (shared_slots ignored); out [N, H]
 * bf16; every plane 16-byte aligned (with 32-byte aligned planes and
 * H % 16 == 0, large batches read 32 bytes at a time; every form adds the
 * same values in the same order).  moe_forward ends with the same kernels,
 * its k + C slots per token all in ypair.
 * ---------------------------------------------------------------------- */
moe_status_t moe_combine(const moe_bf16_t *ypair_hi, const int8_t *ypair_res,
                         const moe_bf16_t *yshared_hi, const int8_t *yshared_res,
                         int shared_slots, int64_t N, int H, int k, moe_bf16_t *out,
                         cudaStream_t stream);

/* moe_combine over pair rows held in another order: pair p = n*k + j reads
 * row row_index[p] of yrows ([num_rows, H] pair rows; the order in which
 * expert-parallel results come back, moe_ep_dispatch's inv_order).  An index
 * outside [0, num_rows) (a pair that was never sent) contributes nothing.
 * row_index: [N*k] int32 on the device. */
moe_status_t moe_combine_indexed(const moe_bf16_t *yrows_hi, const int8_t *yrows_res,
                                 int64_t num_rows, const int32_t *row_index,
                                 const moe_bf16_t *yshared_hi, const int8_t *yshared_res,
                                 int shared_slots, int64_t N, int H, int k,
                                 moe_bf16_t *out, cudaStream_t stream);

/* -------------------------------------------------------------------------
 * moe_ep_dispatch -- the sending side of expert-parallel dispatch (M03 drill,
 * level-3 follow-up: the (token, expert) table drives an all-to-all), on the
 * device.  The layer's E experts are split over `world` ranks, rank r owning
 * [r*E_r, (r+1)*E_r) with E_r = ceil(E / world).  For this rank's routed
 * tokens:
 *   send_counts [world] int32 out: pairs whose expert rank r owns
 *   send rows i = 0 .. N*k-1 (those with a valid id) in rank order, pairs
 *     in ascending p = n*k + j within a rank:
 *     send_x   [N*k, H] bf16 out: x[p / k]
 *     send_ids [N*k] int32 out: the expert id local to its rank, id - r*E_r
 *     send_w   [N*k] fp32 out: topk_w[p]
 *   inv_order [N*k] int32 out: the send row of pair p (-1 for an id outside
 *     [0, E), which is also recorded as MOE_ERR_DEVICE_CHECK), i.e. the row
 *     index moe_combine_indexed takes once the results come back in send
 *     order
 *   x [N, H] bf16, topk_ids / topk_w [N, k] (moe_route's outputs)
 *   workspace >= moe_ep_dispatch_workspace_bytes(N, k, world), 256-byte
 *     aligned; its first 4 bytes are the status word
 * The grouping is moe_align's, with `world` groups and blocks of one row.
 * Limits: 1 <= world <= 1024, N*k < 2^30.
 * ---------------------------------------------------------------------- */
size_t moe_ep_dispatch_workspace_bytes(int64_t N, int k, int world);
moe_status_t moe_ep_dispatch(const moe_bf16_t *x, const int32_t *topk_ids,
                             const float *topk_w, int64_t N, int H, int k, int E,
                             int world, moe_bf16_t *send_x, int32_t *send_ids,
                             float *send_w, int32_t *send_counts, int32_t *inv_order,
                             void *workspace, size_t workspace_bytes,
                             cudaStream_t stream);

/* -------------------------------------------------------------------------
 * moe_convert_bf16_to_f16 -- the load-time step that makes the fp16 down
 * weights the *_prepared entry points take: dst[i] = fp16(src[i]) for i < n, round to
 * nearest even (exact for |src| >= 2^-14 and for zero; below, the nearest
 * fp16 subnormal).  src, dst: device, 16-byte aligned, not overlapping.
 * device_status (nullable, int32 on the device) is set to
 * MOE_ERR_DEVICE_CHECK if some |src[i]| exceeds fp16's range (65504; such
 * a value becomes infinity) or is NaN; it is left untouched otherwise.
 * ---------------------------------------------------------------------- */
moe_status_t moe_convert_bf16_to_f16(const moe_bf16_t *src, moe_f16_t *dst, int64_t n,
                                     int32_t *device_status, cudaStream_t stream);

/* -------------------------------------------------------------------------
 * moe_forward_host -- moe_forward for activations that live in host memory:
 * the end-to-end call of a loop whose tokens come from the host (the pages
 * have no counterpart; their layer works on device tensors).  Enqueued on
 * `stream`: copy x_host -> x_dev, the layer x_dev -> out_dev, copy out_dev ->
 * out_host.  The result is in out_host once the stream reaches that point.
 * Pinned host buffers mapped into the device's address space (and 16-byte
 * aligned) are copied by kernels on all SMs; other host memory by
 * cudaMemcpyAsync.
 *   x_host, out_host  [N, H] bf16 host memory (pinned for asynchronous copies;
 *                     pageable memory makes the copies synchronous)
 *   x_dev, out_dev    [N, H] bf16 device buffers owned by the caller, 16-byte
 *                     aligned, aliasing no input
 * Every other argument, limit and error as moe_forward (with x_dev as x and
 * out_dev as out); all argument errors are returned before anything is
 * enqueued, plus MOE_ERR_INVALID_ARG for a null host pointer with N > 0.
 * ---------------------------------------------------------------------- */
moe_status_t moe_forward_host(const moe_bf16_t *x_host, moe_bf16_t *out_host,
                              moe_bf16_t *x_dev, moe_bf16_t *out_dev,
                              const moe_bf16_t *router, const moe_bf16_t *w_gate,
                              const moe_bf16_t *w_up, const moe_bf16_t *w_down,
                              const moe_bf16_t *shared_gate_proj,
                              const moe_bf16_t *shared_up_proj,
                              const moe_bf16_t *shared_down_proj,
                              const moe_bf16_t *shared_gate, int64_t N, int H, int E,
                              int I, int I_s, int k, int norm_topk_prob,
                              void *workspace, size_t workspace_bytes,
                              cudaStream_t stream);
/* moe_forward_host with fp16 down weights: the layer step is
 * moe_forward_prepared. */
moe_status_t moe_forward_host_prepared(
    const moe_bf16_t *x_host, moe_bf16_t *out_host, moe_bf16_t *x_dev,
    moe_bf16_t *out_dev, const moe_bf16_t *router, const moe_bf16_t *w_gate,
    const moe_bf16_t *w_up, const moe_f16_t *w_down_f16,
    const moe_bf16_t *shared_gate_proj, const moe_bf16_t *shared_up_proj,
    const moe_f16_t *shared_down_proj_f16, const moe_bf16_t *shared_gate, int64_t N,
    int H, int E, int I, int I_s, int k, int norm_topk_prob, void *workspace,
    size_t workspace_bytes, cudaStream_t stream);

/* -------------------------------------------------------------------------
 * moe_add_rmsnorm -- the decoder layer's step that feeds the MoE, in one
 * kernel (Nano-vLLM notes, question 4 on the decoder layer; Qwen3.5
 * walkthrough section 2.1): r = x + residual in the model's bf16 dtype;
 * residual = r; normed = r / sqrt(mean(r^2) + eps) * weight, or
 * * (1 + weight) when gemma != 0 (GemmaRMSNorm).
 *
 *   x        [N, H] bf16 in (the sub-layer's output)
 *   residual [N, H] bf16 in/out (becomes r)
 *   weight   [H]    bf16
 *   normed   [N, H] bf16 out (the MoE's input x; may not alias x or residual)
 * Precision: the sum of squares in fp32, one bf16 rounding of normed; the
 * residual equals bf16(x + residual) bit for bit.  Limits: H % 8 == 0.
 * ---------------------------------------------------------------------- */
moe_status_t moe_add_rmsnorm(const moe_bf16_t *x, moe_bf16_t *residual,
                             const moe_bf16_t *weight, int64_t N, int H,
                             float eps, int gemma, moe_bf16_t *normed,
                             cudaStream_t stream);

/* -------------------------------------------------------------------------
 * moe_dense_mlp -- the dense SwiGLU MLP of the non-MoE layers (Qwen3MLP of
 * the Nano-vLLM notes, used for mlp_only_layers; section 2.5A of the
 * Qwen3.5 walkthrough): out = (silu(x Wg^T) * (x Wu^T)) Wd^T, the layer with
 * E = k = 1, run on the same grouped GEMM kernels as one dense group.
 *
 *   x [N, H], w_gate / w_up [I, H], w_down [H, I], out [N, H]: bf16
 *   (moe_dense_mlp_prepared: w_down_f16 [H, I] fp16)
 *   workspace >= moe_dense_mlp_workspace_bytes(N, H, I), 256-byte aligned
 * Precision as moe_forward (moe_forward_prepared).  Limits: H % 8 == 0,
 * I % 8 == 0, N < 2^30.
 * ---------------------------------------------------------------------- */
size_t moe_dense_mlp_workspace_bytes(int64_t N, int H, int I);
moe_status_t moe_dense_mlp(const moe_bf16_t *x, const moe_bf16_t *w_gate,
                           const moe_bf16_t *w_up, const moe_bf16_t *w_down,
                           int64_t N, int H, int I, moe_bf16_t *out,
                           void *workspace, size_t workspace_bytes,
                           cudaStream_t stream);
moe_status_t moe_dense_mlp_prepared(const moe_bf16_t *x, const moe_bf16_t *w_gate,
                                    const moe_bf16_t *w_up, const moe_f16_t *w_down_f16,
                                    int64_t N, int H, int I, moe_bf16_t *out,
                                    void *workspace, size_t workspace_bytes,
                                    cudaStream_t stream);

/* Byte offsets of moe_forward's workspace sub-buffers (for inspecting the
 * intermediate results; every offset is 256-byte aligned).
 *
 * With the shared expert (I_s > 0) the layer runs it inside the grouped
 * GEMMs: its intermediate rows are cut into C = ceil(I_s / I) chunks of I
 * rows (the last one padded with zero weights), and chunk c is a virtual
 * expert E + c that every token uses with weight gamma = sigmoid(x . g).
 * Every token then has `slots` = k + C (expert, weight) slots, the routed
 * ones first, grouped over `groups` = E + C experts; the sizes below that
 * name k and E mean `slots` and `groups`. */
typedef struct {
    size_t status;        /* int32 device status word (a moe_status_t)       */
    size_t topk_w;        /* fp32 [N, slots]: routed weights, then gamma      */
    size_t topk_ids;      /* int32 [N, slots]: routed experts, then E + c     */
    size_t gamma;         /* fp32 [N] (shared expert only)                    */
    size_t counts;        /* int32 [groups]                                   */
    size_t offsets;       /* int32 [groups+1]                                 */
    size_t pad_offsets;   /* int32 [groups+1]                                 */
    size_t num_padded;    /* int32 [1]                                        */
    size_t align_scratch; /* int32 [chunks, groups]                           */
    size_t sorted_pair;   /* int32 [capacity]                                 */
    size_t block_expert;  /* int32 [capacity / 128]                           */
    size_t ready;         /* int32 [max(groups, capacity/128)] GEMM hand-off counts */
    size_t x_sorted;      /* bf16 [capacity, H]   x rows in expert order (dense blocks) */
    size_t act;           /* a = silu(x Wg^T) * (x Wu^T): bf16 hi [capacity, I]
                             then bf16 lo [capacity, I] (moe_forward), or fp16
                             [capacity, I] (moe_forward_prepared)           */
    size_t ypair;         /* bf16 [N*slots, H]  w * Expert(x) per slot: hi plane */
    size_t ypair_res;     /* int8 [N*slots, H]  ... residual plane (pair rows)   */
    size_t total;         /* = moe_forward_workspace_bytes                    */
    int64_t capacity;     /* moe_align_capacity(N, slots, groups, 128)        */
    int slots;            /* k + C (k without the shared expert)              */
    int groups;           /* E + C (E without the shared expert)              */
} moe_forward_layout_t;

moe_status_t moe_forward_layout(int64_t N, int H, int E, int I, int k, int I_s,
                                moe_forward_layout_t *layout);

/* Waits for `stream`, then returns the status word kept in `workspace` by the
 * last moe_route / moe_align / moe_forward call that used it (MOE_OK if no
 * kernel recorded a failure).  The only synchronising entry point. */
moe_status_t moe_read_device_status(const void *workspace, cudaStream_t stream);

/* Failure-detection self-check (not part of the layer; the pages have no
 * counterpart).  Enqueues a one-thread kernel that waits on a device barrier
 * nothing ever completes and then on a hand-off counter nothing ever
 * increments, through the same bounded waits the layer's kernels use, each
 * giving up after limit_ns (0 < limit_ns <= 10 s).  The status word at
 * the start of `workspace` (>= 4 bytes) then reads MOE_ERR_DEVICE_TIMEOUT and
 * the CUDA context stays usable. */
moe_status_t moe_selftest_wait_timeout(void *workspace, size_t workspace_bytes,
                                       uint64_t limit_ns, cudaStream_t stream);

/* -------------------------------------------------------------------------
 * Instrumentation
 * ---------------------------------------------------------------------- */

/* Stages of moe_forward, in launch order. */
enum {
    MOE_STAGE_ROUTE = 0,
    MOE_STAGE_ALIGN = 1,   /* empty when routing groups the pairs itself (N <= 128,
                              no shared expert) */
    MOE_STAGE_GATHER = 2,  /* x rows of full row blocks copied into expert order */
    MOE_STAGE_GATE_UP = 3,
    MOE_STAGE_DOWN = 4,
    MOE_STAGE_SHARED = 5, /* always empty: the shared expert runs inside the
                             gate/up and down stages (kept for the layout) */
    MOE_STAGE_COMBINE = 6,
    MOE_NUM_STAGES = 7
};

/* Total number of kernels this library has launched in the process. */
uint64_t moe_kernel_launch_count(void);

/* Ask the next moe_forward calls on this thread to record events[i] (created
 * by the caller with timing enabled) on their stream before stage i, and
 * events[MOE_NUM_STAGES] after the last stage; NULL entries are skipped.
 * n_events must be MOE_NUM_STAGES + 1, or 0 with events NULL to stop. */
moe_status_t moe_set_stage_events(cudaEvent_t *events, int n_events);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_MOE_FFN_MOE_H */
