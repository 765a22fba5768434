// kernels.cuh -- parameter blocks and host-side launchers of the kernels of
// libsparse_moe_ffn (router, align, grouped GEMMs, combine).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe.h"

namespace moe {

// Launches `kernel` with programmatic stream serialization (the kernel may be
// scheduled while its predecessor finishes; it calls griddep_wait before
// touching memory) and, when cluster_x > 1, as clusters of cluster_x CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, unsigned cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kBlockM = MOE_BLOCK_M;  // GEMM row block (tokens / pairs per tile)
constexpr int kBlockK = 64;           // 64 bf16 = one 128-byte swizzle row

// ------------------------------------------------------------------ router

struct RouterArgs {
    int64_t N;
    int H, E, k, norm;
    int e_pad;      // MMA N: columns of the logits tile (multiple of 16, <= 256)
    int gamma_col;  // column holding x . g, or -1 without a shared gate
    int split;      // CTAs per cluster along H (router_split(H))
    int reset_status;  // CTA 0 clears *status first (the layer's first kernel)
    float *topk_w;
    int32_t *topk_ids;
    uint16_t *topk_w_bf16;
    float *gamma;
    int32_t *status;
    // row stride of topk_w / topk_ids / topk_w_bf16 (k, or k + virt_slots)
    int out_ld;
    // > 0: after its k routed slots every token gets virt_slots more, the
    // shared expert's chunks as virtual experts virt_base, virt_base + 1, ...,
    // each with weight sigmoid(x . g) (the shared gate)
    int virt_slots;
    int virt_base;
    // grouping fused into the routing kernel (set only when one cluster
    // routes every token: N <= 128, and no virtual slots): the cluster
    // writes what moe_align writes for block size 128 -- sorted_pair,
    // block_expert, counts, offsets, pad_offsets, num_padded -- and zeroes
    // the GEMMs' hand-off counters ready[0 .. ready_n)
    int fuse_align;
    int32_t *sorted_pair;
    int32_t *block_expert;
    int32_t *counts;
    int32_t *offsets;
    int32_t *pad_offsets;
    int32_t *num_padded;
    int32_t *ready;
    int ready_n;
};

int router_split(int H);  // 1, 2, 4 or 8: depends on H only (batch invariance)
size_t router_smem_bytes(int e_pad, int k, int table_bytes);
cudaError_t launch_router(const CUtensorMap &tm_x, const CUtensorMap &tm_router,
                          const CUtensorMap &tm_gate, const RouterArgs &a, cudaStream_t s);

// ------------------------------------------------------------------- align

struct AlignArgs {
    const int32_t *ids;
    int64_t P;       // pairs N*k
    int E, block_m;
    int chunk;       // pairs per CTA in the count / scatter kernels
    int nchunks;
    int32_t *chunk_counts;  // [nchunks, E], becomes the per-chunk base in place
    int32_t *counts, *offsets, *pad_offsets, *num_padded;
    int32_t *sorted_pair, *block_expert;
    int32_t *status;
    // nullable: GEMM hand-off counters, ready[i] = 0 for i < max(E, padded
    // rows / block_m) (per expert at decode, per block pair at prefill)
    int32_t *ready;
};

constexpr int kAlignChunk = 2048;
cudaError_t launch_align(const AlignArgs &a, cudaStream_t s, int *launches);

// ------------------------------------------------------------ grouped GEMM

// kDown multiplies an fp16 activation by fp16 down weights (one MMA per K
// step); kDownSplit multiplies the activation, held as a bf16 pair
// hi + lo, by the model's bf16 down weights (two MMAs per K step: hi, then
// lo, into the same accumulator).  Both keep about 11 or more significant
// bits of the activation, which the output tolerance needs.
enum GemmMode { kGateUp = 0, kDown = 1, kDownSplit = 2 };

__host__ __device__ constexpr bool is_down(int mode) { return mode != kGateUp; }

struct GemmArgs {
    // row map: tile row r of block b holds q = sorted_pair[b*128 + r] (or
    // b*128 + r when sorted_pair is null); the row is real iff q < q_limit
    const int32_t *sorted_pair;
    const int32_t *block_expert;  // null: every block belongs to expert 0
    const int32_t *num_padded;    // device row count; null: use num_rows_host
    int64_t num_rows_host;
    int64_t q_limit;
    int k_div;          // gate/up: the A row gathered for q is q / k_div
    int K;              // reduction length (H for gate/up, I for down)
    int n_out;          // output columns (I for gate/up, H for down)
    int64_t w_rows;     // weight rows per expert (I or H)
    // gate/up: act [rows, I], fp16, or bf16 hi with the bf16 lo rows lo_rows
    // rows further on.  down: the pair rows y [q_limit, H] in the pair-row
    // format (pair_rows.cuh): bf16 hi at out, int8 residual at out_res
    void *out;
    int8_t *out_res;
    int64_t out_ld;
    // 0: fp16 activation.  Otherwise the activation is a bf16 pair: gate/up
    // stores hi at row r and lo = bf16(a - hi) at row r + lo_rows; the
    // kDownSplit GEMM reads its A lo rows lo_rows rows after the hi rows.
    int64_t lo_rows;
    const float *scale; // down: per-q weight (null: 1)
    int32_t *status;
    int stream_weights; // weight tiles read once per call: load them evict-first
    // CTA-pair kernel only: group g (expert) owns padded rows
    // [pad_offsets[g], pad_offsets[g+1]); null: one group of num_rows_host rows
    const int32_t *pad_offsets;
    int num_groups;
    // sparse kernel: tile t = (expert t / n_tiles, N tile t % n_tiles) when set,
    // for batches where every expert owns at most one row block (N <= 128);
    // the tile order is then known before routing, and each CTA warms L2 with
    // its first tile's weight rows (w0, w1: the Wg and Wu bases) while it
    // waits for the earlier kernels
    int expert_tiles;
    const void *w0;
    const void *w1;
    // hand-off from gate/up to down (null: off).  Sparse kernel (decode):
    // gate/up adds 1 to act_ready[e] when a tile of expert e is stored.
    // CTA-pair kernel (prefill): each epilogue warp of both CTAs adds 1 to
    // act_ready[j] when it has stored its rows of a tile of block pair j.
    // Down then waits, per tile, for act_ready[e or j] == act_ready_count
    // instead of for the whole gate/up grid, so its CTAs start on the SMs
    // that gate/up frees first.
    int32_t *act_ready;
    int act_ready_count;
    int max_tiles;      // upper bound on tiles (sizes the persistent grid)
    int grid;           // persistent CTAs
    // the shared expert folded in as virtual experts: groups (experts) from
    // virt_base on are its chunks of virt_chunk intermediate rows, whose
    // weights come from the shared maps (tm_s0 / tm_s1 of the launchers):
    // gate/up, chunk v: rows v * virt_chunk + n0 of shared gate_proj /
    // up_proj; down, chunk v: K columns from v * virt_chunk of shared
    // down_proj.  Rows or columns past I_s read as zero (TMA fill).
    int virt_base;      // INT_MAX without a shared expert
    int virt_chunk;
    // CTA-pair gate/up: the shared expert's blocks load x directly (tm_xv)
    int a_from_x;
};

// Tile widths: gate/up 96 or 128 columns (of each of gate and up), down 256.
// The width changes no output element's arithmetic, only the tile count.
bool gemm_block_n_supported(GemmMode mode, int bn);
// A operands: x (or x_sorted) rows in bf16 for gate/up, the activation rows
// for down (fp16, or the bf16 hi rows followed lo_rows later by the lo
// rows).  B operands: Wg / Wu (bf16) for gate/up, Wd (fp16 for kDown, bf16
// for kDownSplit) for down.
// tm_a: 1-row boxes for gather4 of sparse blocks; tm_a_box: 128-row boxes over
// rows that are contiguous per block; tm_b0 / tm_b1: weight rows, boxes of bn
// rows.
// tm_s0 / tm_s1 (nullable): the shared expert's weight maps (see
// GemmArgs::virt_base), boxes as tm_b0 / tm_b1
cudaError_t launch_gemm(GemmMode mode, int bn, const CUtensorMap &tm_a,
                        const CUtensorMap &tm_a_box, const CUtensorMap &tm_b0,
                        const CUtensorMap &tm_b1, const GemmArgs &a, cudaStream_t s,
                        const CUtensorMap *tm_s0 = nullptr, const CUtensorMap *tm_s1 = nullptr);
// x rows copied into expert order (x_sorted [cap, H]): the real rows of dense
// blocks, or of every block when all_blocks is set
// Blocks whose pairs sit in slots >= skip_slot (the shared expert's chunks,
// whose rows are x in token order) are skipped; skip_slot >= k skips none.
cudaError_t launch_gather_rows(const uint16_t *x, int H, int k, const int32_t *sorted_pair,
                               const int32_t *num_padded, int64_t P, int64_t cap,
                               uint16_t *x_sorted, int all_blocks, int skip_slot, int num_sms,
                               cudaStream_t s);

// CTA-pair grouped GEMM (cta_group::2, M = 256 over two row blocks of one
// group): tm_a: 128-row boxes over A rows that are contiguous per block
// (x_sorted for gate/up, act for down); tm_b0 / tm_b1: weight rows, Wg / Wu
// in boxes of pair_gemm_block_n(kGateUp) rows for gate/up, Wd in boxes of
// pair_gemm_block_n(kDown) / 2 rows for down.  a.grid must be even (two CTAs
// per cluster).
int pair_gemm_block_n(GemmMode mode);

// Grouped GEMM for blocks holding few real rows (decode): activation rows in
// 32-row passes, gathered with tile::gather4 (tm_a: 1-row boxes of x rows for
// gate/up, act rows for down), more weight stages in flight; tm_b0 / tm_b1 as
// for launch_gemm (boxes of bn rows).  Needs the routed block list
// (sorted_pair, block_expert, num_padded).
cudaError_t launch_sparse_gemm(GemmMode mode, int bn, const CUtensorMap &tm_a,
                               const CUtensorMap &tm_b0, const CUtensorMap &tm_b1,
                               const GemmArgs &a, cudaStream_t s,
                               const CUtensorMap *tm_s0 = nullptr,
                               const CUtensorMap *tm_s1 = nullptr);
// tm_xv (nullable, gate/up): 128-row boxes over x; the row blocks of the
// shared expert's chunks (groups >= a.virt_base) then load their A rows
// from x directly, block j of a chunk being tokens [128 j, 128 j + 128)
// (the grouping keeps pairs in token order), instead of from tm_a
cudaError_t launch_pair_gemm(GemmMode mode, const CUtensorMap &tm_a, const CUtensorMap &tm_b0,
                             const CUtensorMap &tm_b1, const GemmArgs &a, cudaStream_t s,
                             const CUtensorMap *tm_s0 = nullptr,
                             const CUtensorMap *tm_s1 = nullptr,
                             const CUtensorMap *tm_xv = nullptr);

// ----------------------------------------------------------------- combine

// ypair / yshared: pair rows (bf16 hi plane, int8 residual plane); pair p's
// row is row_index[p] when row_index is given (the order in which
// expert-parallel results come back; an index outside [0, rows) adds
// nothing), else p; yshared (nullable): shared_slots rows per token, row
// n * shared_slots + c, added after the k slots in chunk order
cudaError_t launch_combine(const uint16_t *ypair_hi, const int8_t *ypair_res,
                           const int32_t *row_index, int64_t rows, const uint16_t *yshared_hi,
                           const int8_t *yshared_res, int shared_slots, int64_t N, int H, int k,
                           uint16_t *out, int num_sms, cudaStream_t s);

// ------------------------------------------- expert-parallel dispatch plan

// dest[p] = ids[p] / e_local (-1 and MOE_ERR_DEVICE_CHECK for an id outside
// [0, E)); inv[p] = -1
cudaError_t launch_ep_dest(const int32_t *ids, int64_t P, int E, int e_local, int32_t *dest,
                           int32_t *inv, int32_t *status, int num_sms, cudaStream_t s);
// send row i <- pair order[i] (i < *num_rows): x row, local expert id,
// weight; inv[order[i]] = i
cudaError_t launch_ep_pack(const uint16_t *x, const int32_t *ids, const float *weights,
                           const int32_t *order, const int32_t *num_rows, int64_t P, int H, int k,
                           int e_local, uint16_t *send_x, int32_t *send_ids, float *send_w,
                           int32_t *inv, int num_sms, cudaStream_t s);
// ids[n*C + c] = c, w[n*C + c] = gamma[n]: the slots of the shared expert's
// C chunks when it runs on its own
cudaError_t launch_shared_slots(const float *gamma, int64_t N, int C, int32_t *ids, float *w,
                                int num_sms, cudaStream_t s);

// ------------------------------------------- bf16 -> fp16 weight conversion

// dst[i] = fp16(src[i]) (round to nearest even) for i < n; src and dst
// 16-byte aligned; a magnitude above 65504 or a NaN records
// MOE_ERR_DEVICE_CHECK in *status (nullable)
cudaError_t launch_convert_bf16_to_f16(const uint16_t *src, uint16_t *dst, int64_t n,
                                       int32_t *status, int num_sms, cudaStream_t s);

// ------------------------------------------------- residual add + RMSNorm

cudaError_t launch_add_rmsnorm(const uint16_t *x, uint16_t *residual, const uint16_t *w,
                               int64_t N, int H, float eps, int gemma, uint16_t *normed,
                               int num_sms, cudaStream_t s);

// Sets the message moe_last_error() returns on this thread.
void set_last_error(const char *msg);

// ---------------------------------------------------------------- selftest

cudaError_t launch_wait_timeout_probe(int32_t *status, uint64_t limit_ns, cudaStream_t s);

}  // namespace moe
