// api.cu -- the C ABI of libsparse_moe_ffn (declared in include/moe.h):
// argument checks, workspace carving, TMA tensor maps and kernel launches.
// Host code only; it allocates nothing, frees nothing and synchronises
// nothing (except moe_read_device_status).
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "kernels.cuh"
#include "moe.h"

using namespace moe;

namespace {

thread_local std::string g_last_error;
thread_local cudaEvent_t g_stage_events[MOE_NUM_STAGES + 1];
thread_local bool g_stage_events_on = false;
std::atomic<uint64_t> g_launches{0};

moe_status_t fail(moe_status_t s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

moe_status_t cuda_fail(cudaError_t e, const char *what) {
    return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define MOE_CUDA(call, what)                                   \
    do {                                                       \
        cudaError_t e_ = (call);                               \
        if (e_ != cudaSuccess) return cuda_fail(e_, (what));   \
    } while (0)

constexpr size_t kAlign = 256;
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int64_t round_up64(int64_t v, int64_t a) { return (v + a - 1) / a * a; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// --------------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 16-bit matrix [rows, cols] (row stride `ld` elements), 128-byte swizzled
// box of box_rows x box_cols (box_cols * 2 <= 128).  Out-of-range elements
// read 0.  Used for bf16 and fp16 data alike: the copy moves 16-bit elements
// unchanged, and zero has the same bits in both formats.
moe_status_t make_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                      uint64_t ld, uint32_t box_cols, uint32_t box_rows, const char *what) {
    auto fn = encode_tiled();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {ld * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MOE_ERR_CUDA, "tensor map for %s rejected (CUresult %d)", what,
                    static_cast<int>(r));
    return MOE_OK;
}

int num_sms_of_current_device() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 148;
    }
    return cache[dev];
}

moe_status_t record_stage(int i, cudaStream_t s) {
    if (!g_stage_events_on || g_stage_events[i] == nullptr) return MOE_OK;
    cudaError_t e = cudaEventRecord(g_stage_events[i], s);
    if (e != cudaSuccess) return cuda_fail(e, "stage event record");
    return MOE_OK;
}

// ------------------------------------------------------------ tile choice

// Expected number of 128-row blocks after grouping P pairs over E experts
// (near-uniform routing): touched experts times blocks per touched expert.
double expected_blocks(int64_t P, int E) {
    const double touched = E * (1.0 - std::exp(-static_cast<double>(P) / E));
    if (touched < 1.0) return 1.0;
    const double per = static_cast<double>(P) / touched;
    return touched * (per <= kBlockM ? 1.0 : per / kBlockM + 0.5);
}

// Fraction of SM time lost to the last, partial wave of `tiles` tiles.
double wave_loss(double tiles, int sms) {
    const double waves = tiles / sms;
    return std::ceil(waves) / waves - 1.0;
}

// Wave loss averaged over +-3% around the expected block count (the real
// count is only known on the device, and the loss jumps at wave boundaries).
double mean_wave_loss(double blocks, int tiles_per_block, int sms) {
    double sum = 0.0;
    for (double f : {0.97, 0.985, 1.0, 1.015, 1.03})
        sum += wave_loss(blocks * f * tiles_per_block, sms);
    return sum / 5.0;
}

// Gate/up tile width: the one losing less SM time to wave quantisation; when
// blocks are dense (compute bound) 96 must win by 3 points to be taken,
// since wider tiles reuse each A tile over more columns.
int choose_gate_up_bn(double blocks, double rows_per_expert, int I, int sms) {
    const double l128 = mean_wave_loss(blocks, (I + 127) / 128, sms);
    const double l96 = mean_wave_loss(blocks, (I + 95) / 96, sms);
    const double margin = rows_per_expert >= kBlockM ? 0.03 : 0.0;
    return l96 + margin < l128 ? 96 : 128;
}

constexpr int kDownBN = 256;

// ------------------------------------------------------------------ layouts

int align_chunks(int64_t P) { return static_cast<int>((P + kAlignChunk - 1) / kAlignChunk); }

int router_e_pad(int E, bool shared) {
    const int e8 = (E + 7) / 8 * 8;
    const int cols = shared ? e8 + 8 : E;
    return (cols < 16 ? 16 : (cols + 15) / 16 * 16);
}

moe_status_t check_route_args(const void *x, const void *router, const void *shared_gate,
                              int64_t N, int H, int E, int k, float *topk_w, int32_t *topk_ids,
                              float *gamma) {
    if (N < 0) return fail(MOE_ERR_INVALID_ARG, "N must be >= 0 (got %lld)", (long long)N);
    if (H < 8 || H % 8) return fail(MOE_ERR_INVALID_ARG, "H must be a positive multiple of 8 (got %d)", H);
    if (E < 1) return fail(MOE_ERR_INVALID_ARG, "E must be >= 1 (got %d)", E);
    if (k < 1 || k > E) return fail(MOE_ERR_INVALID_ARG, "k must be in [1, E] (k=%d, E=%d)", k, E);
    if (router_e_pad(E, shared_gate != nullptr) > MOE_MAX_EXPERTS)
        return fail(MOE_ERR_UNSUPPORTED, "E=%d exceeds the fused router's limit", E);
    if (N == 0) return MOE_OK;
    if (!x || !router || !topk_w || !topk_ids)
        return fail(MOE_ERR_INVALID_ARG, "x, router, topk_w and topk_ids must be non-null");
    if (shared_gate && !gamma)
        return fail(MOE_ERR_INVALID_ARG, "shared_gamma must be given with shared_gate");
    if (!aligned16(x) || !aligned16(router) || (shared_gate && !aligned16(shared_gate)))
        return fail(MOE_ERR_INVALID_ARG, "bf16 matrices must be 16-byte aligned");
    if (N > (int64_t(1) << 31) / k)
        return fail(MOE_ERR_UNSUPPORTED, "N*k must stay below 2^31");
    return MOE_OK;
}

struct AlignBuffers {
    int32_t *sorted_pair, *block_expert, *counts, *offsets, *pad_offsets, *num_padded, *scratch;
    int32_t *status;
    int32_t *ready = nullptr;
};

moe_status_t enqueue_route(const moe_bf16_t *x, const moe_bf16_t *router,
                           const moe_bf16_t *shared_gate, int64_t N, int H, int E, int k,
                           int norm, float *topk_w, int32_t *topk_ids, moe_bf16_t *topk_w_bf16,
                           float *gamma, int32_t *status, bool reset_status,
                           cudaStream_t stream, int virt_slots = 0,
                           const AlignBuffers *fused = nullptr, int ready_n = 0) {
    const bool shared = shared_gate != nullptr;
    RouterArgs ra;
    ra.N = N;
    ra.H = H;
    ra.E = E;
    ra.k = k;
    ra.norm = norm ? 1 : 0;
    ra.e_pad = router_e_pad(E, shared);
    ra.gamma_col = shared ? (E + 7) / 8 * 8 : -1;
    ra.split = router_split(H);
    ra.reset_status = reset_status ? 1 : 0;
    ra.topk_w = topk_w;
    ra.topk_ids = topk_ids;
    ra.topk_w_bf16 = topk_w_bf16;
    ra.gamma = gamma;
    ra.status = status;
    ra.out_ld = k + virt_slots;
    ra.virt_slots = virt_slots;
    ra.virt_base = E;
    // the grouping done by the routing cluster itself (one cluster routes
    // every token): moe_align's outputs for 128-row blocks
    ra.fuse_align = fused ? 1 : 0;
    ra.sorted_pair = fused ? fused->sorted_pair : nullptr;
    ra.block_expert = fused ? fused->block_expert : nullptr;
    ra.counts = fused ? fused->counts : nullptr;
    ra.offsets = fused ? fused->offsets : nullptr;
    ra.pad_offsets = fused ? fused->pad_offsets : nullptr;
    ra.num_padded = fused ? fused->num_padded : nullptr;
    ra.ready = fused ? fused->ready : nullptr;
    ra.ready_n = fused ? ready_n : 0;
    CUtensorMap tm_x, tm_r, tm_g;
    moe_status_t st;
    if ((st = make_map(&tm_x, x, H, N, H, kBlockK, kBlockM, "x")) != MOE_OK) return st;
    if ((st = make_map(&tm_r, router, H, E, H, kBlockK, E, "router")) != MOE_OK) return st;
    if (shared) {
        if ((st = make_map(&tm_g, shared_gate, H, 1, H, kBlockK, 8, "shared_gate")) != MOE_OK)
            return st;
    } else {
        tm_g = tm_r;  // unused placeholder
    }
    MOE_CUDA(launch_router(tm_x, tm_r, tm_g, ra, stream), "router kernel launch");
    g_launches += 1;
    return MOE_OK;
}


moe_status_t enqueue_align(const int32_t *ids, int64_t N, int k, int E, int block_m,
                           const AlignBuffers &b, cudaStream_t stream) {
    AlignArgs aa;
    aa.ids = ids;
    aa.P = N * k;
    aa.E = E;
    aa.block_m = block_m;
    aa.chunk = kAlignChunk;
    aa.nchunks = align_chunks(aa.P);
    aa.chunk_counts = b.scratch;
    aa.counts = b.counts;
    aa.offsets = b.offsets;
    aa.pad_offsets = b.pad_offsets;
    aa.num_padded = b.num_padded;
    aa.sorted_pair = b.sorted_pair;
    aa.block_expert = b.block_expert;
    aa.status = b.status;
    aa.ready = b.ready;
    int launches = 0;
    cudaError_t e = launch_align(aa, stream, &launches);
    g_launches += launches;
    if (e != cudaSuccess) return cuda_fail(e, "align kernel launch");
    return MOE_OK;
}

// The CTA-pair GEMMs pay from one row block per expert on average: every
// weight tile then serves 256 rows instead of 128, and a pair whose second
// block is padding still loads each weight byte once (its idle MMA rows cost
// little while weights dominate).  Talker-sized batches (1.5 blocks per
// expert) run 3% faster this way; decode-sized ones stream weights anyway.
bool use_pair_tiles(int64_t P, int E) { return P >= static_cast<int64_t>(kBlockM) * E; }

// Fewer than 32 pairs per expert on average (decode-sized batches): most row
// blocks hold a handful of real rows, and the GEMMs that stage activation
// rows in 32-row passes keep more weight bytes in flight.
bool use_sparse_tiles(int64_t P, int E) { return P < 32 * static_cast<int64_t>(E); }

// The shared expert runs as shared_chunks(I, I_s) virtual experts E, E+1, ...
// of I intermediate rows each (the last one padded with zero weights by the
// TMA fill), which every token uses with the shared gate as its weight: its
// slots k, k+1, ... of the routing and grouping.
int shared_chunks(int I, int I_s) { return I_s > 0 ? (I_s + I - 1) / I : 0; }

moe_status_t forward_layout(int64_t N, int H, int E_routed, int I, int k_routed, int I_s,
                            moe_forward_layout_t *L) {
    const bool shared = I_s > 0;
    const int C = shared_chunks(I, I_s);
    const int k = k_routed + C;  // slots per token, routed then shared chunks
    const int E = E_routed + C;  // groups: the experts, then the shared chunks
    const int64_t P = N * k;
    const int64_t cap = moe_align_capacity(N, k, E, kBlockM);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = round_up(off + bytes, kAlign);
        return at;
    };
    L->status = take(4);
    L->topk_w = take(sizeof(float) * P);
    L->topk_ids = take(sizeof(int32_t) * P);
    L->gamma = take(shared ? sizeof(float) * N : 0);
    L->counts = take(sizeof(int32_t) * E);
    L->offsets = take(sizeof(int32_t) * (E + 1));
    L->pad_offsets = take(sizeof(int32_t) * (E + 1));
    L->num_padded = take(sizeof(int32_t));
    L->align_scratch = take(sizeof(int32_t) * static_cast<size_t>(align_chunks(P)) * E);
    L->sorted_pair = take(sizeof(int32_t) * cap);
    L->block_expert = take(sizeof(int32_t) * (cap / kBlockM));
    L->ready = take(sizeof(int32_t) * (E > cap / kBlockM ? E : cap / kBlockM));
    L->x_sorted = take(2 * static_cast<size_t>(cap) * H);
    // the activation: fp16, or a bf16 hi/lo pair (4 bytes a value either way
    // is reserved, so one workspace serves both forms of the down weights)
    L->act = take(4 * static_cast<size_t>(cap) * I);
    // pair rows: bf16 hi plane and int8 residual plane
    L->ypair = take(2 * static_cast<size_t>(P) * H);
    L->ypair_res = take(static_cast<size_t>(P) * H);
    L->total = off;
    L->capacity = cap;
    L->slots = k;
    L->groups = E;
    return MOE_OK;
}

// Every argument check of moe_forward, before anything is enqueued; on
// success *shared_out tells whether the shared expert is present and *L holds
// the workspace layout.
moe_status_t check_forward_args(const moe_bf16_t *x, const moe_bf16_t *router,
                                const moe_bf16_t *w_gate, const moe_bf16_t *w_up,
                                const void *w_down, const moe_bf16_t *shared_gate_proj,
                                const moe_bf16_t *shared_up_proj,
                                const void *shared_down_proj, const moe_bf16_t *shared_gate,
                                int64_t N, int H, int E, int I, int I_s, int k,
                                const moe_bf16_t *out, const void *workspace,
                                size_t workspace_bytes, bool *shared_out,
                                moe_forward_layout_t *L) {
    const int nshared = (shared_gate_proj != nullptr) + (shared_up_proj != nullptr) +
                        (shared_down_proj != nullptr) + (shared_gate != nullptr);
    if (nshared != 0 && nshared != 4)
        return fail(MOE_ERR_INVALID_ARG,
                    "give all four shared-expert tensors or none (got %d of 4)", nshared);
    const bool shared = nshared == 4;
    *shared_out = shared;
    if (!shared) I_s = 0;
    if (shared && (I_s < 8 || I_s % 8))
        return fail(MOE_ERR_INVALID_ARG, "I_s must be a positive multiple of 8 (got %d)", I_s);
    if (I < 8 || I % 8) return fail(MOE_ERR_INVALID_ARG, "I must be a positive multiple of 8 (got %d)", I);
    float dummy_gamma;
    int32_t dummy_ids;
    moe_status_t st = check_route_args(x, router, shared ? shared_gate : nullptr, N, H, E, k,
                                       reinterpret_cast<float *>(&dummy_gamma), &dummy_ids,
                                       &dummy_gamma);
    if (st != MOE_OK || N == 0) return st;
    if (!w_gate || !w_up || !w_down || !out || !workspace)
        return fail(MOE_ERR_INVALID_ARG, "w_gate, w_up, w_down, out and workspace must be non-null");
    if (!aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(out) ||
        (shared && (!aligned16(shared_gate_proj) || !aligned16(shared_up_proj) ||
                    !aligned16(shared_down_proj))))
        return fail(MOE_ERR_INVALID_ARG, "bf16 matrices must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    // the hi and lo rows of a split activation share one row index space
    const int C = shared_chunks(I, shared ? I_s : 0);
    if (E + C > MOE_MAX_EXPERTS)
        return fail(MOE_ERR_UNSUPPORTED,
                    "E + ceil(I_s / I) (the shared expert's chunks) must be <= %d (got %d)",
                    MOE_MAX_EXPERTS, E + C);
    if (N * (k + C) + static_cast<int64_t>(E + C) * kBlockM >= (int64_t(1) << 30))
        return fail(MOE_ERR_UNSUPPORTED, "N*(k + chunks) + (E + chunks)*128 must stay below 2^30");
    forward_layout(N, H, E, I, k, shared ? I_s : 0, L);
    if (workspace_bytes < L->total)
        return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "forward workspace needs %zu bytes, got %zu",
                    L->total, workspace_bytes);
    return MOE_OK;
}


// Grouping, gate/up and down for N rows with k (expert, weight) slots each:
// ypair[p] = weights[p] * Expert_{ids[p]}(x[p / k]) in fp32, p = n * k + j.
// w_down is bf16 (down_f16 false: the activation kept as a bf16 hi/lo pair)
// or its fp16 copy (down_f16 true: an fp16 activation).  The workspace
// follows moe_forward_layout(N, H, E, I, k, 0); its status word is not reset
// here.  Records the align .. down stage events.
// The shared expert folded into the grouped GEMMs (see shared_chunks):
// groups from E_routed on read these weights.
struct SharedWeights {
    const moe_bf16_t *gate_proj, *up_proj;  // [I_s, H]
    const void *down_proj;                  // [H, I_s], bf16 or fp16 as w_down
    int I_s;
    int E_routed;
};

// moe_align's outputs inside a forward workspace
AlignBuffers align_buffers_of(const moe_forward_layout_t &L, uint8_t *ws) {
    AlignBuffers b;
    b.sorted_pair = reinterpret_cast<int32_t *>(ws + L.sorted_pair);
    b.block_expert = reinterpret_cast<int32_t *>(ws + L.block_expert);
    b.counts = reinterpret_cast<int32_t *>(ws + L.counts);
    b.offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    b.pad_offsets = reinterpret_cast<int32_t *>(ws + L.pad_offsets);
    b.num_padded = reinterpret_cast<int32_t *>(ws + L.num_padded);
    b.scratch = reinterpret_cast<int32_t *>(ws + L.align_scratch);
    b.status = reinterpret_cast<int32_t *>(ws + L.status);
    b.ready = reinterpret_cast<int32_t *>(ws + L.ready);
    return b;
}

// hand-off counters in a forward workspace (max(E, capacity / 128))
int ready_count_of(const moe_forward_layout_t &L) {
    const int blocks = static_cast<int>(L.capacity / kBlockM);
    return L.groups > blocks ? L.groups : blocks;
}

// Routing can group the pairs itself when one cluster routes every token
// and no shared-expert slots follow the routed ones.
bool route_groups(int64_t N, int E, bool shared) {
    return N <= kBlockM && E <= 256 && !shared;
}

moe_status_t enqueue_experts(const moe_bf16_t *x, const int32_t *ids, const float *weights,
                             int64_t N, int k, int H, int E, int I, const moe_bf16_t *w_gate,
                             const moe_bf16_t *w_up, const void *w_down, bool down_f16,
                             const moe_forward_layout_t &L, uint8_t *ws, uint16_t *ypair,
                             int8_t *ypair_res, cudaStream_t stream,
                             const SharedWeights *sh = nullptr, bool grouped = false) {
    moe_status_t st;
    auto at = [&](size_t off) { return ws + off; };
    int32_t *status = reinterpret_cast<int32_t *>(at(L.status));
    uint16_t *x_sorted = reinterpret_cast<uint16_t *>(at(L.x_sorted));
    uint16_t *act = reinterpret_cast<uint16_t *>(at(L.act));
    const int64_t P = N * k;
    const int64_t cap = L.capacity;
    const int sms = num_sms_of_current_device();

    // Decode hand-off: with expert-indexed gate/up tiles (every expert owns
    // at most one row block) the down GEMM waits per expert for its
    // activation rows instead of for the whole gate/up grid (the grouping
    // kernel zeroes the counters).
    const bool handoff = !use_pair_tiles(P, E) && use_sparse_tiles(P, E) && N <= kBlockM;
    // the same for the CTA-pair GEMMs (prefill), per block pair
    const bool pair_handoff = use_pair_tiles(P, E);
    int32_t *ready = reinterpret_cast<int32_t *>(at(L.ready));

    // K2: grouping
    if ((st = record_stage(MOE_STAGE_ALIGN, stream)) != MOE_OK) return st;
    AlignBuffers b = align_buffers_of(L, ws);
    b.ready = handoff || pair_handoff ? ready : nullptr;
    if (!grouped) {  // (else the routing kernel has grouped the pairs)
        st = enqueue_align(ids, N, k, E, kBlockM, b, stream);
        if (st != MOE_OK) return st;
    }

    // K3: gathered gate/up GEMM + silu * up
    CUtensorMap tm_xrows, tm_xsorted, tm_wg, tm_wu, tm_act, tm_act_box, tm_wd;
    if ((st = make_map(&tm_xrows, x, H, N, H, kBlockK, 1, "x rows")) != MOE_OK) return st;
    if ((st = make_map(&tm_xsorted, x_sorted, H, cap, H, kBlockK, kBlockM, "x_sorted")) != MOE_OK)
        return st;
    const int bn_gu = choose_gate_up_bn(expected_blocks(P, E), static_cast<double>(P) / E, I, sms);
    // the routed experts' weights; the shared expert's chunks (groups from
    // E_routed on) read the shared maps
    const int E_map = sh ? sh->E_routed : E;
    // no routed experts (the shared expert on its own): the routed maps are
    // never read, so they describe the shared weights
    const bool all_virtual = sh && sh->E_routed == 0;
    if (all_virtual) {
        w_gate = sh->gate_proj;
        w_up = sh->up_proj;
        w_down = sh->down_proj;
    }
    const uint64_t gu_rows = all_virtual ? sh->I_s : static_cast<uint64_t>(E_map) * I;
    const uint64_t down_rows = all_virtual ? H : static_cast<uint64_t>(E_map) * H;
    if ((st = make_map(&tm_wg, w_gate, H, gu_rows, H, kBlockK, bn_gu, "w_gate")) != MOE_OK)
        return st;
    if ((st = make_map(&tm_wu, w_up, H, gu_rows, H, kBlockK, bn_gu, "w_up")) != MOE_OK)
        return st;
    CUtensorMap tm_sg, tm_su, tm_sd;
    const CUtensorMap *psg = nullptr, *psu = nullptr, *psd = nullptr;
    auto shared_gate_up_maps = [&](int box_rows) -> moe_status_t {
        if (!sh) return MOE_OK;
        moe_status_t r;
        if ((r = make_map(&tm_sg, sh->gate_proj, H, sh->I_s, H, kBlockK, box_rows,
                          "shared_gate_proj")) != MOE_OK ||
            (r = make_map(&tm_su, sh->up_proj, H, sh->I_s, H, kBlockK, box_rows,
                          "shared_up_proj")) != MOE_OK)
            return r;
        psg = &tm_sg;
        psu = &tm_su;
        return MOE_OK;
    };
    auto shared_down_map = [&](int box_rows) -> moe_status_t {
        if (!sh) return MOE_OK;
        moe_status_t r = make_map(&tm_sd, sh->down_proj, sh->I_s, H, sh->I_s, kBlockK, box_rows,
                                  "shared_down_proj");
        if (r != MOE_OK) return r;
        psd = &tm_sd;
        return MOE_OK;
    };
    const bool pairs = use_pair_tiles(P, E);
    const bool sparse = !pairs && use_sparse_tiles(P, E);
    GemmArgs g;
    g.sorted_pair = b.sorted_pair;
    g.block_expert = b.block_expert;
    g.pad_offsets = b.pad_offsets;
    g.num_groups = E;
    g.expert_tiles = 0;
    g.w0 = g.w1 = nullptr;
    g.act_ready = nullptr;
    g.act_ready_count = 0;
    g.virt_base = sh ? sh->E_routed : INT_MAX;
    g.virt_chunk = I;
    g.a_from_x = 0;
    g.num_padded = b.num_padded;
    g.num_rows_host = cap;
    g.q_limit = P;
    g.k_div = k;
    g.K = H;
    g.n_out = I;
    g.w_rows = I;
    g.out = act;
    g.out_res = nullptr;
    g.out_ld = I;
    g.lo_rows = down_f16 ? 0 : cap;  // bf16 down weights: hi/lo activation
    g.scale = nullptr;
    g.status = status;
    // fewer than a block of pairs per expert: every weight tile is read once
    g.stream_weights = P < static_cast<int64_t>(E) * kBlockM ? 1 : 0;
    {
        const int nt = (I + bn_gu - 1) / bn_gu;
        g.max_tiles = static_cast<int>(cap / kBlockM) * nt;
        g.grid = g.max_tiles < sms ? g.max_tiles : sms;
    }
    if ((st = record_stage(MOE_STAGE_GATHER, stream)) != MOE_OK) return st;
    // the CTA-pair gate/up loads the shared expert's rows (x in token order)
    // from x itself; its blocks are not gathered
    const bool shared_from_x = pairs && sh != nullptr;
    if (!sparse) {  // the sparse GEMM gathers its x rows itself
        const int skip_slot = shared_from_x ? k - (E - sh->E_routed) : INT_MAX;
        MOE_CUDA(launch_gather_rows(x, H, k, b.sorted_pair, b.num_padded, P, cap, x_sorted,
                                    pairs ? 1 : 0, skip_slot, sms, stream),
                 "gather kernel launch");
        g_launches += 1;
    }
    if ((st = record_stage(MOE_STAGE_GATE_UP, stream)) != MOE_OK) return st;
    if (sparse) {
        if (N <= kBlockM) {
            // every expert owns at most one row block: tiles indexed by
            // expert, the first ones' weight rows warmed into L2 during routing
            g.expert_tiles = 1;
            g.w0 = w_gate;
            g.w1 = w_up;
            g.max_tiles = E * ((I + bn_gu - 1) / bn_gu);
            g.grid = g.max_tiles < sms ? g.max_tiles : sms;
            if (handoff) {  // kept for the down GEMM below
                g.act_ready = ready;
                g.act_ready_count = (I + bn_gu - 1) / bn_gu;
            }
        }
        if ((st = shared_gate_up_maps(bn_gu)) != MOE_OK) return st;
        MOE_CUDA(launch_sparse_gemm(kGateUp, bn_gu, tm_xrows, tm_wg, tm_wu, g, stream, psg, psu),
                 "gate/up kernel launch");
        g.expert_tiles = 0;
    } else if (pairs) {
        const int bn = pair_gemm_block_n(kGateUp);
        CUtensorMap tm_wg_tile, tm_wu_tile;
        if ((st = make_map(&tm_wg_tile, w_gate, H, gu_rows, H, kBlockK, bn, "w_gate")) != MOE_OK)
            return st;
        if ((st = make_map(&tm_wu_tile, w_up, H, gu_rows, H, kBlockK, bn, "w_up")) != MOE_OK)
            return st;
        if ((st = shared_gate_up_maps(bn)) != MOE_OK) return st;
        const int max_pairs = static_cast<int>(cap / kBlockM);  // pairs <= blocks
        g.max_tiles = max_pairs * ((I + bn - 1) / bn);
        g.grid = 2 * (g.max_tiles < sms / 2 ? g.max_tiles : sms / 2);
        if (pair_handoff) {  // kept for the down GEMM below
            // one arrival per epilogue warp (4) of both CTAs per gate/up tile
            g.act_ready = ready;
            g.act_ready_count = 8 * ((I + bn - 1) / bn);
        }
        CUtensorMap tm_xv;
        if (shared_from_x) {
            if ((st = make_map(&tm_xv, x, H, N, H, kBlockK, kBlockM, "x")) != MOE_OK) return st;
            g.a_from_x = 1;
        }
        MOE_CUDA(launch_pair_gemm(kGateUp, tm_xsorted, tm_wg_tile, tm_wu_tile, g, stream, psg,
                                  psu, shared_from_x ? &tm_xv : nullptr),
                 "gate/up kernel launch");
        g.a_from_x = 0;
    } else {
        if ((st = shared_gate_up_maps(bn_gu)) != MOE_OK) return st;
        MOE_CUDA(launch_gemm(kGateUp, bn_gu, tm_xrows, tm_xsorted, tm_wg, tm_wu, g, stream, psg,
                             psu),
                 "gate/up kernel launch");
    }
    g_launches += 1;

    // K4: down GEMM * routing weight, one row per pair
    if ((st = record_stage(MOE_STAGE_DOWN, stream)) != MOE_OK) return st;
    const GemmMode down = down_f16 ? kDown : kDownSplit;
    const int64_t act_rows = down_f16 ? cap : 2 * cap;  // split: hi rows, then lo rows
    if ((st = make_map(&tm_act, act, I, act_rows, I, kBlockK, 1, "act rows")) != MOE_OK) return st;
    if ((st = make_map(&tm_act_box, act, I, act_rows, I, kBlockK, kBlockM, "act")) != MOE_OK)
        return st;
    const uint64_t down_cols = all_virtual ? sh->I_s : I;
    if ((st = make_map(&tm_wd, w_down, down_cols, down_rows, down_cols, kBlockK, kDownBN,
                       "w_down")) != MOE_OK)
        return st;
    g.k_div = 1;
    g.K = I;
    g.n_out = H;
    g.w_rows = H;
    g.out = ypair;
    g.out_res = ypair_res;
    g.out_ld = H;
    g.scale = weights;
    {
        const int nt = (H + kDownBN - 1) / kDownBN;
        g.max_tiles = static_cast<int>(cap / kBlockM) * nt;
        g.grid = g.max_tiles < sms ? g.max_tiles : sms;
    }
    if (sparse) {
        if ((st = shared_down_map(kDownBN)) != MOE_OK) return st;
        MOE_CUDA(launch_sparse_gemm(down, kDownBN, tm_act, tm_wd, tm_wd, g, stream, psd, psd),
                 "down kernel launch");
    } else if (pairs) {
        const int bn = pair_gemm_block_n(down);
        CUtensorMap tm_wd_half;
        if ((st = make_map(&tm_wd_half, w_down, down_cols, down_rows, down_cols, kBlockK, bn / 2,
                           "w_down")) != MOE_OK)
            return st;
        if ((st = shared_down_map(bn / 2)) != MOE_OK) return st;
        g.max_tiles = static_cast<int>(cap / kBlockM) * ((H + bn - 1) / bn);
        g.grid = 2 * (g.max_tiles < sms / 2 ? g.max_tiles : sms / 2);
        MOE_CUDA(launch_pair_gemm(down, tm_act_box, tm_wd_half, tm_wd_half, g, stream, psd, psd),
                 "down kernel launch");
    } else {
        if ((st = shared_down_map(kDownBN)) != MOE_OK) return st;
        MOE_CUDA(launch_gemm(down, kDownBN, tm_act, tm_act_box, tm_wd, tm_wd, g, stream, psd,
                             psd),
                 "down kernel launch");
    }
    g_launches += 1;

    return MOE_OK;
}

}  // namespace

void moe::set_last_error(const char *msg) { g_last_error = msg; }

// =========================================================================
extern "C" {

const char *moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MOE_ERR_UNSUPPORTED: return "unsupported size";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_CHECK: return "device-side check failed (bad input value)";
        case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

const char *moe_last_error(void) { return g_last_error.c_str(); }

uint64_t moe_kernel_launch_count(void) { return g_launches.load(); }

moe_status_t moe_set_stage_events(cudaEvent_t *events, int n_events) {
    if (n_events == 0 && events == nullptr) {
        g_stage_events_on = false;
        return MOE_OK;
    }
    if (!events || n_events != MOE_NUM_STAGES + 1)
        return fail(MOE_ERR_INVALID_ARG, "need %d events", MOE_NUM_STAGES + 1);
    for (int i = 0; i <= MOE_NUM_STAGES; ++i) g_stage_events[i] = events[i];
    g_stage_events_on = true;
    return MOE_OK;
}

size_t moe_route_workspace_bytes(void) { return kAlign; }

moe_status_t moe_route(const moe_bf16_t *x, const moe_bf16_t *router,
                       const moe_bf16_t *shared_gate, int64_t N, int H, int E, int k,
                       int norm_topk_prob, float *topk_w, int32_t *topk_ids,
                       moe_bf16_t *topk_w_bf16, float *shared_gamma, void *workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
    g_last_error.clear();
    moe_status_t st = check_route_args(x, router, shared_gate, N, H, E, k, topk_w, topk_ids,
                                       shared_gamma);
    if (st != MOE_OK || N == 0) return st;
    if (workspace && workspace_bytes < moe_route_workspace_bytes())
        return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "route workspace needs %zu bytes",
                    moe_route_workspace_bytes());
    int32_t *status = static_cast<int32_t *>(workspace);
    if (status) MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(int32_t), stream), "status reset");
    return enqueue_route(x, router, shared_gate, N, H, E, k, norm_topk_prob, topk_w, topk_ids,
                         topk_w_bf16, shared_gamma, status, false, stream);
}

int64_t moe_align_capacity(int64_t N, int k, int E, int block_m) {
    if (N < 0 || k < 1 || E < 1 || block_m < 1) return 0;
    return round_up64(N * k + static_cast<int64_t>(E) * (block_m - 1), block_m);
}

size_t moe_align_workspace_bytes(int64_t N, int k, int E, int block_m) {
    if (N < 0 || k < 1 || E < 1 || block_m < 1) return 0;
    return kAlign + round_up(sizeof(int32_t) * (E + 1), kAlign) +
           round_up(sizeof(int32_t) * static_cast<size_t>(align_chunks(N * k)) * E, kAlign);
}

moe_status_t moe_align(const int32_t *topk_ids, int64_t N, int k, int E, int block_m,
                       int32_t *sorted_pair, int32_t *block_expert, int32_t *counts,
                       int32_t *offsets, int32_t *num_padded, void *workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
    g_last_error.clear();
    if (N < 0 || k < 1 || E < 1 || block_m < 1)
        return fail(MOE_ERR_INVALID_ARG, "need N >= 0, k >= 1, E >= 1, block_m >= 1");
    if (E > 1024 || block_m > 1024)
        return fail(MOE_ERR_UNSUPPORTED, "E and block_m must be <= 1024");
    if (N * k + static_cast<int64_t>(E) * block_m >= (int64_t(1) << 31))
        return fail(MOE_ERR_UNSUPPORTED, "N*k + E*block_m must stay below 2^31");
    if (N == 0) return MOE_OK;
    if (!topk_ids || !sorted_pair || !block_expert || !counts || !offsets || !num_padded ||
        !workspace)
        return fail(MOE_ERR_INVALID_ARG, "every moe_align pointer must be non-null");
    const size_t need = moe_align_workspace_bytes(N, k, E, block_m);
    if (workspace_bytes < need)
        return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "align workspace needs %zu bytes, got %zu", need,
                    workspace_bytes);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    AlignBuffers b;
    b.status = reinterpret_cast<int32_t *>(ws);
    b.pad_offsets = reinterpret_cast<int32_t *>(ws + kAlign);
    b.scratch = reinterpret_cast<int32_t *>(ws + kAlign + round_up(sizeof(int32_t) * (E + 1), kAlign));
    b.sorted_pair = sorted_pair;
    b.block_expert = block_expert;
    b.counts = counts;
    b.offsets = offsets;
    b.num_padded = num_padded;
    MOE_CUDA(cudaMemsetAsync(b.status, 0, sizeof(int32_t), stream), "status reset");
    return enqueue_align(topk_ids, N, k, E, block_m, b, stream);
}

moe_status_t moe_forward_layout(int64_t N, int H, int E, int I, int k, int I_s,
                                moe_forward_layout_t *layout) {
    if (!layout) return fail(MOE_ERR_INVALID_ARG, "layout must be non-null");
    if (N < 0 || H < 1 || E < 1 || I < 1 || k < 1 || I_s < 0)
        return fail(MOE_ERR_INVALID_ARG, "bad sizes");
    return forward_layout(N, H, E, I, k, I_s, layout);
}

size_t moe_forward_workspace_bytes(int64_t N, int H, int E, int I, int k, int I_s) {
    moe_forward_layout_t L;
    if (N < 0 || H < 1 || E < 1 || I < 1 || k < 1 || I_s < 0) return 0;
    forward_layout(N, H, E, I, k, I_s, &L);
    return L.total;
}

// The whole layer; w_down / shared_down_proj are bf16 (down_f16 false) or
// their fp16 copies (down_f16 true).
static moe_status_t forward_impl(const moe_bf16_t *x, const moe_bf16_t *router,
                                 const moe_bf16_t *w_gate, const moe_bf16_t *w_up,
                                 const void *w_down, const moe_bf16_t *shared_gate_proj,
                                 const moe_bf16_t *shared_up_proj, const void *shared_down_proj,
                                 const moe_bf16_t *shared_gate, int64_t N, int H, int E, int I,
                                 int I_s, int k, int norm_topk_prob, bool down_f16,
                                 moe_bf16_t *out, void *workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
    g_last_error.clear();
    bool shared = false;
    moe_forward_layout_t L;
    moe_status_t st = check_forward_args(x, router, w_gate, w_up, w_down, shared_gate_proj,
                                         shared_up_proj, shared_down_proj, shared_gate, N, H, E,
                                         I, I_s, k, out, workspace, workspace_bytes, &shared, &L);
    if (st != MOE_OK || N == 0) return st;
    if (!shared) I_s = 0;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    auto at = [&](size_t off) { return ws + off; };
    int32_t *status = reinterpret_cast<int32_t *>(at(L.status));
    float *topk_w = reinterpret_cast<float *>(at(L.topk_w));
    int32_t *topk_ids = reinterpret_cast<int32_t *>(at(L.topk_ids));
    float *gamma = shared ? reinterpret_cast<float *>(at(L.gamma)) : nullptr;
    uint16_t *ypair = reinterpret_cast<uint16_t *>(at(L.ypair));
    int8_t *ypair_res = reinterpret_cast<int8_t *>(at(L.ypair_res));
    const int sms = num_sms_of_current_device();

    // K1: routing (its first CTA also clears the status word, so that no
    // memset node breaks the chain of programmatically serialized launches);
    // with the shared expert every token also gets its chunks' slots
    const int C = L.slots - k;
    if ((st = record_stage(MOE_STAGE_ROUTE, stream)) != MOE_OK) return st;
    const bool grouped = route_groups(N, E, shared);
    const AlignBuffers ab = align_buffers_of(L, ws);
    st = enqueue_route(x, router, shared ? shared_gate : nullptr, N, H, E, k, norm_topk_prob,
                       topk_w, topk_ids, nullptr, gamma, status, true, stream, C,
                       grouped ? &ab : nullptr, ready_count_of(L));
    if (st != MOE_OK) return st;

    // K2-K4: grouping, gate/up, down over the routed experts and the shared
    // expert's chunks together
    SharedWeights sw{shared_gate_proj, shared_up_proj, shared_down_proj, I_s, E};
    if ((st = enqueue_experts(x, topk_ids, topk_w, N, L.slots, H, L.groups, I, w_gate, w_up,
                              w_down, down_f16, L, ws, ypair, ypair_res, stream,
                              shared ? &sw : nullptr, grouped)) != MOE_OK)
        return st;
    // (the shared stage has no launches of its own any more)
    if ((st = record_stage(MOE_STAGE_SHARED, stream)) != MOE_OK) return st;

    // K5: out[n] = sum_j ypair[n*slots + j], the routed slots then the
    // shared expert's chunks
    if ((st = record_stage(MOE_STAGE_COMBINE, stream)) != MOE_OK) return st;
    MOE_CUDA(launch_combine(ypair, ypair_res, nullptr, N * L.slots, nullptr, nullptr, 0, N, H,
                            L.slots, out, sms, stream),
             "combine kernel launch");
    g_launches += 1;
    if ((st = record_stage(MOE_NUM_STAGES, stream)) != MOE_OK) return st;
    return MOE_OK;
}

moe_status_t moe_forward(const moe_bf16_t *x, const moe_bf16_t *router, const moe_bf16_t *w_gate,
                         const moe_bf16_t *w_up, const moe_bf16_t *w_down,
                         const moe_bf16_t *shared_gate_proj, const moe_bf16_t *shared_up_proj,
                         const moe_bf16_t *shared_down_proj, const moe_bf16_t *shared_gate,
                         int64_t N, int H, int E, int I, int I_s, int k, int norm_topk_prob,
                         moe_bf16_t *out, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
    return forward_impl(x, router, w_gate, w_up, w_down, shared_gate_proj, shared_up_proj,
                        shared_down_proj, shared_gate, N, H, E, I, I_s, k, norm_topk_prob, false,
                        out, workspace, workspace_bytes, stream);
}

moe_status_t moe_forward_prepared(const moe_bf16_t *x, const moe_bf16_t *router,
                                  const moe_bf16_t *w_gate, const moe_bf16_t *w_up,
                                  const moe_f16_t *w_down_f16,
                                  const moe_bf16_t *shared_gate_proj,
                                  const moe_bf16_t *shared_up_proj,
                                  const moe_f16_t *shared_down_proj_f16,
                                  const moe_bf16_t *shared_gate, int64_t N, int H, int E, int I,
                                  int I_s, int k, int norm_topk_prob, moe_bf16_t *out,
                                  void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return forward_impl(x, router, w_gate, w_up, w_down_f16, shared_gate_proj, shared_up_proj,
                        shared_down_proj_f16, shared_gate, N, H, E, I, I_s, k, norm_topk_prob,
                        true, out, workspace, workspace_bytes, stream);
}

// what moe_experts and moe_shared_expert use of moe_forward's layout: all but
// the pair-row planes, which they write to the caller's y
static size_t experts_workspace(int64_t N, int H, int E, int I, int k, int I_s) {
    moe_forward_layout_t L;
    forward_layout(N, H, E, I, k, I_s, &L);
    return L.ypair;
}

size_t moe_experts_workspace_bytes(int64_t R, int H, int E, int I) {
    if (R < 0 || H < 1 || E < 1 || I < 1) return 0;
    return experts_workspace(R, H, E, I, 1, 0);
}

static moe_status_t experts_impl(const moe_bf16_t *x_rows, const int32_t *ids,
                                 const float *weights, int64_t R, int H, int E, int I,
                                 const moe_bf16_t *w_gate, const moe_bf16_t *w_up,
                                 const void *w_down, bool down_f16, moe_bf16_t *y_hi,
                                 int8_t *y_res, void *workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
    g_last_error.clear();
    if (R < 0) return fail(MOE_ERR_INVALID_ARG, "R must be >= 0 (got %lld)", (long long)R);
    if (H < 8 || H % 8 || I < 8 || I % 8)
        return fail(MOE_ERR_INVALID_ARG, "H and I must be positive multiples of 8 (H=%d, I=%d)", H, I);
    if (E < 1 || E > MOE_MAX_EXPERTS)
        return fail(MOE_ERR_UNSUPPORTED, "E must be in [1, %d] (got %d)", MOE_MAX_EXPERTS, E);
    if (R == 0) return MOE_OK;
    if (!x_rows || !ids || !weights || !w_gate || !w_up || !w_down || !y_hi || !y_res ||
        !workspace)
        return fail(MOE_ERR_INVALID_ARG, "every moe_experts pointer must be non-null");
    if (!aligned16(x_rows) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
        !aligned16(y_hi) || !aligned16(y_res))
        return fail(MOE_ERR_INVALID_ARG, "matrices must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (R + static_cast<int64_t>(E) * kBlockM >= (int64_t(1) << 30))
        return fail(MOE_ERR_UNSUPPORTED, "R + E*128 must stay below 2^30");
    moe_forward_layout_t L;
    forward_layout(R, H, E, I, 1, 0, &L);
    if (workspace_bytes < L.ypair)
        return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "experts workspace needs %zu bytes, got %zu",
                    L.ypair, workspace_bytes);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    MOE_CUDA(cudaMemsetAsync(ws + L.status, 0, sizeof(int32_t), stream), "status reset");
    return enqueue_experts(x_rows, ids, weights, R, 1, H, E, I, w_gate, w_up, w_down, down_f16,
                           L, ws, y_hi, y_res, stream);
}

moe_status_t moe_experts(const moe_bf16_t *x_rows, const int32_t *ids, const float *weights,
                         int64_t R, int H, int E, int I, const moe_bf16_t *w_gate,
                         const moe_bf16_t *w_up, const moe_bf16_t *w_down, moe_bf16_t *y_hi,
                         int8_t *y_res, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
    return experts_impl(x_rows, ids, weights, R, H, E, I, w_gate, w_up, w_down, false, y_hi,
                        y_res, workspace, workspace_bytes, stream);
}

moe_status_t moe_experts_prepared(const moe_bf16_t *x_rows, const int32_t *ids,
                                  const float *weights, int64_t R, int H, int E, int I,
                                  const moe_bf16_t *w_gate, const moe_bf16_t *w_up,
                                  const moe_f16_t *w_down_f16, moe_bf16_t *y_hi, int8_t *y_res,
                                  void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return experts_impl(x_rows, ids, weights, R, H, E, I, w_gate, w_up, w_down_f16, true, y_hi,
                        y_res, workspace, workspace_bytes, stream);
}

int moe_shared_chunks(int I, int I_s) { return I >= 1 && I_s >= 1 ? shared_chunks(I, I_s) : 0; }

size_t moe_shared_expert_workspace_bytes(int64_t N, int H, int I, int I_s) {
    if (N < 0 || H < 1 || I < 1 || I_s < 1) return 0;
    return experts_workspace(N, H, 0, I, 0, I_s);
}

static moe_status_t shared_expert_impl(const moe_bf16_t *x, const float *shared_gamma, int64_t N,
                                       int H, int I, int I_s, const moe_bf16_t *shared_gate_proj,
                                       const moe_bf16_t *shared_up_proj,
                                       const void *shared_down_proj, bool down_f16,
                                       moe_bf16_t *y_hi, int8_t *y_res, void *workspace,
                                       size_t workspace_bytes, cudaStream_t stream) {
    g_last_error.clear();
    if (N < 0) return fail(MOE_ERR_INVALID_ARG, "N must be >= 0 (got %lld)", (long long)N);
    if (H < 8 || H % 8 || I < 8 || I % 8 || I_s < 8 || I_s % 8)
        return fail(MOE_ERR_INVALID_ARG,
                    "H, I and I_s must be positive multiples of 8 (H=%d, I=%d, I_s=%d)", H, I, I_s);
    const int C = shared_chunks(I, I_s);
    if (C > MOE_MAX_EXPERTS)
        return fail(MOE_ERR_UNSUPPORTED, "ceil(I_s / I) must be <= %d (got %d)", MOE_MAX_EXPERTS,
                    C);
    if (N == 0) return MOE_OK;
    if (!x || !shared_gamma || !shared_gate_proj || !shared_up_proj || !shared_down_proj ||
        !y_hi || !y_res || !workspace)
        return fail(MOE_ERR_INVALID_ARG, "every moe_shared_expert pointer must be non-null");
    if (!aligned16(x) || !aligned16(shared_gate_proj) || !aligned16(shared_up_proj) ||
        !aligned16(shared_down_proj) || !aligned16(y_hi) || !aligned16(y_res))
        return fail(MOE_ERR_INVALID_ARG, "matrices must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (N * C + static_cast<int64_t>(C) * kBlockM >= (int64_t(1) << 30))
        return fail(MOE_ERR_UNSUPPORTED, "N*C + C*128 must stay below 2^30");
    moe_forward_layout_t L;
    forward_layout(N, H, 0, I, 0, I_s, &L);
    if (workspace_bytes < L.ypair)
        return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "shared expert workspace needs %zu bytes, got %zu",
                    L.ypair, workspace_bytes);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *ids = reinterpret_cast<int32_t *>(ws + L.topk_ids);
    float *w = reinterpret_cast<float *>(ws + L.topk_w);
    MOE_CUDA(cudaMemsetAsync(ws + L.status, 0, sizeof(int32_t), stream), "status reset");
    MOE_CUDA(launch_shared_slots(shared_gamma, N, C, ids, w, num_sms_of_current_device(), stream),
             "shared slots kernel launch");
    g_launches += 1;
    SharedWeights sw{shared_gate_proj, shared_up_proj, shared_down_proj, I_s, 0};
    return enqueue_experts(x, ids, w, N, C, H, C, I, shared_gate_proj, shared_up_proj,
                           shared_down_proj, down_f16, L, ws, reinterpret_cast<uint16_t *>(y_hi),
                           y_res, stream, &sw);
}

moe_status_t moe_shared_expert(const moe_bf16_t *x, const float *shared_gamma, int64_t N, int H,
                               int I, int I_s, const moe_bf16_t *shared_gate_proj,
                               const moe_bf16_t *shared_up_proj,
                               const moe_bf16_t *shared_down_proj, moe_bf16_t *y_hi,
                               int8_t *y_res, void *workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
    return shared_expert_impl(x, shared_gamma, N, H, I, I_s, shared_gate_proj, shared_up_proj,
                              shared_down_proj, false, y_hi, y_res, workspace, workspace_bytes,
                              stream);
}

moe_status_t moe_shared_expert_prepared(const moe_bf16_t *x, const float *shared_gamma,
                                        int64_t N, int H, int I, int I_s,
                                        const moe_bf16_t *shared_gate_proj,
                                        const moe_bf16_t *shared_up_proj,
                                        const moe_f16_t *shared_down_proj_f16, moe_bf16_t *y_hi,
                                        int8_t *y_res, void *workspace, size_t workspace_bytes,
                                        cudaStream_t stream) {
    return shared_expert_impl(x, shared_gamma, N, H, I, I_s, shared_gate_proj, shared_up_proj,
                              shared_down_proj_f16, true, y_hi, y_res, workspace,
                              workspace_bytes, stream);
}

static moe_status_t combine_impl(const moe_bf16_t *ypair_hi, const int8_t *ypair_res,
                                 const int32_t *row_index, int64_t rows,
                                 const moe_bf16_t *yshared_hi, const int8_t *yshared_res,
                                 int shared_slots, int64_t N, int H, int k, moe_bf16_t *out,
                                 cudaStream_t stream) {
    g_last_error.clear();
    if (N < 0 || H < 8 || H % 8 || k < 1)
        return fail(MOE_ERR_INVALID_ARG, "need N >= 0, H a positive multiple of 8, k >= 1");
    if (N == 0) return MOE_OK;
    if (!ypair_hi || !ypair_res || !out)
        return fail(MOE_ERR_INVALID_ARG, "ypair_hi, ypair_res and out must be non-null");
    if ((yshared_hi == nullptr) != (yshared_res == nullptr))
        return fail(MOE_ERR_INVALID_ARG, "give both planes of yshared or neither");
    if (yshared_hi && (shared_slots < 1 || shared_slots > MOE_MAX_EXPERTS))
        return fail(MOE_ERR_INVALID_ARG, "shared_slots must be in [1, %d] with yshared (got %d)",
                    MOE_MAX_EXPERTS, shared_slots);
    if (!aligned16(ypair_hi) || !aligned16(ypair_res) || !aligned16(out) ||
        (yshared_hi && (!aligned16(yshared_hi) || !aligned16(yshared_res))))
        return fail(MOE_ERR_INVALID_ARG, "pair planes and out must be 16-byte aligned");
    if (N > (int64_t(1) << 31) / k) return fail(MOE_ERR_UNSUPPORTED, "N*k must stay below 2^31");
    if (rows < 0) return fail(MOE_ERR_INVALID_ARG, "num_rows must be >= 0");
    if (yshared_hi && N > (int64_t(1) << 31) / shared_slots)
        return fail(MOE_ERR_UNSUPPORTED, "N*shared_slots must stay below 2^31");
    MOE_CUDA(launch_combine(ypair_hi, ypair_res, row_index, rows, yshared_hi, yshared_res,
                            yshared_hi ? shared_slots : 0, N, H, k, out,
                            num_sms_of_current_device(), stream),
             "combine kernel launch");
    g_launches += 1;
    return MOE_OK;
}

moe_status_t moe_combine(const moe_bf16_t *ypair_hi, const int8_t *ypair_res,
                         const moe_bf16_t *yshared_hi, const int8_t *yshared_res,
                         int shared_slots, int64_t N, int H, int k, moe_bf16_t *out,
                         cudaStream_t stream) {
    return combine_impl(ypair_hi, ypair_res, nullptr, N * k, yshared_hi, yshared_res,
                        shared_slots, N, H, k, out, stream);
}

moe_status_t moe_combine_indexed(const moe_bf16_t *yrows_hi, const int8_t *yrows_res,
                                 int64_t num_rows, const int32_t *row_index,
                                 const moe_bf16_t *yshared_hi, const int8_t *yshared_res,
                                 int shared_slots, int64_t N, int H, int k, moe_bf16_t *out,
                                 cudaStream_t stream) {
    g_last_error.clear();
    if (N > 0 && !row_index) return fail(MOE_ERR_INVALID_ARG, "row_index must be non-null");
    if (N > 0 && num_rows > 0 && (!yrows_hi || !yrows_res))
        return fail(MOE_ERR_INVALID_ARG, "yrows_hi and yrows_res must be non-null");
    // nothing was sent (num_rows = 0): no row is read, so any aligned
    // stand-in address passes the checks below
    alignas(16) static const uint8_t kNone[16] = {};
    const moe_bf16_t *hi = num_rows > 0 ? yrows_hi : reinterpret_cast<const moe_bf16_t *>(kNone);
    const int8_t *res = num_rows > 0 ? yrows_res : reinterpret_cast<const int8_t *>(kNone);
    return combine_impl(hi, res, row_index, num_rows, yshared_hi, yshared_res, shared_slots, N, H,
                        k, out, stream);
}

// ------------------------------------------------- expert-parallel dispatch

// workspace: status | dest [P] | pad_offsets [R+1] | align scratch |
// order [P] | block owners [P] | offsets [R+1] | row count [1]
struct EpLayout {
    size_t status, dest, pad_offsets, scratch, order, owners, offsets, num_rows, total;
};

static EpLayout ep_layout(int64_t N, int k, int world) {
    const int64_t P = N * k;
    EpLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = round_up(off + bytes, kAlign);
        return at;
    };
    L.status = take(4);
    L.dest = take(sizeof(int32_t) * P);
    L.pad_offsets = take(sizeof(int32_t) * (world + 1));
    L.scratch = take(sizeof(int32_t) * static_cast<size_t>(align_chunks(P)) * world);
    L.order = take(sizeof(int32_t) * P);
    L.owners = take(sizeof(int32_t) * P);
    L.offsets = take(sizeof(int32_t) * (world + 1));
    L.num_rows = take(sizeof(int32_t));
    L.total = off;
    return L;
}

size_t moe_ep_dispatch_workspace_bytes(int64_t N, int k, int world) {
    if (N < 0 || k < 1 || world < 1) return 0;
    return ep_layout(N, k, world).total;
}

moe_status_t moe_ep_dispatch(const moe_bf16_t *x, const int32_t *topk_ids, const float *topk_w,
                             int64_t N, int H, int k, int E, int world, moe_bf16_t *send_x,
                             int32_t *send_ids, float *send_w, int32_t *send_counts,
                             int32_t *inv_order, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
    g_last_error.clear();
    if (N < 0 || H < 8 || H % 8 || k < 1 || E < 1 || world < 1)
        return fail(MOE_ERR_INVALID_ARG, "need N >= 0, H a positive multiple of 8, k, E, world >= 1");
    if (world > 1024) return fail(MOE_ERR_UNSUPPORTED, "world must be <= 1024");
    if (N > (int64_t(1) << 30) / k) return fail(MOE_ERR_UNSUPPORTED, "N*k must stay below 2^30");
    if (N == 0) return MOE_OK;
    if (!x || !topk_ids || !topk_w || !send_x || !send_ids || !send_w || !send_counts ||
        !inv_order || !workspace)
        return fail(MOE_ERR_INVALID_ARG, "every moe_ep_dispatch pointer must be non-null");
    if (!aligned16(x) || !aligned16(send_x))
        return fail(MOE_ERR_INVALID_ARG, "x and send_x must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const EpLayout L = ep_layout(N, k, world);
    if (workspace_bytes < L.total)
        return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "dispatch workspace needs %zu bytes, got %zu",
                    L.total, workspace_bytes);
    const int64_t P = N * k;
    const int e_local = (E + world - 1) / world;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    int32_t *dest = reinterpret_cast<int32_t *>(ws + L.dest);
    const int sms = num_sms_of_current_device();
    MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(int32_t), stream), "status reset");
    MOE_CUDA(launch_ep_dest(topk_ids, P, E, e_local, dest, inv_order, status, sms, stream),
             "dispatch kernel launch");
    g_launches += 1;
    // group the pairs by destination rank: moe_align's kernels with `world`
    // groups and blocks of one row (no padding: the grouped order is the
    // send order, the counts are the send counts)
    AlignBuffers b;
    b.sorted_pair = reinterpret_cast<int32_t *>(ws + L.order);
    b.block_expert = reinterpret_cast<int32_t *>(ws + L.owners);
    b.counts = send_counts;
    b.offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    b.pad_offsets = reinterpret_cast<int32_t *>(ws + L.pad_offsets);
    b.num_padded = reinterpret_cast<int32_t *>(ws + L.num_rows);
    b.scratch = reinterpret_cast<int32_t *>(ws + L.scratch);
    b.status = status;
    moe_status_t st = enqueue_align(dest, P, 1, world, 1, b, stream);
    if (st != MOE_OK) return st;
    MOE_CUDA(launch_ep_pack(x, topk_ids, topk_w, b.sorted_pair, b.num_padded, P, H, k, e_local,
                            send_x, send_ids, send_w, inv_order, sms, stream),
             "dispatch pack kernel launch");
    g_launches += 1;
    return MOE_OK;
}

moe_status_t moe_convert_bf16_to_f16(const moe_bf16_t *src, moe_f16_t *dst, int64_t n,
                                     int32_t *device_status, cudaStream_t stream) {
    g_last_error.clear();
    if (n < 0) return fail(MOE_ERR_INVALID_ARG, "n must be >= 0 (got %lld)", (long long)n);
    if (n == 0) return MOE_OK;
    if (!src || !dst) return fail(MOE_ERR_INVALID_ARG, "src and dst must be non-null");
    if (!aligned16(src) || !aligned16(dst))
        return fail(MOE_ERR_INVALID_ARG, "src and dst must be 16-byte aligned");
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
    const uintptr_t bytes = static_cast<uintptr_t>(n) * 2;
    if (s0 < d0 + bytes && d0 < s0 + bytes)
        return fail(MOE_ERR_INVALID_ARG, "src and dst must not overlap");
    MOE_CUDA(launch_convert_bf16_to_f16(src, dst, n, device_status, num_sms_of_current_device(),
                                        stream),
             "convert kernel launch");
    g_launches += 1;
    return MOE_OK;
}

}  // extern "C"

namespace moe {
// dst = src, bytes a multiple of 16, both 16-byte aligned device addresses
// (one of them may be mapped pinned host memory); waits for the previous
// kernel in the stream (convert.cu)
cudaError_t launch_copy16(const void *src, void *dst, size_t bytes, int num_sms, cudaStream_t s);
}  // namespace moe

extern "C" {

// The device address of pinned host memory mapped into the current device's
// address space, 16-byte aligned; null for anything else (pageable memory,
// unaligned buffers), which then takes cudaMemcpyAsync.
static void *mapped_device_pointer(const void *host) {
    if (!aligned16(host)) return nullptr;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, host) != cudaSuccess) {
        (void)cudaGetLastError();  // not a CUDA allocation: clear the error it left
        return nullptr;
    }
    if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return nullptr;
    return aligned16(attr.devicePointer) ? attr.devicePointer : nullptr;
}

static moe_status_t forward_host_impl(const moe_bf16_t *x_host, moe_bf16_t *out_host,
                                      moe_bf16_t *x_dev, moe_bf16_t *out_dev,
                                      const moe_bf16_t *router, const moe_bf16_t *w_gate,
                                      const moe_bf16_t *w_up, const void *w_down,
                                      const moe_bf16_t *shared_gate_proj,
                                      const moe_bf16_t *shared_up_proj,
                                      const void *shared_down_proj, const moe_bf16_t *shared_gate,
                                      int64_t N, int H, int E, int I, int I_s, int k,
                                      int norm_topk_prob, bool down_f16, void *workspace,
                                      size_t workspace_bytes, cudaStream_t stream) {
    g_last_error.clear();
    bool shared = false;
    moe_forward_layout_t L;
    moe_status_t st = check_forward_args(x_dev, router, w_gate, w_up, w_down, shared_gate_proj,
                                         shared_up_proj, shared_down_proj, shared_gate, N, H, E,
                                         I, I_s, k, out_dev, workspace, workspace_bytes, &shared,
                                         &L);
    if (st != MOE_OK || N == 0) return st;
    if (!x_host || !out_host)
        return fail(MOE_ERR_INVALID_ARG, "x_host and out_host must be non-null");
    const size_t bytes = static_cast<size_t>(N) * H * sizeof(moe_bf16_t);
    // pinned, mapped host buffers are copied by kernels on all SMs over the
    // CPU-GPU link; other host memory by the copy engines
    const int sms = num_sms_of_current_device();
    const void *x_map = mapped_device_pointer(x_host);
    void *out_map = mapped_device_pointer(out_host);
    if (x_map) {
        MOE_CUDA(launch_copy16(x_map, x_dev, bytes, sms, stream), "input copy kernel launch");
        g_launches += 1;
    } else {
        MOE_CUDA(cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, stream),
                 "input copy");
    }
    st = forward_impl(x_dev, router, w_gate, w_up, w_down, shared_gate_proj, shared_up_proj,
                      shared_down_proj, shared_gate, N, H, E, I, I_s, k, norm_topk_prob, down_f16,
                      out_dev, workspace, workspace_bytes, stream);
    if (st != MOE_OK) return st;
    if (out_map) {
        MOE_CUDA(launch_copy16(out_dev, out_map, bytes, sms, stream), "output copy kernel launch");
        g_launches += 1;
    } else {
        MOE_CUDA(cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, stream),
                 "output copy");
    }
    return MOE_OK;
}

moe_status_t moe_forward_host(const moe_bf16_t *x_host, moe_bf16_t *out_host, moe_bf16_t *x_dev,
                              moe_bf16_t *out_dev, const moe_bf16_t *router,
                              const moe_bf16_t *w_gate, const moe_bf16_t *w_up,
                              const moe_bf16_t *w_down, const moe_bf16_t *shared_gate_proj,
                              const moe_bf16_t *shared_up_proj,
                              const moe_bf16_t *shared_down_proj, const moe_bf16_t *shared_gate,
                              int64_t N, int H, int E, int I, int I_s, int k, int norm_topk_prob,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return forward_host_impl(x_host, out_host, x_dev, out_dev, router, w_gate, w_up, w_down,
                             shared_gate_proj, shared_up_proj, shared_down_proj, shared_gate, N,
                             H, E, I, I_s, k, norm_topk_prob, false, workspace, workspace_bytes,
                             stream);
}

moe_status_t moe_forward_host_prepared(
    const moe_bf16_t *x_host, moe_bf16_t *out_host, moe_bf16_t *x_dev, moe_bf16_t *out_dev,
    const moe_bf16_t *router, const moe_bf16_t *w_gate, const moe_bf16_t *w_up,
    const moe_f16_t *w_down_f16, const moe_bf16_t *shared_gate_proj,
    const moe_bf16_t *shared_up_proj, const moe_f16_t *shared_down_proj_f16,
    const moe_bf16_t *shared_gate, int64_t N, int H, int E, int I, int I_s, int k,
    int norm_topk_prob, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return forward_host_impl(x_host, out_host, x_dev, out_dev, router, w_gate, w_up, w_down_f16,
                             shared_gate_proj, shared_up_proj, shared_down_proj_f16, shared_gate,
                             N, H, E, I, I_s, k, norm_topk_prob, true, workspace,
                             workspace_bytes, stream);
}

// ----------------------------------------------------- add + RMSNorm

moe_status_t moe_add_rmsnorm(const moe_bf16_t *x, moe_bf16_t *residual, const moe_bf16_t *weight,
                             int64_t N, int H, float eps, int gemma, moe_bf16_t *normed,
                             cudaStream_t stream) {
    g_last_error.clear();
    if (N < 0) return fail(MOE_ERR_INVALID_ARG, "N must be >= 0");
    if (H < 8 || H % 8) return fail(MOE_ERR_INVALID_ARG, "H must be a positive multiple of 8 (got %d)", H);
    if (!(eps >= 0.f)) return fail(MOE_ERR_INVALID_ARG, "eps must be >= 0");
    if (N == 0) return MOE_OK;
    if (!x || !residual || !weight || !normed)
        return fail(MOE_ERR_INVALID_ARG, "x, residual, weight and normed must be non-null");
    if (!aligned16(x) || !aligned16(residual) || !aligned16(weight) || !aligned16(normed))
        return fail(MOE_ERR_INVALID_ARG, "bf16 arrays must be 16-byte aligned");
    MOE_CUDA(launch_add_rmsnorm(x, residual, weight, N, H, eps, gemma ? 1 : 0, normed,
                                num_sms_of_current_device(), stream),
             "add+rmsnorm kernel launch");
    g_launches += 1;
    return MOE_OK;
}

// ------------------------------------------------------------ dense MLP

size_t moe_dense_mlp_workspace_bytes(int64_t N, int H, int I) {
    if (N < 0 || H < 1 || I < 1) return 0;
    const size_t rows = static_cast<size_t>(round_up64(N, kBlockM));
    // the activation (fp16, or a bf16 hi/lo pair: 4 bytes a value reserved),
    // then the down projection as pair rows (bf16 hi plane, int8 residual)
    return kAlign + round_up(4 * rows * I, kAlign) + round_up(2 * static_cast<size_t>(N) * H, kAlign) +
           round_up(static_cast<size_t>(N) * H, kAlign);
}

static moe_status_t dense_mlp_impl(const moe_bf16_t *x, const moe_bf16_t *w_gate,
                                   const moe_bf16_t *w_up, const void *w_down, bool down_f16,
                                   int64_t N, int H, int I, moe_bf16_t *out, void *workspace,
                                   size_t workspace_bytes, cudaStream_t stream) {
    g_last_error.clear();
    if (N < 0) return fail(MOE_ERR_INVALID_ARG, "N must be >= 0");
    if (H < 8 || H % 8 || I < 8 || I % 8)
        return fail(MOE_ERR_INVALID_ARG, "H and I must be positive multiples of 8 (H=%d, I=%d)", H, I);
    if (N == 0) return MOE_OK;
    if (!x || !w_gate || !w_up || !w_down || !out || !workspace)
        return fail(MOE_ERR_INVALID_ARG, "every moe_dense_mlp pointer must be non-null");
    if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
        !aligned16(out))
        return fail(MOE_ERR_INVALID_ARG, "matrices must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (N >= (int64_t(1) << 30) - kBlockM) return fail(MOE_ERR_UNSUPPORTED, "N must stay below 2^30");
    const size_t need = moe_dense_mlp_workspace_bytes(N, H, I);
    if (workspace_bytes < need)
        return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "dense MLP workspace needs %zu bytes, got %zu", need,
                    workspace_bytes);
    const int64_t rows = round_up64(N, kBlockM);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    uint16_t *act = reinterpret_cast<uint16_t *>(ws + kAlign);
    uint16_t *y = reinterpret_cast<uint16_t *>(ws + kAlign + round_up(4 * rows * I, kAlign));
    int8_t *y_res = reinterpret_cast<int8_t *>(ws + kAlign + round_up(4 * rows * I, kAlign) +
                                               round_up(2 * static_cast<size_t>(N) * H, kAlign));
    const int sms = num_sms_of_current_device();
    const GemmMode down = down_f16 ? kDown : kDownSplit;
    const int64_t act_rows = down_f16 ? rows : 2 * rows;  // split: hi rows, then lo rows
    moe_status_t st;
    CUtensorMap tm_x, tm_g, tm_u, tm_act, tm_d;
    const int bn = choose_gate_up_bn(static_cast<double>(rows / kBlockM), static_cast<double>(N), I, sms);
    if ((st = make_map(&tm_x, x, H, N, H, kBlockK, kBlockM, "x")) != MOE_OK) return st;
    if ((st = make_map(&tm_g, w_gate, H, I, H, kBlockK, bn, "w_gate")) != MOE_OK) return st;
    if ((st = make_map(&tm_u, w_up, H, I, H, kBlockK, bn, "w_up")) != MOE_OK) return st;
    if ((st = make_map(&tm_act, act, I, act_rows, I, kBlockK, kBlockM, "act")) != MOE_OK) return st;
    if ((st = make_map(&tm_d, w_down, I, H, I, kBlockK, kDownBN, "w_down")) != MOE_OK) return st;
    MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(int32_t), stream), "status reset");
    // one dense group: every token row, weight 1
    GemmArgs g = {};
    g.virt_base = INT_MAX;  // no virtual experts
    g.sorted_pair = nullptr;
    g.block_expert = nullptr;
    g.num_padded = nullptr;
    g.num_rows_host = N;
    g.q_limit = N;
    g.k_div = 1;
    g.K = H;
    g.n_out = I;
    g.w_rows = I;
    g.out = act;
    g.out_res = nullptr;
    g.out_ld = I;
    g.lo_rows = down_f16 ? 0 : rows;
    g.scale = nullptr;
    g.status = status;
    g.stream_weights = N <= kBlockM ? 1 : 0;
    g.max_tiles = static_cast<int>(rows / kBlockM) * ((I + bn - 1) / bn);
    g.grid = g.max_tiles < sms ? g.max_tiles : sms;
    // more than one row block: two-CTA tiles over consecutive blocks
    const bool pairs = rows >= 2 * kBlockM;
    if (pairs) {
        const int bnp = pair_gemm_block_n(kGateUp);
        CUtensorMap tm_g2, tm_u2;
        if ((st = make_map(&tm_g2, w_gate, H, I, H, kBlockK, bnp, "w_gate")) != MOE_OK ||
            (st = make_map(&tm_u2, w_up, H, I, H, kBlockK, bnp, "w_up")) != MOE_OK)
            return st;
        g.max_tiles = static_cast<int>((rows / kBlockM + 1) / 2) * ((I + bnp - 1) / bnp);
        g.grid = 2 * (g.max_tiles < sms / 2 ? g.max_tiles : sms / 2);
        MOE_CUDA(launch_pair_gemm(kGateUp, tm_x, tm_g2, tm_u2, g, stream),
                 "dense gate/up kernel launch");
    } else {
        MOE_CUDA(launch_gemm(kGateUp, bn, tm_x, tm_x, tm_g, tm_u, g, stream),
                 "dense gate/up kernel launch");
    }
    g.K = I;
    g.n_out = H;
    g.w_rows = H;
    g.out = y;
    g.out_res = y_res;
    g.out_ld = H;
    if (pairs) {
        const int bnp = pair_gemm_block_n(down);
        CUtensorMap tm_d2;
        if ((st = make_map(&tm_d2, w_down, I, H, I, kBlockK, bnp / 2, "w_down")) != MOE_OK)
            return st;
        g.max_tiles = static_cast<int>((rows / kBlockM + 1) / 2) * ((H + bnp - 1) / bnp);
        g.grid = 2 * (g.max_tiles < sms / 2 ? g.max_tiles : sms / 2);
        MOE_CUDA(launch_pair_gemm(down, tm_act, tm_d2, tm_d2, g, stream),
                 "dense down kernel launch");
    } else {
        g.max_tiles = static_cast<int>(rows / kBlockM) * ((H + kDownBN - 1) / kDownBN);
        g.grid = g.max_tiles < sms ? g.max_tiles : sms;
        MOE_CUDA(launch_gemm(down, kDownBN, tm_act, tm_act, tm_d, tm_d, g, stream),
                 "dense down kernel launch");
    }
    // pair rows -> bf16 out (the combine with one slot per token)
    MOE_CUDA(launch_combine(y, y_res, nullptr, N, nullptr, nullptr, 0, N, H, 1, out, sms, stream),
             "combine kernel launch");
    g_launches += 3;
    return MOE_OK;
}

moe_status_t moe_dense_mlp(const moe_bf16_t *x, const moe_bf16_t *w_gate, const moe_bf16_t *w_up,
                           const moe_bf16_t *w_down, int64_t N, int H, int I, moe_bf16_t *out,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return dense_mlp_impl(x, w_gate, w_up, w_down, false, N, H, I, out, workspace,
                          workspace_bytes, stream);
}

moe_status_t moe_dense_mlp_prepared(const moe_bf16_t *x, const moe_bf16_t *w_gate,
                                    const moe_bf16_t *w_up, const moe_f16_t *w_down_f16,
                                    int64_t N, int H, int I, moe_bf16_t *out, void *workspace,
                                    size_t workspace_bytes, cudaStream_t stream) {
    return dense_mlp_impl(x, w_gate, w_up, w_down_f16, true, N, H, I, out, workspace,
                          workspace_bytes, stream);
}

moe_status_t moe_selftest_wait_timeout(void *workspace, size_t workspace_bytes,
                                       uint64_t limit_ns, cudaStream_t stream) {
    g_last_error.clear();
    if (!workspace || workspace_bytes < sizeof(int32_t))
        return fail(MOE_ERR_INVALID_ARG, "need a workspace of at least 4 bytes");
    if (limit_ns == 0 || limit_ns > 10000000000ull)
        return fail(MOE_ERR_INVALID_ARG, "limit_ns must be in (0, 10 s]");
    int32_t *status = static_cast<int32_t *>(workspace);
    MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(int32_t), stream), "status reset");
    MOE_CUDA(launch_wait_timeout_probe(status, limit_ns, stream), "self-test kernel launch");
    g_launches += 1;
    return MOE_OK;
}

moe_status_t moe_read_device_status(const void *workspace, cudaStream_t stream) {
    if (!workspace) return fail(MOE_ERR_INVALID_ARG, "workspace must be non-null");
    MOE_CUDA(cudaStreamSynchronize(stream), "stream synchronize");
    int32_t v = 0;
    MOE_CUDA(cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost), "status read");
    return static_cast<moe_status_t>(v);
}

}  // extern "C"
