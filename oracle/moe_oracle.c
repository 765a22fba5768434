/*
 * moe_oracle.c -- plain fp64 CPU oracle of the sparse MoE FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA library; it reads raw bf16 bit patterns and widens them itself.
 *
 * What it computes follows the pages on the method:
 *   - "M03 · Sparse MoE: routing, per-expert grouped compute, shared expert"
 *     (nano-vllm-omni drills, hints/m03_overview): the routing block of its
 *     problem overview (logits, fp32 softmax over all E experts, top-k,
 *     optional norm_topk_prob renorm, out[n] = sum_j w[n,j] Expert_ids(x[n]),
 *     Expert(h) = (silu(h Wg^T) * (h Wu^T)) Wd^T), its shared-expert line
 *     (out += sigmoid(x g^T) * SharedMLP(x), scalar gate) and its grouping
 *     bookkeeping walk-through (flatten, stable sort, counts, prefix starts).
 *   - "Nano-vLLM notes" (lshu.cn), section "Qwen3MoeSparseMoeBlock": the same
 *     routing in HF form (softmax in fp32, topk, renorm, cast).
 *   - the FusedMoE "moe_align_block_size" step named in the M03 shape-trace
 *     section: pad each expert's segment to the GEMM block size.
 *
 * Precision: every arithmetic step is fp64; inputs are the exact bf16 values
 * the GPU receives, widened without rounding.  Top-k is taken on the
 * probabilities in descending order, ties going to the lower expert index.
 *
 * Parity pins (tests/test_oracle_pins.py): the printed worked examples of the
 * M03 drill (bookkeeping, route I/O, scalar end-to-end, shared expert),
 * brute force over all experts with a top-k mask, closed forms (E=k=1 is a
 * dense SwiGLU; k=E with renorm gives the full softmax; renormalised weights
 * equal a softmax over the top-k logits), numpy's stable argsort for the
 * grouping order, and batch invariance.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* dot(row of bf16 matrix, fp64 vector) */
static double dot_bf16(const uint16_t *row, const double *v, int64_t len)
{
    double s = 0.0;
    for (int64_t i = 0; i < len; ++i)
        s += widen_bf16(row[i]) * v[i];
    return s;
}

/*
 * Routing of one token (M03 problem overview, routing block):
 *   logits = x @ router^T                  (all E experts)
 *   probs  = softmax(logits) over all E    (exp(l - max) / sum exp(l - max))
 *   w, ids = topk(probs, k), descending    (ties -> lower expert index)
 *   if norm: w /= sum_j w
 * logits_out / probs_out may be NULL.
 */
static void route_token(const double *xd, const uint16_t *router, int H, int E,
                        int k, int norm, double *logits, double *probs,
                        char *taken, double *w_out, int32_t *ids_out)
{
    double mx = -INFINITY;
    for (int e = 0; e < E; ++e) {
        logits[e] = dot_bf16(router + (int64_t)e * H, xd, H);
        if (logits[e] > mx) mx = logits[e];
    }
    double den = 0.0;
    for (int e = 0; e < E; ++e) {
        probs[e] = exp(logits[e] - mx);
        den += probs[e];
    }
    for (int e = 0; e < E; ++e) probs[e] /= den;

    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e]) continue;
            /* strict '>' while scanning e upwards keeps the lower index on ties */
            if (best < 0 || probs[e] > probs[best]) best = e;
        }
        taken[best] = 1;
        ids_out[j] = best;
        w_out[j] = probs[best];
    }
    if (norm) {
        double s = 0.0;
        for (int j = 0; j < k; ++j) s += w_out[j];
        for (int j = 0; j < k; ++j) w_out[j] /= s;
    }
}

/*
 * One SwiGLU expert applied to one token (M03: Expert(h) =
 * (silu(h Wg^T) * (h Wu^T)) Wd^T with Wg, Wu [I, H] and Wd [H, I]).
 * Adds scale * Expert(x) into acc[H].  a is scratch of length I.
 */
static void swiglu_add(const double *xd, const uint16_t *wg, const uint16_t *wu,
                       const uint16_t *wd, int H, int I, double scale,
                       double *a, double *acc)
{
    for (int i = 0; i < I; ++i) {
        double g = dot_bf16(wg + (int64_t)i * H, xd, H);
        double u = dot_bf16(wu + (int64_t)i * H, xd, H);
        a[i] = silu(g) * u;
    }
    for (int h = 0; h < H; ++h)
        acc[h] += scale * dot_bf16(wd + (int64_t)h * I, a, I);
}

/* ------------------------------------------------------------------------ */
/* route: all N tokens                                                       */
/* ------------------------------------------------------------------------ */

int oracle_route(const uint16_t *x, const uint16_t *router, int64_t N, int H,
                 int E, int k, int norm, double *logits_out, double *probs_out,
                 double *topk_w, int32_t *topk_ids)
{
    if (N < 0 || H < 1 || E < 1 || k < 1 || k > E) return 1;
    double *xd = malloc(sizeof(double) * (size_t)H);
    double *lg = malloc(sizeof(double) * (size_t)E);
    double *pr = malloc(sizeof(double) * (size_t)E);
    char *taken = malloc((size_t)E);
    if (!xd || !lg || !pr || !taken) { free(xd); free(lg); free(pr); free(taken); return 2; }
    for (int64_t n = 0; n < N; ++n) {
        for (int h = 0; h < H; ++h) xd[h] = widen_bf16(x[n * H + h]);
        route_token(xd, router, H, E, k, norm, lg, pr, taken, topk_w + n * k,
                    topk_ids + n * k);
        if (logits_out) memcpy(logits_out + n * E, lg, sizeof(double) * (size_t)E);
        if (probs_out) memcpy(probs_out + n * E, pr, sizeof(double) * (size_t)E);
    }
    free(xd); free(lg); free(pr); free(taken);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* align: the grouping bookkeeping of the M03 walk-through, plus FusedMoE's   */
/* padding of every expert segment to the GEMM block size BM.                 */
/* ------------------------------------------------------------------------ */

/*
 * ids      [N*k]   expert id of pair p = n*k + j (row-major flatten)
 * counts   [E]     bincount of ids
 * offsets  [E+1]   exclusive prefix sum of counts (segment starts in order)
 * order    [P]     stable argsort of the pairs by expert
 * sorted_pair [cap] padded layout: expert e's pairs (ascending p) start at
 *                  pad_off[e] = sum_{e'<e} round_up(counts[e'], BM), followed
 *                  by the sentinel P up to the next multiple of BM.
 * block_expert [cap/BM]  owner expert of each BM-row block
 * num_padded [1]   pad_off[E]
 * Slots at or beyond num_padded are left untouched.
 */
int oracle_align(const int32_t *ids, int64_t N, int k, int E, int BM,
                 int32_t *counts, int32_t *offsets, int32_t *order,
                 int32_t *sorted_pair, int64_t cap, int32_t *block_expert,
                 int32_t *num_padded)
{
    if (N < 0 || k < 1 || E < 1 || BM < 1) return 1;
    const int64_t P = N * (int64_t)k;
    for (int64_t p = 0; p < P; ++p)
        if (ids[p] < 0 || ids[p] >= E) return 3;

    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t p = 0; p < P; ++p) counts[ids[p]] += 1;

    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];

    /* stable grouping: for each expert in turn, its pairs in ascending p */
    int64_t w = 0;
    for (int e = 0; e < E; ++e)
        for (int64_t p = 0; p < P; ++p)
            if (ids[p] == e) order[w++] = (int32_t)p;

    int64_t pad = 0;
    for (int e = 0; e < E; ++e) {
        int64_t c = counts[e];
        int64_t seg = (c + BM - 1) / BM * BM;
        if (pad + seg > cap) return 4;
        for (int64_t i = 0; i < seg; ++i)
            sorted_pair[pad + i] = (i < c) ? order[offsets[e] + i] : (int32_t)P;
        for (int64_t b = pad / BM; b < (pad + seg) / BM; ++b) block_expert[b] = e;
        pad += seg;
    }
    *num_padded = (int32_t)pad;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* forward: the plain per-token definition, for a chosen subset of tokens    */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *x, *router, *wg, *wu, *wd, *sg, *su, *sd, *sgate;
    int64_t N;
    int H, E, I, Is, k, norm;
    const int64_t *rows;
    int64_t r0, r1;
    double *out;
    int status;
} fwd_job;

static void *forward_rows(void *arg)
{
    fwd_job *J = (fwd_job *)arg;
    const int H = J->H, E = J->E, I = J->I, Is = J->Is, k = J->k;
    int amax = I > Is ? I : Is;
    double *xd = malloc(sizeof(double) * (size_t)H);
    double *lg = malloc(sizeof(double) * (size_t)E);
    double *pr = malloc(sizeof(double) * (size_t)E);
    double *a = malloc(sizeof(double) * (size_t)(amax > 0 ? amax : 1));
    double *w = malloc(sizeof(double) * (size_t)k);
    int32_t *ids = malloc(sizeof(int32_t) * (size_t)k);
    char *taken = malloc((size_t)E);
    if (!xd || !lg || !pr || !a || !w || !ids || !taken) {
        J->status = 2;
        goto done;
    }
    for (int64_t r = J->r0; r < J->r1; ++r) {
        int64_t n = J->rows[r];
        double *acc = J->out + r * H;
        if (n < 0 || n >= J->N) { J->status = 3; goto done; }
        for (int h = 0; h < H; ++h) xd[h] = widen_bf16(J->x[n * H + h]);
        for (int h = 0; h < H; ++h) acc[h] = 0.0;

        route_token(xd, J->router, H, E, k, J->norm, lg, pr, taken, w, ids);
        /* out[n] = sum_j w[n,j] * Expert_{ids[n,j]}(x[n]), accumulated */
        for (int j = 0; j < k; ++j) {
            int64_t e = ids[j];
            swiglu_add(xd, J->wg + e * (int64_t)I * H, J->wu + e * (int64_t)I * H,
                       J->wd + e * (int64_t)H * I, H, I, w[j], a, acc);
        }
        /* shared expert: out += sigmoid(x . g) * SharedMLP(x) */
        if (J->sg) {
            double gamma = sigmoid(dot_bf16(J->sgate, xd, H));
            swiglu_add(xd, J->sg, J->su, J->sd, H, Is, gamma, a, acc);
        }
    }
done:
    free(xd); free(lg); free(pr); free(a); free(w); free(ids); free(taken);
    return NULL;
}

/* ------------------------------------------------------------------------ */
/* fused residual add + RMSNorm (the decoder layer's step before the MoE)    */
/* ------------------------------------------------------------------------ */

/* IEEE binary32 -> bf16 bits, round to nearest even (finite inputs). */
static uint16_t round_to_bf16(double v)
{
    float f = (float)v; /* exact for the sums formed below (see caller) */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/*
 * Nano-vLLM notes (question 4 on the decoder layer) and the Qwen3.5
 * walkthrough (section 2.1): hidden = hidden + residual; residual = hidden;
 * hidden = norm(hidden), with RMSNorm(r) = r / sqrt(mean(r^2) + eps) * w
 * (Qwen3 tutorial, RMSNorm section) or, when gemma != 0, * (1 + w)
 * (GemmaRMSNorm, walkthrough section 2.1).  The add happens in the model's
 * bf16 dtype: r = bf16(x + residual) is the new residual and the norm's input.
 *   residual_out [N, H] bf16 bits;  normed [N, H] fp64 (before any rounding)
 */
int oracle_add_rmsnorm(const uint16_t *x, const uint16_t *residual, const uint16_t *w,
                       int64_t N, int H, double eps, int gemma, uint16_t *residual_out,
                       double *normed)
{
    if (N < 0 || H < 1 || eps < 0) return 1;
    double *r = malloc(sizeof(double) * (size_t)H);
    if (!r) return 2;
    for (int64_t n = 0; n < N; ++n) {
        double ss = 0.0;
        for (int h = 0; h < H; ++h) {
            /* the sum of two bf16 values is exact in binary32 unless their
             * exponents differ by more than 16, where the smaller one is far
             * below half a bf16 ulp and cannot change the rounded result */
            uint16_t b = round_to_bf16(widen_bf16(x[n * H + h]) + widen_bf16(residual[n * H + h]));
            residual_out[n * H + h] = b;
            r[h] = widen_bf16(b);
            ss += r[h] * r[h];
        }
        double inv = 1.0 / sqrt(ss / H + eps);
        for (int h = 0; h < H; ++h) {
            double wh = widen_bf16(w[h]);
            normed[n * H + h] = r[h] * inv * (gemma ? 1.0 + wh : wh);
        }
    }
    free(r);
    return 0;
}

int oracle_hardware_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * out[r, :] = MoE(x[rows[r], :]) for r < n_rows, in fp64.
 * The shared expert is present iff all four shared pointers are non-NULL.
 * nthreads <= 0 uses every online core.  Rows are split into contiguous
 * ranges, one per thread; each row is computed exactly as above.
 */
int oracle_moe_forward(const uint16_t *x, const uint16_t *router,
                       const uint16_t *w_gate, const uint16_t *w_up,
                       const uint16_t *w_down, const uint16_t *s_gate_proj,
                       const uint16_t *s_up_proj, const uint16_t *s_down_proj,
                       const uint16_t *s_gate, int64_t N, int H, int E, int I,
                       int I_s, int k, int norm, const int64_t *rows,
                       int64_t n_rows, double *out, int nthreads)
{
    if (N < 0 || H < 1 || E < 1 || I < 1 || k < 1 || k > E || n_rows < 0) return 1;
    int nshared = (s_gate_proj != 0) + (s_up_proj != 0) + (s_down_proj != 0) + (s_gate != 0);
    if (nshared != 0 && nshared != 4) return 1;
    if (nshared == 4 && I_s < 1) return 1;
    if (n_rows == 0) return 0;
    if (nthreads <= 0) nthreads = oracle_hardware_threads();
    if (nthreads > n_rows) nthreads = (int)n_rows;

    fwd_job *jobs = calloc((size_t)nthreads, sizeof(fwd_job));
    pthread_t *th = calloc((size_t)nthreads, sizeof(pthread_t));
    char *started = calloc((size_t)nthreads, 1);
    if (!jobs || !th || !started) { free(jobs); free(th); free(started); return 2; }
    int64_t per = (n_rows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        fwd_job *J = &jobs[t];
        J->x = x; J->router = router; J->wg = w_gate; J->wu = w_up; J->wd = w_down;
        J->sg = nshared ? s_gate_proj : NULL; J->su = s_up_proj; J->sd = s_down_proj;
        J->sgate = s_gate;
        J->N = N; J->H = H; J->E = E; J->I = I; J->Is = I_s; J->k = k; J->norm = norm;
        J->rows = rows; J->out = out;
        J->r0 = t * per;
        J->r1 = (t + 1) * per < n_rows ? (t + 1) * per : n_rows;
        if (J->r0 >= J->r1) continue;
        if (nthreads > 1 && pthread_create(&th[t], NULL, forward_rows, J) == 0)
            started[t] = 1;
        else
            forward_rows(J); /* single thread, or no thread to be had */
    }
    int status = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (started[t]) pthread_join(th[t], NULL);
        if (jobs[t].status) status = jobs[t].status;
    }
    free(jobs); free(th); free(started);
    return status;
}
