/*
 * oracle.c -- plain, slow, fp64 CPU reference for MLA tree-verify attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this file's library.  It shares
 * no code, header, table or helper with the CUDA path and includes nothing
 * from it.
 *
 * What it computes (the step the pages call "verify attention"):
 *   The Milestone Commit, "Input Knowledge Required": the kernel computes
 *   attention of the draft tokens against the full KV cache.  The Checkpoint
 *   Report, "Input Knowledge Required": DDTree builds a tree of draft tokens
 *   which the target model verifies in one pass; "Mistakes and Incorrect
 *   Assumptions": in the extend layout the prefix keys come first, the draft
 *   tokens' own KV follows, and each draft row of the mask has stride
 *   prefix + q_len.  The Milestone Commit, "Context": the cache is the MLA
 *   latent cache, one shared row per token addressed with page_size=1.
 *
 * Readings (the pages give no formula):
 *   - a key row is 576 bf16: 512 latent columns followed by 64 rotary columns;
 *     the value is the first 512 columns of the same row;
 *   - score s_j = sm_scale * <q, k_j> over all 576 columns;
 *   - node i sees every prefix key and the tree keys of itself and its
 *     ancestors (parent < i, -1 = hangs off the prefix);
 *   - lse = m + ln(sum_j exp(s_j - m)), natural log of scaled logits;
 *   - out = sum_j exp(s_j - lse) * v_j.
 *   Everything is evaluated in double precision from bf16 inputs widened
 *   exactly.  A key whose slot is outside the pool is skipped.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 -> double, exact: a bf16 is the top half of an IEEE binary32. */
static double widen_bf16(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Ancestor-or-self sets of a draft tree.
 * The Checkpoint Report, "Mistakes and Incorrect Assumptions" (mask rows of
 * the draft tokens) and "Input Knowledge Required" (DDTree draft tree).
 * parent[i] must satisfy -1 <= parent[i] < i (nodes in topological order).
 * A node with an invalid parent is treated as hanging off the prefix (it sees
 * only itself among the tree keys) and is counted in the return value.
 * T <= 64 so that one node's set fits in a 64-bit word.
 */
int oracle_tree_bits(const int32_t *parent, int T, uint64_t *bits)
{
    int bad = 0;
    /* nodes are in topological order, so a node's set is its own bit plus
       the (already built) set of its parent */
    for (int i = 0; i < T; ++i) {
        uint64_t set = 1ull << i;
        int p = parent[i];
        if (p < -1 || p >= i) ++bad;
        else if (p >= 0) set |= bits[p];
        bits[i] = set;
    }
    return bad;
}

typedef struct {
    const uint16_t *q;        /* [B*T, H, D] bf16 bits                    */
    const uint16_t *kv;       /* [num_slots, row_stride] bf16 bits        */
    int64_t num_slots, row_stride;
    const int32_t *slots;     /* per request: N_b slots, prefix then tree */
    const int64_t *indptr;    /* [B+1] offsets into slots                 */
    const int32_t *prefix;    /* [B]                                      */
    const uint64_t *bits;     /* [B, T]                                   */
    int B, T, H, D, Dv;
    double sm_scale;
    int64_t k0, k1;           /* key window [k0, k1) within each request  */
    const int64_t *rows;      /* optional list of rows to evaluate        */
    int64_t nrows;
    double *out;              /* [rows, Dv]                               */
    double *lse;              /* [rows]                                   */
    int nthreads, tid;
    int64_t skipped;          /* keys skipped for an out-of-range slot    */
} job_t;

/* Is key j of request b visible to draft node i? */
static int visible(const job_t *J, int b, int i, int64_t j)
{
    int64_t P = J->prefix[b];
    if (j < P) return 1;
    int64_t k = j - P;
    if (k >= J->T) return 0;
    return (int)((J->bits[(int64_t)b * J->T + i] >> k) & 1ull);
}

/* One output row: request b, node i, head h -> out[Dv], lse. */
static int64_t one_row(const job_t *J, int64_t row, double *out, double *lse,
                       double *score, int64_t *keys)
{
    int64_t TH = (int64_t)J->T * J->H;
    int b = (int)(row / TH);
    int i = (int)((row / J->H) % J->T);
    const uint16_t *qr = J->q + row * J->D;
    int64_t N = (int64_t)J->prefix[b] + J->T;
    int64_t lo = J->k0 < 0 ? 0 : J->k0;
    int64_t hi = J->k1 < N ? J->k1 : N;
    int64_t n = 0, skipped = 0;

    /* pass 1: scores of every visible key */
    for (int64_t j = lo; j < hi; ++j) {
        if (!visible(J, b, i, j)) continue;
        int64_t s = J->slots[J->indptr[b] + j];
        if (s < 0 || s >= J->num_slots) { ++skipped; continue; }
        const uint16_t *kr = J->kv + s * J->row_stride;
        double dot = 0.0;
        for (int d = 0; d < J->D; ++d) dot += widen_bf16(qr[d]) * widen_bf16(kr[d]);
        score[n] = J->sm_scale * dot;
        keys[n] = s;
        ++n;
    }
    for (int d = 0; d < J->Dv; ++d) out[d] = 0.0;
    if (n == 0) { *lse = -INFINITY; return skipped; }

    double m = score[0];
    for (int64_t t = 1; t < n; ++t) if (score[t] > m) m = score[t];
    double z = 0.0;
    for (int64_t t = 0; t < n; ++t) z += exp(score[t] - m);
    double L = m + log(z);
    *lse = L;

    /* pass 2: softmax-weighted sum of the value columns */
    for (int64_t t = 0; t < n; ++t) {
        double w = exp(score[t] - L);
        const uint16_t *vr = J->kv + keys[t] * J->row_stride;
        for (int d = 0; d < J->Dv; ++d) out[d] += w * widen_bf16(vr[d]);
    }
    return skipped;
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    int64_t maxN = 0;
    for (int b = 0; b < J->B; ++b) {
        int64_t N = (int64_t)J->prefix[b] + J->T;
        if (N > maxN) maxN = N;
    }
    double *score = (double *)malloc(sizeof(double) * (size_t)(maxN + 1));
    int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(maxN + 1));
    int64_t total = J->rows ? J->nrows : (int64_t)J->B * J->T * J->H;
    J->skipped = 0;
    for (int64_t r = J->tid; r < total; r += J->nthreads) {
        int64_t row = J->rows ? J->rows[r] : r;
        J->skipped += one_row(J, row, J->out + r * J->Dv, J->lse + r, score, keys);
    }
    free(score);
    free(keys);
    return NULL;
}

/*
 * Masked softmax attention for every (request, node, head) row, or for the
 * rows listed in `rows` (nrows of them; outputs are packed in list order).
 * Only keys with index in [k0, k1) of each request are used: [0, INT64_MAX)
 * is the whole step, a narrower window is one split of the key range.
 * Returns the number of keys skipped for an out-of-range slot (summed over
 * rows), or -1 on an argument error.
 */
int64_t oracle_verify_attn(const uint16_t *q, const uint16_t *kv, int64_t num_slots,
                           int64_t row_stride, const int32_t *slots, const int64_t *indptr,
                           const int32_t *prefix_len, const uint64_t *bits, int B, int T, int H,
                           int D, int Dv, double sm_scale, int64_t k0, int64_t k1,
                           const int64_t *rows, int64_t nrows, double *out, double *lse,
                           int nthreads)
{
    if (!q || !kv || !slots || !indptr || !prefix_len || !bits || !out || !lse) return -1;
    if (B < 1 || T < 1 || T > 64 || H < 1 || D < Dv || Dv < 1 || row_stride < D) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) {
        job_t *J = &jobs[t];
        J->q = q; J->kv = kv; J->num_slots = num_slots; J->row_stride = row_stride;
        J->slots = slots; J->indptr = indptr; J->prefix = prefix_len; J->bits = bits;
        J->B = B; J->T = T; J->H = H; J->D = D; J->Dv = Dv; J->sm_scale = sm_scale;
        J->k0 = k0; J->k1 = k1; J->rows = rows; J->nrows = nrows;
        J->out = out; J->lse = lse; J->nthreads = nthreads; J->tid = t;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, worker, &jobs[t]);
    worker(&jobs[0]);
    int64_t skipped = jobs[0].skipped;
    for (int t = 1; t < nthreads; ++t) {
        pthread_join(th[t], NULL);
        skipped += jobs[t].skipped;
    }
    free(jobs);
    free(th);
    return skipped;
}

/*
 * Merge of split partials.  The Commit That Locked In 6x Decode, "Input
 * Knowledge Required" (NSPLIT and partial-reduce) and The Milestone Commit,
 * "The Deeper Significance" (the reduction kernel).  Each part s holds a
 * normalised partial output o_s[Dv] and its lse_s over a disjoint key subset;
 *   lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s.
 * Parts with lse_s = -inf (no visible key) carry no weight.
 */
void oracle_lse_merge(int nparts, const double *lse_parts, const double *o_parts, int Dv,
                      double *out, double *lse)
{
    double m = -INFINITY;
    for (int s = 0; s < nparts; ++s) if (lse_parts[s] > m) m = lse_parts[s];
    for (int d = 0; d < Dv; ++d) out[d] = 0.0;
    if (m == -INFINITY) { *lse = -INFINITY; return; }
    double z = 0.0;
    for (int s = 0; s < nparts; ++s)
        if (lse_parts[s] != -INFINITY) z += exp(lse_parts[s] - m);
    double L = m + log(z);
    for (int s = 0; s < nparts; ++s) {
        if (lse_parts[s] == -INFINITY) continue;
        double w = exp(lse_parts[s] - L);
        for (int d = 0; d < Dv; ++d) out[d] += w * o_parts[(int64_t)s * Dv + d];
    }
    *lse = L;
}

/*
 * KV defragmentation: copy each request's scattered rows into a contiguous
 * destination range.  The Checkpoint Report, "Input Knowledge Required"
 * (defragmentation keeps per-request KV contiguous) and "The Architecture of
 * the Report" (the deferred defragmentation phase).  Reading: out of place,
 * row i of request b goes to dst_base[b] + i and its slot entry is rewritten
 * to that row.  Rows are copied whole (row_stride elements).
 */
int oracle_defrag(uint16_t *pool, int64_t num_slots, int64_t row_stride, const int32_t *src,
                  const int64_t *indptr, const int64_t *dst_base, int B, int32_t *slots_out)
{
    for (int b = 0; b < B; ++b) {
        for (int64_t i = 0; indptr[b] + i < indptr[b + 1]; ++i) {
            int64_t s = src[indptr[b] + i];
            int64_t d = dst_base[b] + i;
            if (s < 0 || s >= num_slots || d < 0 || d >= num_slots) return -1;
            memmove(pool + d * row_stride, pool + s * row_stride,
                    sizeof(uint16_t) * (size_t)row_stride);
            if (slots_out) slots_out[indptr[b] + i] = (int32_t)d;
        }
    }
    return 0;
}
