/*
 * Oracle for EAGLE target-verify attention at speculative topk = 1.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, plainly correct CPU
 * statement of what the verify-attention path computes. Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it. It shares no
 * code, header, table or helper with the CUDA library under
 * speculative_decoding_verify_topk_gb300/csrc, and it includes nothing from it.
 *
 * Sources (titles of the pull-request pages the method is taken from):
 *  - "Split-KV flash-decode attention for EAGLE target-verify (Triton backend)",
 *    Motivation / Modifications: at topk = 1 the EAGLE draft tree is a chain,
 *    so verification is plain causal attention of the draft-token queries over
 *    the sequence's KV prefix plus the drafts themselves; splitting the prefix
 *    and merging partial results by log-sum-exp is an exact reorganisation of
 *    the same softmax.
 *  - "Support Page Size > 1 (when top k = 1) for FA3 Spec Decode": at topk = 1
 *    the tokens of a sequence are consecutive in its page table, so logical
 *    token j lives in page table entry j / page_size at offset j % page_size.
 *  - "Enable EAGLE speculative decoding ... with aiter's unified attention",
 *    review of the target-verify call: paged K/V pools are viewed as
 *    [pages, page_size, kv_heads, head_dim], the output as
 *    [tokens, q_heads, v_head_dim] (v_head_dim, not qk_head_dim), and a sliding
 *    window is passed as a left bound (window, -1).
 *
 * Readings taken where the pages are silent (each one is also a test pin):
 *  - seq_lens[b] is the committed prefix length P_b; the D_b draft tokens'
 *    K/V sit in the same paged cache at logical positions P_b .. P_b+D_b-1.
 *  - Query row i of sequence b sits at position p = P_b + i and sees keys
 *    j in [lo, p] with lo = max(0, p - window) when window >= 0, else 0
 *    (causal including the diagonal; the window counts window+1 keys).
 *  - GQA: q-head h reads kv-head h / (Hq / Hkv) (contiguous groups).
 *  - The page table is CSR over pages: sequence b's logical page k is
 *    page_table[kv_indptr[b] + k].
 *  - lse is the natural logarithm of sum_j exp(scale * q . k_j).
 *  - Absorbed MLA (v_aliases_k): V is the first Dv entries of the K row.
 *  - FP8 KV ("Split-KV flash-decode attention for EAGLE target-verify (Triton
 *    backend)", Modifications: the prefix stage applies the fp8 k_scale /
 *    v_scale dequant multipliers as the extend kernel does): pools stored as
 *    FP8 E4M3 hold K / scale and V / scale per tensor; K = k_scale * stored,
 *    V = v_scale * stored, and q stays in its 16-bit type.
 *  - Tree verify (topk > 1, the follow-up the split-KV page defers; its
 *    baseline applies the tree's custom mask): when tree_mask is given, row i
 *    of sequence b sees every prefix key 0 .. P_b - 1 and the draft key
 *    P_b + d exactly when bit d of tree_mask[qoff_b + i] is set (d < D_b; an
 *    EAGLE tree row sees its ancestors and itself); the drafts keep their
 *    logical positions P_b .. P_b + D_b - 1 in the page table. A sliding window
 *    is not defined for tree rows (window must be < 0). A row that sees no key
 *    at all gives out = 0 and lse = -inf.
 *
 * Arithmetic: every input element is decoded to double exactly (fp32, bf16
 * and fp16 all embed exactly in binary64), and all sums, the exponentials and
 * the logarithm are taken in double.
 *
 * num_splits <= 1 evaluates the softmax in one pass over the allowed keys:
 * m = max_j s_j, lse = m + log sum_j exp(s_j - m), o = sum_j exp(s_j - lse) v_j.
 * num_splits = S > 1 cuts the allowed key range [lo, p] into S contiguous,
 * near-equal pieces, computes each piece's normalised partial (o_s, lse_s) the
 * same way, and merges them: lse = log sum_s exp(lse_s),
 * o = sum_s exp(lse_s - lse) o_s. An empty piece contributes nothing. This is
 * the split-KV + log-sum-exp merge of the split-KV page, written out so that
 * the merge itself can be checked against the single pass.
 *
 * Build with: cc -O2 -fopenmp -shared -fPIC -o liboracle.so verify_attn_oracle.c -lm
 * Defining ORACLE_MUTANT=n at compile time plants one deliberate mistake
 * (see the #if blocks); the test suite builds those variants to show that its
 * pins catch each of them. The default build plants nothing.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2, ORACLE_FP8_E4M3 = 3 };

enum {
    ORACLE_OK = 0,
    ORACLE_BAD_ARG = 1,
    ORACLE_BAD_PAGE = 2,      /* a page id outside [0, num_pages) */
    ORACLE_SHORT_TABLE = 3,   /* fewer page-table entries than the KV needs */
    ORACLE_NO_MEMORY = 4
};

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);                 /* subnormal: frac * 2^-24 */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(frac | 0x400), expo - 25); /* (1.frac) * 2^(e-15) */
    return sign ? -mag : mag;
}

/* bfloat16 is the top half of a binary32. */
static double decode_bf16(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits,
 * no infinities; exponent 15 with fraction 7 is NaN, every other pattern is a
 * number (so the largest is 1.75 * 2^8 = 448).
 */
static double decode_e4m3(uint8_t x)
{
    int sign = (x >> 7) & 1;
    int expo = (x >> 3) & 0xf;
    int frac = x & 0x7;
    double mag;
    if (expo == 15 && frac == 7)
        mag = NAN;
    else if (expo == 0)
        mag = ldexp((double)frac, -9);                  /* subnormal: frac/8 * 2^-6 */
    else
        mag = ldexp((double)(frac | 0x8), expo - 10);   /* (1.frac) * 2^(e-7) */
    return sign ? -mag : mag;
}

/* Exported for the decoder pin (all 256 codes against an independent decoder). */
double oracle_decode_e4m3(int x) { return decode_e4m3((uint8_t)x); }

static double elem(const void *base, int dtype, int64_t idx)
{
    switch (dtype) {
    case ORACLE_F32: return (double)((const float *)base)[idx];
    case ORACLE_BF16: return decode_bf16(((const uint16_t *)base)[idx]);
    case ORACLE_FP8_E4M3: return decode_e4m3(((const uint8_t *)base)[idx]);
    default: return decode_f16(((const uint16_t *)base)[idx]);
    }
}

typedef struct {
    int bs, hq, hkv, dqk, dv, page_size, dtype, kv_dtype, v_aliases_k, window, num_splits;
    int64_t num_pages;
    double scale, k_scale, v_scale;
    const void *q, *k, *v;
    const int32_t *page_table, *kv_indptr, *seq_lens, *num_draft;
    const uint32_t *tree_mask;   /* NULL: causal */
    const int64_t *qoff;
} problem;

/* Physical token slot of logical position j of sequence b (64-bit). */
static int64_t slot_of(const problem *pb, int b, int64_t j)
{
    int64_t page = pb->page_table[(int64_t)pb->kv_indptr[b] + j / pb->page_size];
#if ORACLE_MUTANT == 4
    return page * pb->page_size; /* planted: drops the in-page offset */
#else
    return page * pb->page_size + j % pb->page_size;
#endif
}

static int kv_head_of(const problem *pb, int h)
{
#if ORACLE_MUTANT == 2
    return h % pb->hkv; /* planted: interleaved instead of contiguous groups */
#else
    return h / (pb->hq / pb->hkv);
#endif
}

/* Dequantised K / V elements: the stored value times the per-tensor scale. */
static double key_elem(const problem *pb, int64_t slot, int g, int d)
{
    return pb->k_scale * elem(pb->k, pb->kv_dtype, (slot * pb->hkv + g) * pb->dqk + d);
}

static double value_elem(const problem *pb, int64_t slot, int g, int d)
{
#if ORACLE_MUTANT == 12
    const double vs = 1.0; /* planted: the V scale dropped */
#else
    const double vs = pb->v_scale;
#endif
    if (pb->v_aliases_k)
        return vs * elem(pb->k, pb->kv_dtype, (slot * pb->hkv + g) * pb->dqk + d);
#if ORACLE_MUTANT == 9
    return vs * elem(pb->k, pb->kv_dtype, (slot * pb->hkv + g) * pb->dqk + d); /* planted: V read from K */
#else
    return vs * elem(pb->v, pb->kv_dtype, (slot * pb->hkv + g) * pb->dv + d);
#endif
}

/*
 * Softmax attention of one query row over keys [j0, j1) (j1 > j0), given the
 * row's scores s[j - lo]. Writes the normalised output o[Dv] and returns lse.
 */
static double attend_range(const problem *pb, int b, int g, const double *s,
                           int64_t lo, int64_t j0, int64_t j1, double *o)
{
    double m = -INFINITY, sum = 0.0, lse;
    int64_t j;
    int d;
    for (j = j0; j < j1; ++j)
        if (s[j - lo] > m) m = s[j - lo];
    if (m == -INFINITY) { /* no visible key in the range (tree rows only) */
        for (d = 0; d < pb->dv; ++d) o[d] = 0.0;
        return -INFINITY;
    }
    for (j = j0; j < j1; ++j)
        sum += exp(s[j - lo] - m);
#if ORACLE_MUTANT == 5
    lse = log(sum); /* planted: forgets to add the running max back */
#else
    lse = m + log(sum);
#endif
    for (d = 0; d < pb->dv; ++d) o[d] = 0.0;
    for (j = j0; j < j1; ++j) {
        double w = exp(s[j - lo] - lse);
        int64_t slot = slot_of(pb, b, j);
        for (d = 0; d < pb->dv; ++d) o[d] += w * value_elem(pb, slot, g, d);
    }
    return lse;
}

/* One output row (b, i, h): out_row[Dv], *lse_out. Returns an ORACLE_ code. */
static int one_row(const problem *pb, int b, int i, int h, double *out_row, double *lse_out,
                   double *s)
{
    int g = kv_head_of(pb, h);
    int64_t p = (int64_t)pb->seq_lens[b] + i;
    int64_t lo = 0, j, n;
    int d;
#if ORACLE_MUTANT == 7
    const int64_t qrow = (int64_t)i * pb->hq + h; /* planted: ignores earlier sequences' rows */
#else
    const int64_t qrow = (pb->qoff[b] + i) * pb->hq + h;
#endif
#if ORACLE_MUTANT == 1
    int64_t hi = p;     /* planted: excludes the diagonal (strictly causal) */
#else
    int64_t hi = p + 1; /* exclusive end: keys lo .. p */
#endif
#if ORACLE_MUTANT == 6
    if (pb->window >= 0) lo = p - pb->window + 1 > 0 ? p - pb->window + 1 : 0; /* planted: W keys, not W+1 */
#else
    if (pb->window >= 0) lo = p - pb->window > 0 ? p - pb->window : 0;
#endif
    if (pb->tree_mask) hi = (int64_t)pb->seq_lens[b] + pb->num_draft[b]; /* the mask picks the drafts */
    n = hi - lo;
    if (n <= 0) { /* only reachable through a planted mistake */
        for (d = 0; d < pb->dv; ++d) out_row[d] = NAN;
        *lse_out = NAN;
        return ORACLE_OK;
    }
    for (j = lo; j < hi; ++j) {
        int64_t slot = slot_of(pb, b, j);
        double dot = 0.0;
        if (pb->tree_mask && j >= pb->seq_lens[b]) {
            const uint32_t bits = pb->tree_mask[pb->qoff[b] + i];
#if ORACLE_MUTANT == 10
            const int64_t dj = j - pb->seq_lens[b] + 1; /* planted: bit index off by one */
#else
            const int64_t dj = j - pb->seq_lens[b];
#endif
#if ORACLE_MUTANT == 11
            const int seen = j <= p; /* planted: ignores the tree, keeps the causal chain */
#else
            const int seen = dj < 32 && ((bits >> dj) & 1u);
#endif
            if (!seen) { s[j - lo] = -INFINITY; continue; }
        }
        for (d = 0; d < pb->dqk; ++d)
            dot += elem(pb->q, pb->dtype, qrow * pb->dqk + d) * key_elem(pb, slot, kv_head_of(pb, h), d);
#if ORACLE_MUTANT == 3
        s[j - lo] = dot; /* planted: drops the softmax scale */
#else
        s[j - lo] = pb->scale * dot;
#endif
    }
    if (pb->num_splits <= 1) {
        *lse_out = attend_range(pb, b, g, s, lo, lo, hi, out_row);
        return ORACLE_OK;
    }
    {
        /* Piece k covers [lo + k*n/S, lo + (k+1)*n/S): contiguous, near-equal. */
        int S = pb->num_splits, k;
        double big = -INFINITY, acc = 0.0, lse;
        double *lse_s = (double *)malloc(sizeof(double) * (size_t)S);
        double *o_s = (double *)malloc(sizeof(double) * (size_t)S * (size_t)pb->dv);
        if (!lse_s || !o_s) { free(lse_s); free(o_s); return ORACLE_NO_MEMORY; }
        for (k = 0; k < S; ++k) {
            int64_t a = lo + (n * k) / S, e = lo + (n * (k + 1)) / S;
            if (e > a) {
                lse_s[k] = attend_range(pb, b, g, s, lo, a, e, o_s + (size_t)k * pb->dv);
            } else {
                lse_s[k] = -INFINITY; /* empty piece: weight zero */
                for (d = 0; d < pb->dv; ++d) o_s[(size_t)k * pb->dv + d] = 0.0;
            }
            if (lse_s[k] > big) big = lse_s[k];
        }
        if (big == -INFINITY) { /* no visible key at all */
            for (d = 0; d < pb->dv; ++d) out_row[d] = 0.0;
            *lse_out = -INFINITY;
            free(lse_s);
            free(o_s);
            return ORACLE_OK;
        }
        for (k = 0; k < S; ++k) acc += exp(lse_s[k] - big);
        lse = big + log(acc);
        for (d = 0; d < pb->dv; ++d) out_row[d] = 0.0;
        for (k = 0; k < S; ++k) {
#if ORACLE_MUTANT == 8
            double w = lse_s[k] > -INFINITY ? 1.0 / S : 0.0; /* planted: unweighted merge */
#else
            double w = exp(lse_s[k] - lse);
#endif
            if (w == 0.0) continue;
            for (d = 0; d < pb->dv; ++d) out_row[d] += w * o_s[(size_t)k * pb->dv + d];
        }
        *lse_out = lse;
        free(lse_s);
        free(o_s);
    }
    return ORACLE_OK;
}

/*
 * Checks the page table before anything is read: every sequence needs
 * ceil((P_b + D_b) / page_size) entries and every entry it uses must name a
 * page of the pool.
 */
static int check_tables(const problem *pb)
{
    int b;
    for (b = 0; b < pb->bs; ++b) {
        int64_t t = (int64_t)pb->seq_lens[b] + pb->num_draft[b];
        int64_t need = (t + pb->page_size - 1) / pb->page_size, k;
        if (pb->seq_lens[b] < 0 || pb->num_draft[b] < 0) return ORACLE_BAD_ARG;
        if ((int64_t)pb->kv_indptr[b + 1] - pb->kv_indptr[b] < need) return ORACLE_SHORT_TABLE;
        for (k = 0; k < need; ++k) {
            int64_t page = pb->page_table[(int64_t)pb->kv_indptr[b] + k];
            if (page < 0 || page >= pb->num_pages) return ORACLE_BAD_PAGE;
        }
    }
    return ORACLE_OK;
}

/*
 * Computes the verify-attention rows.
 *
 * Layouts (row-major, contiguous):
 *   q           [sum_b D_b, hq, dqk]   rows grouped by sequence, drafts in order
 *   k_cache     [num_pages, page_size, hkv, dqk]
 *   v_cache     [num_pages, page_size, hkv, dv]   (ignored when v_aliases_k)
 *   page_table  int32, CSR over pages; kv_indptr int32 [bs + 1]
 *   seq_lens    int32 [bs] prefix lengths; num_draft int32 [bs]
 *   dtype       0 fp32, 1 bf16, 2 fp16: q (and k_cache / v_cache unless kv_dtype says
 *               otherwise)
 *   kv_dtype    -1: same as dtype; 3: FP8 E4M3 pools (bytes)
 *   k_scale, v_scale  per-tensor dequantisation scales: K = k_scale * stored,
 *               V = v_scale * stored (1.0 for unquantised pools); the split-KV page
 *               applies them in the prefix stage exactly as the extend kernel does
 *   window      < 0: no window (required with tree_mask)
 *   tree_mask   NULL: causal rows; else uint32 [sum D_b], bit d of row i's word:
 *               the row sees draft d (tree verify)
 *   rows        NULL: compute every (b, i, h) into out [sum D_b, hq, dv] and
 *               lse [sum D_b, hq]; otherwise n_rows triples (b, i, h) and the
 *               results go to out [n_rows, dv], lse [n_rows].
 *   threads     0: OpenMP default
 * Returns 0 on success, otherwise an ORACLE_ code and writes nothing useful.
 */
int oracle_verify_attn(int bs, int hq, int hkv, int dqk, int dv, int page_size, int dtype,
                       int kv_dtype, double k_scale, double v_scale,
                       const void *q, const void *k_cache, const void *v_cache, int v_aliases_k,
                       const int32_t *page_table, const int32_t *kv_indptr, int64_t num_pages,
                       const int32_t *seq_lens, const int32_t *num_draft, double scale, int window,
                       const uint32_t *tree_mask, int num_splits, const int32_t *rows, int64_t n_rows,
                       double *out, double *lse, int threads)
{
    problem pb;
    int64_t *qoff, total_q = 0, r, nr;
    int64_t max_keys = 1;
    int b, status = ORACLE_OK;

    if (bs < 0 || hq <= 0 || hkv <= 0 || hq % hkv != 0 || dqk <= 0 || dv <= 0 || page_size <= 0)
        return ORACLE_BAD_ARG;
    if (dtype < ORACLE_F32 || dtype > ORACLE_F16) return ORACLE_BAD_ARG;
    if (kv_dtype < 0) kv_dtype = dtype;
    if (kv_dtype < ORACLE_F32 || kv_dtype > ORACLE_FP8_E4M3) return ORACLE_BAD_ARG;
    if (v_aliases_k && dv > dqk) return ORACLE_BAD_ARG;
    if (tree_mask && window >= 0) return ORACLE_BAD_ARG;
    if (bs == 0) return ORACLE_OK;

    pb.bs = bs; pb.hq = hq; pb.hkv = hkv; pb.dqk = dqk; pb.dv = dv;
    pb.page_size = page_size; pb.dtype = dtype; pb.v_aliases_k = v_aliases_k;
    pb.kv_dtype = kv_dtype; pb.k_scale = k_scale; pb.v_scale = v_scale;
    pb.window = window; pb.num_splits = num_splits; pb.num_pages = num_pages;
    pb.scale = scale; pb.q = q; pb.k = k_cache; pb.v = v_cache;
    pb.page_table = page_table; pb.kv_indptr = kv_indptr;
    pb.seq_lens = seq_lens; pb.num_draft = num_draft; pb.tree_mask = tree_mask;

    status = check_tables(&pb);
    if (status != ORACLE_OK) return status;

    qoff = (int64_t *)malloc(sizeof(int64_t) * ((size_t)bs + 1));
    if (!qoff) return ORACLE_NO_MEMORY;
    for (b = 0; b < bs; ++b) {
        int64_t t = (int64_t)seq_lens[b] + num_draft[b];
        qoff[b] = total_q;
        total_q += num_draft[b];
        if (t > max_keys) max_keys = t;
    }
    qoff[bs] = total_q;
    pb.qoff = qoff;

    nr = rows ? n_rows : total_q * hq;
    if (rows) {
        for (r = 0; r < nr; ++r) {
            int rb = rows[3 * r], ri = rows[3 * r + 1], rh = rows[3 * r + 2];
            if (rb < 0 || rb >= bs || ri < 0 || ri >= num_draft[rb] || rh < 0 || rh >= hq) {
                free(qoff);
                return ORACLE_BAD_ARG;
            }
        }
    }

    /* the thread count of this call only (a num_threads clause, so a
     * one-thread call leaves later calls on the default count) */
#ifdef _OPENMP
    const int nthreads = threads > 0 ? threads : omp_get_max_threads();
#else
    (void)threads;
#endif

#pragma omp parallel num_threads(nthreads)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)max_keys);
        int local = (s == NULL) ? ORACLE_NO_MEMORY : ORACLE_OK;
        int64_t rr;
#pragma omp for schedule(dynamic, 4)
        for (rr = 0; rr < nr; ++rr) {
            int rb, ri, rh;
            int64_t dst;
            if (local != ORACLE_OK) continue;
            if (rows) {
                rb = rows[3 * rr]; ri = rows[3 * rr + 1]; rh = rows[3 * rr + 2];
                dst = rr;
            } else {
                /* rr = (global query row) * hq + h; find its sequence */
                int64_t gq = rr / hq;
                int lo_b = 0, hi_b = bs - 1;
                while (lo_b < hi_b) { /* last b with qoff[b] <= gq */
                    int mid = (lo_b + hi_b + 1) / 2;
                    if (qoff[mid] <= gq) lo_b = mid; else hi_b = mid - 1;
                }
                while (num_draft[lo_b] == 0 || qoff[lo_b] + num_draft[lo_b] <= gq) ++lo_b;
                rb = lo_b; ri = (int)(gq - qoff[lo_b]); rh = (int)(rr % hq);
                dst = rr;
            }
            local = one_row(&pb, rb, ri, rh, out + dst * dv, lse + dst, s);
        }
        free(s);
#pragma omp critical
        if (local != ORACLE_OK) status = local;
    }
    free(qoff);
    return status;
}

/* Threads an OpenMP parallel region of this library actually gets. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }
