/*
 * Plain fp64 CPU oracle for the ModernBERT-base bidirectional attention block.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may load, link or
 * call this file.  It exists so that the CUDA library can be checked against
 * an independent, slow, obviously correct statement of what the block
 * computes.  Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline
 * and reference legs may use it.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * Sources (page title, section):
 *  - "ModernBERT-base Architecture Teardown" (kgptalkie), "How Does
 *    Self-Attention Work?": scores are q.k divided by sqrt(head size), a
 *    softmax along the keys makes every row sum to 1, the output is the
 *    weighted blend of the value rows; an encoder uses no causal mask.
 *  - same page, "How Does ModernBERT Make Q, K and V?": the fused Wqkv output
 *    of 2304 numbers per token is viewed as (3, 12, 64): Q, K, V, each split
 *    head by head into 12 heads of 64.
 *  - same page, "What Are Local and Global Attention?": a local layer lets a
 *    token see the 64 tokens on each side of it and itself (129 keys in the
 *    interior, fewer at the ends); a global layer sees every token.
 *  - same page, "How Does RoPE Work With Two Bases?": pair i turns by
 *    base^(-2i/64) radians per token; base 160000 on global layers, 10000 on
 *    local layers.
 *  - "ModernBERT" (candding), "The two rope tables": rotate-half convention
 *    over the full 64-wide head; positions count from 0 in every row.
 *  - "ModernBERT" (candding), "The alternating attention": key j is kept for
 *    query i when |i - j| <= 64, inclusive.
 *  - "Encoder-only models" (rayaq), padding mask: padded keys get -inf before
 *    the softmax, so real outputs are unchanged.  Here every packed sequence
 *    is its own attention problem; keys of other sequences are never seen.
 *
 * Readings where the pages are silent:
 *  - rotation sign: y = x*cos(phi) + rotate_half(x)*sin(phi) with
 *    rotate_half(x) = (-x[32..63], x[0..31]), i.e. pair m = (x[m], x[m+32])
 *    is multiplied by exp(+i*phi) when read as the complex number
 *    x[m] + i*x[m+32].
 *  - the frequencies, angles, cos/sin and every sum are evaluated in fp64.
 *  - bf16 inputs are widened to fp64 exactly; the output is left unrounded.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (see build.py in
 * this folder).  -ffp-contract=off keeps every a*b+c a separate multiply and
 * add, so the results are the same on x86 and on Arm.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* element conversion                                                  */
/* ------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; widening it is exact. */
static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round x to the nearest bf16 value (8 significant bits), ties to even.
 * frexp gives x = m * 2^e with 0.5 <= |m| < 1; m * 2^8 rounded to an integer
 * (nearbyint, the default round-to-nearest-even mode) keeps 8 significant
 * bits.  Zero, infinities and NaN pass through; the bf16 overflow and
 * subnormal ranges are not modelled (no input here reaches them). */
double oracle_round_bf16(double x)
{
    if (x == 0.0 || !isfinite(x))
        return x;
    int e;
    double m = frexp(x, &e);
    return ldexp(nearbyint(ldexp(m, 8)), e - 8);
}

/* oracle_round_bf16 over n values. */
void oracle_round_bf16_n(const double *x, int64_t n, double *y)
{
    for (int64_t i = 0; i < n; i++)
        y[i] = oracle_round_bf16(x[i]);
}

/* ------------------------------------------------------------------ */
/* RoPE                                                                */
/* ------------------------------------------------------------------ */

/* inv_freq[m] = theta^(-2m/head_dim), m = 0 .. head_dim/2 - 1
 * (teardown, "How Does RoPE Work With Two Bases?"). */
void oracle_inv_freq(double theta, int head_dim, double *inv_freq)
{
    for (int m = 0; m < head_dim / 2; m++)
        inv_freq[m] = pow(theta, -2.0 * (double)m / (double)head_dim);
}

/* Rotate one head row x[head_dim] sitting at position pos: pair m is
 * (x[m], x[m + head_dim/2]) and turns by pos * inv_freq[m] radians
 * (candding, "The two rope tables": rotate-half over the full head). */
void oracle_rope_row(const double *x, int64_t pos, double theta, int head_dim,
                     double *y)
{
    const int half = head_dim / 2;
    for (int m = 0; m < half; m++) {
        double inv = pow(theta, -2.0 * (double)m / (double)head_dim);
        double phi = (double)pos * inv;
        double c = cos(phi), s = sin(phi);
        double a = x[m], b = x[m + half];
        y[m] = a * c - b * s;
        y[m + half] = b * c + a * s;
    }
}

/* oracle_rope_row over n rows x[n][head_dim], row r at position pos[r]. */
void oracle_rope_rows(const double *x, int64_t n, const int64_t *pos, double theta,
                      int head_dim, double *y)
{
    for (int64_t r = 0; r < n; r++)
        oracle_rope_row(x + r * head_dim, pos[r], theta, head_dim, y + r * head_dim);
}

/* ------------------------------------------------------------------ */
/* the admitted key set                                                */
/* ------------------------------------------------------------------ */

/* Is key position j visible to query position i in a sequence of length L?
 * half_window < 0 means a global layer (every key of the sequence);
 * otherwise |i - j| <= half_window, inclusive (candding, "The alternating
 * attention"; teardown, "What Are Local and Global Attention?"). */
static int oracle_admitted(int64_t i, int64_t j, int64_t L, int half_window)
{
    if (j < 0 || j >= L)
        return 0;
    if (half_window < 0)
        return 1;
    int64_t d = i > j ? i - j : j - i;
    return d <= (int64_t)half_window;
}

/* First and one-past-last key position of the admitted set of query i.
 * The set is an interval; oracle_key_counts below re-derives its size from
 * the predicate alone. */
static void admitted_range(int64_t i, int64_t L, int half_window,
                           int64_t *j0, int64_t *j1)
{
    if (half_window < 0) {
        *j0 = 0;
        *j1 = L;
        return;
    }
    int64_t lo = i - half_window, hi = i + half_window + 1;
    *j0 = lo < 0 ? 0 : lo;
    *j1 = hi > L ? L : hi;
}

static int check_cu(const int32_t *cu, int n_seqs, int64_t T)
{
    if (n_seqs < 0 || cu == NULL)
        return -1;
    if (cu[0] != 0)
        return -2;
    for (int s = 0; s < n_seqs; s++)
        if (cu[s + 1] < cu[s])
            return -3;
    if ((int64_t)cu[n_seqs] != T)
        return -4;
    return 0;
}

/* |A_i| for every packed row, by testing the predicate against every key of
 * the row's own sequence (brute force, O(sum L^2)). */
int oracle_key_counts(const int32_t *cu, int n_seqs, int64_t T, int half_window,
                      int32_t *counts)
{
    int rc = check_cu(cu, n_seqs, T);
    if (rc)
        return rc;
    for (int s = 0; s < n_seqs; s++) {
        int64_t L = cu[s + 1] - cu[s];
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < L; i++) {
            int32_t c = 0;
            for (int64_t j = 0; j < L; j++)
                c += oracle_admitted(i, j, L, half_window);
            counts[cu[s] + i] = c;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* softmax and blend                                                   */
/* ------------------------------------------------------------------ */

/* Two-pass softmax over n scores (max, then sum of exp), followed by the
 * value blend o = sum_j w_j v_j.  vrow(j) is row j of the values; w may be
 * NULL.  Teardown, "How Does Self-Attention Work?": rows of weights sum to 1
 * and the output is the weighted blend of the values. */
typedef const double *(*vrow_fn)(void *ctx, int64_t j);

static void softmax_blend(const double *scores, int64_t n, int dv,
                          vrow_fn vrow, void *ctx, double *w, double *o)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; j++)
        if (scores[j] > m)
            m = scores[j];
    double den = 0.0;
    for (int64_t j = 0; j < n; j++)
        den += exp(scores[j] - m);
    for (int d = 0; d < dv; d++)
        o[d] = 0.0;
    for (int64_t j = 0; j < n; j++) {
        double wj = exp(scores[j] - m) / den;
        if (w)
            w[j] = wj;
        const double *v = vrow(ctx, j);
        for (int d = 0; d < dv; d++)
            o[d] += wj * v[d];
    }
}

/* ------------------------------------------------------------------ */
/* generic dense core: softmax(scale * Q K^T + mask) V                   */
/* ------------------------------------------------------------------ */

struct dense_ctx { const double *V; const int64_t *idx; int dv; };

static const double *dense_vrow(void *p, int64_t j)
{
    struct dense_ctx *c = (struct dense_ctx *)p;
    return c->V + c->idx[j] * c->dv;
}

/* Q[n][d], K[m][d], V[m][dv]; mask[n][m] (1 = keep) or NULL (keep all).
 * weights[n][m] (masked entries 0) and out[n][dv].  A row whose mask keeps
 * nothing gets zero weights and a zero output.  This is the worked example
 * of the teardown's "How Does Self-Attention Work?" section in general form. */
int oracle_sdpa_dense(const double *Q, const double *K, const double *V,
                      int64_t n, int64_t m, int d, int dv, double scale,
                      const uint8_t *mask, double *weights, double *out)
{
    if (n < 0 || m < 0 || d <= 0 || dv <= 0)
        return -1;
    double *sc = (double *)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
    double *wk = (double *)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
    int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * (size_t)(m > 0 ? m : 1));
    if (!sc || !wk || !idx) {
        free(sc); free(wk); free(idx);
        return -2;
    }
    struct dense_ctx ctx = { V, idx, dv };
    for (int64_t i = 0; i < n; i++) {
        int64_t k = 0;
        for (int64_t j = 0; j < m; j++) {
            if (mask && !mask[i * m + j])
                continue;
            double acc = 0.0;
            for (int e = 0; e < d; e++)
                acc += Q[i * d + e] * K[j * d + e];
            sc[k] = acc * scale;
            idx[k] = j;
            k++;
        }
        for (int64_t j = 0; j < m; j++)
            weights[i * m + j] = 0.0;
        if (k == 0) {
            for (int e = 0; e < dv; e++)
                out[i * dv + e] = 0.0;
            continue;
        }
        softmax_blend(sc, k, dv, dense_vrow, &ctx, wk, out + i * dv);
        for (int64_t t = 0; t < k; t++)
            weights[i * m + idx[t]] = wk[t];
    }
    free(sc); free(wk); free(idx);
    return 0;
}

/* ------------------------------------------------------------------ */
/* the attention block over packed variable-length sequences            */
/* ------------------------------------------------------------------ */

/* Per (sequence, head) working state: rotated keys, computed on first use
 * and reused by every query of that (sequence, head), and the value rows
 * in fp64. */
struct seq_ctx {
    const uint16_t *qkv;
    int64_t row0;          /* packed row of position 0 */
    int64_t L;
    int width;             /* 3 * heads * head_dim */
    int heads, head_dim, h;
    double theta;
    int round_operands;    /* rotated q and k rounded to bf16 (see below) */
    double *krot;          /* [L][head_dim] */
    unsigned char *kdone;  /* [L] */
    double *vbuf;          /* [L][head_dim] */
    unsigned char *vdone;  /* [L] */
};

static const double *seq_vrow_from(struct seq_ctx *c, int64_t j)
{
    double *v = c->vbuf + j * c->head_dim;
    if (!c->vdone[j]) {
        /* V block starts at column 2 * heads * head_dim; head h at h*head_dim */
        const uint16_t *src = c->qkv + (c->row0 + j) * c->width
                              + 2 * c->heads * c->head_dim + c->h * c->head_dim;
        for (int e = 0; e < c->head_dim; e++)
            v[e] = bf16_to_f64(src[e]);
        c->vdone[j] = 1;
    }
    return v;
}

static const double *seq_krot(struct seq_ctx *c, int64_t j)
{
    double *k = c->krot + j * c->head_dim;
    if (!c->kdone[j]) {
        double raw[256];
        const uint16_t *src = c->qkv + (c->row0 + j) * c->width
                              + c->heads * c->head_dim + c->h * c->head_dim;
        for (int e = 0; e < c->head_dim; e++)
            raw[e] = bf16_to_f64(src[e]);
        oracle_rope_row(raw, j, c->theta, c->head_dim, k);
        if (c->round_operands)
            for (int e = 0; e < c->head_dim; e++)
                k[e] = oracle_round_bf16(k[e]);
        c->kdone[j] = 1;
    }
    return k;
}

/* The admitted keys of one query are the interval [j0, j1); softmax_blend
 * sees them as 0 .. j1-j0-1. */
struct range_ctx { struct seq_ctx *c; int64_t j0; };

static const double *range_vrow(void *p, int64_t t)
{
    struct range_ctx *r = (struct range_ctx *)p;
    return seq_vrow_from(r->c, r->j0 + t);
}

struct task { int s, h; int64_t r0, r1; };  /* requested-row index range */

/*
 * qkv:     bf16 bits, [T][3*heads*head_dim] row-major (Q block, K block,
 *          V block; head h at columns h*head_dim within each block).
 * cu:      int32 [n_seqs+1] packed-sequence offsets.
 * theta:   RoPE base of this layer; half_window < 0 for a global layer,
 *          else the band half-width (64 for ModernBERT-base).
 * rows:    NULL for every row 0..T-1, else n_rows packed row indices, each in
 *          [0, T) and sorted ascending.
 * out:     fp64 [n_rows or T][heads*head_dim].
 * counts:  int32 [n_rows or T] admitted-key counts (may be NULL).
 * threads: OpenMP threads to use (<= 0: the runtime default).
 * Returns 0, or a negative code for bad arguments.
 */
static int attention_impl(const uint16_t *qkv, int64_t T, int heads, int head_dim,
                          const int32_t *cu, int n_seqs, double theta,
                          int half_window, const int64_t *rows, int64_t n_rows,
                          double *out, int32_t *counts, int threads, int round_operands)
{
    if (!qkv && T > 0)
        return -10;
    if (heads <= 0 || head_dim <= 0 || head_dim % 2 || head_dim > 256)
        return -11;
    int rc = check_cu(cu, n_seqs, T);
    if (rc)
        return rc;
    if (rows) {
        for (int64_t r = 0; r < n_rows; r++) {
            if (rows[r] < 0 || rows[r] >= T)
                return -12;
            if (r && rows[r] < rows[r - 1])
                return -13;
        }
    } else {
        n_rows = T;
    }
    const int width = 3 * heads * head_dim;
    const int64_t chunk = 256;

    /* tasks: (sequence, head, run of at most `chunk` requested rows) */
    int64_t cap = 16, nt = 0;
    struct task *tasks = (struct task *)malloc(sizeof(struct task) * (size_t)cap);
    if (!tasks)
        return -20;
    int64_t r = 0;
    for (int s = 0; s < n_seqs; s++) {
        int64_t b = cu[s], e = cu[s + 1];
        int64_t first = r;
        while (r < n_rows && (rows ? rows[r] : r) < e)
            r++;
        for (int64_t a = first; a < r; a += chunk) {
            for (int h = 0; h < heads; h++) {
                if (nt == cap) {
                    cap *= 2;
                    struct task *t2 = (struct task *)realloc(tasks, sizeof(struct task) * (size_t)cap);
                    if (!t2) { free(tasks); return -20; }
                    tasks = t2;
                }
                tasks[nt].s = s; tasks[nt].h = h;
                tasks[nt].r0 = a;
                tasks[nt].r1 = a + chunk < r ? a + chunk : r;
                nt++;
            }
        }
        (void)b;
    }

    int failed = 0;
#ifdef _OPENMP
    if (threads <= 0)
        threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
    for (int64_t t = 0; t < nt; t++) {
        const struct task *tk = &tasks[t];
        const int64_t row0 = cu[tk->s];
        const int64_t L = cu[tk->s + 1] - row0;
        struct seq_ctx c;
        c.qkv = qkv; c.row0 = row0; c.L = L; c.width = width;
        c.heads = heads; c.head_dim = head_dim; c.h = tk->h; c.theta = theta;
        c.round_operands = round_operands;
        c.krot = (double *)malloc(sizeof(double) * (size_t)(L * head_dim));
        c.vbuf = (double *)malloc(sizeof(double) * (size_t)(L * head_dim));
        c.kdone = (unsigned char *)calloc((size_t)L, 1);
        c.vdone = (unsigned char *)calloc((size_t)L, 1);
        double *sc = (double *)malloc(sizeof(double) * (size_t)L);
        if (!c.krot || !c.vbuf || !c.kdone || !c.vdone || !sc) {
#pragma omp atomic write
            failed = 1;
            free(c.krot); free(c.vbuf); free(c.kdone); free(c.vdone); free(sc);
            continue;
        }
        double qraw[256], qrot[256];
        const double scale = 1.0 / sqrt((double)head_dim);
        for (int64_t k = tk->r0; k < tk->r1; k++) {
            const int64_t row = rows ? rows[k] : k;
            const int64_t i = row - row0;             /* position in its sequence */
            const uint16_t *qsrc = qkv + row * width + tk->h * head_dim;
            for (int e = 0; e < head_dim; e++)
                qraw[e] = bf16_to_f64(qsrc[e]);
            oracle_rope_row(qraw, i, theta, head_dim, qrot);
            if (round_operands)
                for (int e = 0; e < head_dim; e++)
                    qrot[e] = oracle_round_bf16(qrot[e]);

            int64_t j0, j1;
            admitted_range(i, L, half_window, &j0, &j1);
            for (int64_t j = j0; j < j1; j++) {
                const double *kr = seq_krot(&c, j);
                double acc = 0.0;
                for (int e = 0; e < head_dim; e++)
                    acc += qrot[e] * kr[e];
                sc[j - j0] = acc * scale;
            }
            struct range_ctx rcx = { &c, j0 };
            softmax_blend(sc, j1 - j0, head_dim, range_vrow, &rcx, NULL,
                          out + k * heads * head_dim + tk->h * head_dim);
            if (counts && tk->h == 0)
                counts[k] = (int32_t)(j1 - j0);
        }
        free(c.krot); free(c.vbuf); free(c.kdone); free(c.vdone); free(sc);
    }
    free(tasks);
    return failed ? -20 : 0;
}

int oracle_attention(const uint16_t *qkv, int64_t T, int heads, int head_dim,
                     const int32_t *cu, int n_seqs, double theta,
                     int half_window, const int64_t *rows, int64_t n_rows,
                     double *out, int32_t *counts, int threads)
{
    return attention_impl(qkv, T, heads, head_dim, cu, n_seqs, theta, half_window,
                          rows, n_rows, out, counts, threads, 0);
}

/* The same block with the rotated q and k rows rounded to bf16 before the
 * scores are formed, everything else in fp64.  A tensor-core path multiplies
 * bf16 operands, so the rotated rows it multiplies are these rounded rows
 * (the reading of the intermediates' precision); with scores spread over
 * tens of units that rounding alone moves the weights of near-tied keys by
 * more than the output tolerance, while the rest of the computation (the
 * softmax, its rescaling and the blend) is still checked at full tolerance
 * against this variant. */
int oracle_attention_rounded(const uint16_t *qkv, int64_t T, int heads, int head_dim,
                             const int32_t *cu, int n_seqs, double theta,
                             int half_window, const int64_t *rows, int64_t n_rows,
                             double *out, int32_t *counts, int threads)
{
    return attention_impl(qkv, T, heads, head_dim, cu, n_seqs, theta, half_window,
                          rows, n_rows, out, counts, threads, 1);
}

int oracle_max_threads(void);

/* ------------------------------------------------------------------ */
/* output projection and residual add                                  */
/* ------------------------------------------------------------------ */

/* y[t][o] = x[t][o] + sum_c a[t][c] * wo[o][c] over c = 0 .. d - 1: the
 * joined head outputs a (bf16 [T][d]) mapped back to the model width by Wo,
 * stored [out][in] ("ModernBERT-base Architecture Teardown", "How Does
 * ModernBERT Make Q, K and V?": Wo maps the joined heads from 768 back to
 * 768, a Linear weight stored [out, in]), and added to the residual stream
 * x (bf16 [T][d]; "ModernBertModel", "Implementing it": x = x + a Wo^T).
 * Every product and sum in fp64; y is fp64 [T][d].  rows: NULL (every row)
 * or n sorted row indices, y then [n][d]. */
int oracle_out_proj(const uint16_t *a, const uint16_t *wo, const uint16_t *x, int64_t T, int d,
                    const int64_t *rows, int64_t n, double *y, int threads)
{
    if (T < 0 || d <= 0 || n < 0)
        return -1;
    if (!rows)
        n = T;
    double *w = malloc(sizeof(double) * (size_t)d * (size_t)d);
    if (!w)
        return -2;
    for (int64_t e = 0; e < (int64_t)d * d; e++)
        w[e] = bf16_to_f64(wo[e]);
    int bad = 0;
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : oracle_max_threads()) reduction(|:bad)
    for (int64_t k = 0; k < n; k++) {
        const int64_t t = rows ? rows[k] : k;
        if (t < 0 || t >= T) {
            bad = 1;
            continue;
        }
        double *ar = malloc(sizeof(double) * (size_t)d);
        if (!ar) {
            bad = 1;
            continue;
        }
        for (int c = 0; c < d; c++)
            ar[c] = bf16_to_f64(a[t * d + c]);
        for (int o = 0; o < d; o++) {
            double acc = 0.0;
            for (int c = 0; c < d; c++)
                acc += ar[c] * w[(int64_t)o * d + c];
            y[k * d + o] = bf16_to_f64(x[t * d + o]) + acc;
        }
        free(ar);
    }
    free(w);
    return bad ? -3 : 0;
}

/* ------------------------------------------------------------------ */
/* pre-attention LayerNorm and the fused Wqkv projection               */
/* ------------------------------------------------------------------ */

/* One row of the bias-free LayerNorm ("ModernBERT-base Architecture
 * Teardown", "What Does LayerNorm Do?"): subtract the row mean, divide by the
 * population standard deviation with eps added under the square root, then
 * multiply position c by the learned weight w[c]; no bias.  w == NULL is
 * layer 0's attn_norm, an identity ("What Does LayerNorm Do?"; "ModernBERT"
 * (candding), "The pre-norm layer and the final norm"): h = x.  x and w are
 * bf16 bit patterns; h is fp64 [d]. */
static void layernorm_row(const uint16_t *x, const uint16_t *w, int d, double eps, double *h)
{
    if (!w) {
        for (int c = 0; c < d; c++)
            h[c] = bf16_to_f64(x[c]);
        return;
    }
    double sum = 0.0;
    for (int c = 0; c < d; c++)
        sum += bf16_to_f64(x[c]);
    const double mean = sum / d;
    double sq = 0.0;
    for (int c = 0; c < d; c++) {
        const double dev = bf16_to_f64(x[c]) - mean;
        sq += dev * dev;
    }
    const double sd = sqrt(sq / d + eps);
    for (int c = 0; c < d; c++)
        h[c] = (bf16_to_f64(x[c]) - mean) / sd * bf16_to_f64(w[c]);
}

/* h = LayerNorm(x) row by row, fp64 [n][d] (rows: NULL for every row, or n
 * sorted row indices). */
int oracle_layernorm(const uint16_t *x, const uint16_t *w, int64_t T, int d, double eps,
                     const int64_t *rows, int64_t n, double *h, int threads)
{
    if (T < 0 || d <= 0 || n < 0 || eps < 0.0)
        return -1;
    if (!rows)
        n = T;
    int bad = 0;
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : oracle_max_threads()) reduction(|:bad)
    for (int64_t k = 0; k < n; k++) {
        const int64_t t = rows ? rows[k] : k;
        if (t < 0 || t >= T) {
            bad = 1;
            continue;
        }
        layernorm_row(x + t * d, w, d, eps, h + k * d);
    }
    return bad ? -3 : 0;
}

/* qkv[t][j] = sum_c h[t][c] * wqkv[j][c] with h = LayerNorm(x) (w == NULL:
 * h = x), j = 0 .. n_out - 1: the attention block's input, made by the fused
 * Wqkv, a bias-free Linear weight stored [out][in] = [3 * d][d]
 * ("ModernBERT-base Architecture Teardown", "How Does ModernBERT Make Q, K
 * and V?"; "ModernBertModel" (safebydesign), "Implementing it": the norm's
 * output times Wqkv^T, split three ways).  Every sum in fp64, no intermediate
 * rounding; qkv is fp64 [n][n_out]. */
int oracle_ln_qkv(const uint16_t *x, const uint16_t *w, const uint16_t *wqkv, int64_t T, int d,
                  int n_out, double eps, const int64_t *rows, int64_t n, double *qkv, int threads)
{
    if (T < 0 || d <= 0 || n_out <= 0 || n < 0 || eps < 0.0)
        return -1;
    if (!rows)
        n = T;
    double *wm = malloc(sizeof(double) * (size_t)n_out * (size_t)d);
    if (!wm)
        return -2;
    for (int64_t e = 0; e < (int64_t)n_out * d; e++)
        wm[e] = bf16_to_f64(wqkv[e]);
    int bad = 0;
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : oracle_max_threads()) reduction(|:bad)
    for (int64_t k = 0; k < n; k++) {
        const int64_t t = rows ? rows[k] : k;
        if (t < 0 || t >= T) {
            bad = 1;
            continue;
        }
        double *h = malloc(sizeof(double) * (size_t)d);
        if (!h) {
            bad = 1;
            continue;
        }
        layernorm_row(x + t * d, w, d, eps, h);
        for (int j = 0; j < n_out; j++) {
            double acc = 0.0;
            for (int c = 0; c < d; c++)
                acc += h[c] * wm[(int64_t)j * d + c];
            qkv[k * n_out + j] = acc;
        }
        free(h);
    }
    free(wm);
    return bad ? -3 : 0;
}

/* ------------------------------------------------------------------ */
/* the GeGLU MLP block                                                 */
/* ------------------------------------------------------------------ */

/* GELU in its exact form, z * Phi(z) = z / 2 * (1 + erf(z / sqrt 2)), not the
 * tanh approximation ("ModernBERT" (candding), "The feed-forward halves": the
 * activation is the exact erf GELU; "modernbert-base" (nest.franknoh), "Why
 * the GELU matters"). */
static double gelu_erf(double z)
{
    return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));
}

/* out[i] = gelu_erf(z[i]). */
void oracle_gelu(const double *z, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = gelu_erf(z[i]);
}

/* y = x + (GELU(g) * u) Wo^T with g, u = the first and second halves of
 * h Wi^T, h = LayerNorm(x; norm_w) ("ModernBERT-base Architecture
 * Teardown", "What Does the GeGLU MLP Do?": Wi makes two vectors of 1152,
 * the first goes through GELU, the second multiplies it number by number,
 * Wo brings the 1152 back to 768; Wi [2 * inner][d] and Wo [d][inner] are
 * Linear weights stored [out][in]; "modernbert-base" (nest.franknoh), "The
 * fused projections": the first half of Wi's output is the GELU branch;
 * "ModernBertModel" (safebydesign), "Implementing it": x = x + (gelu(g) * u)
 * Wo^T after h = layernorm(x, mlp_norm)).  Every step in fp64, no
 * intermediate rounding; y is fp64 [n][d]. */
int oracle_mlp(const uint16_t *x, const uint16_t *norm_w, const uint16_t *wi, const uint16_t *wo,
               int64_t T, int d, int inner, double eps, const int64_t *rows, int64_t n,
               double *y, int threads)
{
    if (T < 0 || d <= 0 || inner <= 0 || n < 0 || eps < 0.0 || !norm_w)
        return -1;
    if (!rows)
        n = T;
    double *wim = malloc(sizeof(double) * 2 * (size_t)inner * (size_t)d);
    double *wom = malloc(sizeof(double) * (size_t)d * (size_t)inner);
    if (!wim || !wom) {
        free(wim);
        free(wom);
        return -2;
    }
    for (int64_t e = 0; e < 2 * (int64_t)inner * d; e++)
        wim[e] = bf16_to_f64(wi[e]);
    for (int64_t e = 0; e < (int64_t)d * inner; e++)
        wom[e] = bf16_to_f64(wo[e]);
    int bad = 0;
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : oracle_max_threads()) reduction(|:bad)
    for (int64_t k = 0; k < n; k++) {
        const int64_t t = rows ? rows[k] : k;
        if (t < 0 || t >= T) {
            bad = 1;
            continue;
        }
        double *h = malloc(sizeof(double) * (size_t)d);
        double *m = malloc(sizeof(double) * (size_t)inner);
        if (!h || !m) {
            free(h);
            free(m);
            bad = 1;
            continue;
        }
        layernorm_row(x + t * d, norm_w, d, eps, h);
        for (int j = 0; j < inner; j++) {
            double g = 0.0, u = 0.0;
            for (int c = 0; c < d; c++) {
                g += h[c] * wim[(int64_t)j * d + c];
                u += h[c] * wim[(int64_t)(inner + j) * d + c];
            }
            m[j] = gelu_erf(g) * u;
        }
        for (int o = 0; o < d; o++) {
            double acc = 0.0;
            for (int j = 0; j < inner; j++)
                acc += m[j] * wom[(int64_t)o * inner + j];
            y[k * d + o] = bf16_to_f64(x[t * d + o]) + acc;
        }
        free(h);
        free(m);
    }
    free(wim);
    free(wom);
    return bad ? -3 : 0;
}

/* Number of OpenMP threads a parallel region would use by default. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
