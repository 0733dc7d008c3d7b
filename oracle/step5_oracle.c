/*
 * step5_oracle.c -- plain, slow CPU oracle for the Step-5 sparse-indexer attention.
 *
 * TEST INFRASTRUCTURE ONLY (tests, the smoke check and the benchmark's CPU-baseline
 * leg).  No code is shared with the CUDA library.  Every function follows the
 * definition stated in "Step-5-Preview on one 256 GB Mac" (TensorFold PR #903,
 * the commit adding the CSA indexer for contexts up to 1M tokens), written out in the
 * page's order with no blocking, fusion or reordering.  Compile with
 * -ffp-contract=off so that the arithmetic is the same on every host.
 */
#include "step5_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------------ */
/* Codecs: from the format definitions.                                            */
/* ------------------------------------------------------------------------------ */

/* Round a non-negative double to an integer, ties to even. */
static double round_half_even(double v) {
    double f = floor(v);
    double frac = v - f; /* exact */
    if (frac > 0.5) return f + 1.0;
    if (frac < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* Nearest value with `sig_bits` significant bits whose quantum never drops below
 * 2^min_quantum_exp (the subnormal spacing), ties to even. */
static double round_to_format(double x, int sig_bits, int min_quantum_exp) {
    if (isnan(x) || x == 0.0 || isinf(x)) return x;
    double a = fabs(x);
    int e;
    frexp(a, &e); /* a in [2^(e-1), 2^e) */
    int qexp = e - sig_bits;
    if (qexp < min_quantum_exp) qexp = min_quantum_exp;
    double q = ldexp(round_half_even(ldexp(a, -qexp)), qexp);
    return copysign(q, x);
}

/* bfloat16: 8 significant bits, exponent range of binary32 (min normal 2^-126,
 * subnormal spacing 2^-133, largest finite (2 - 2^-7) * 2^127). */
double orc_round_bf16(double x) {
    double q = round_to_format(x, 8, -133);
    const double bf16_max = ldexp(255.0, 120); /* 1.1111111b * 2^127 */
    if (fabs(q) > bf16_max) q = copysign(INFINITY, x);
    return q;
}

/* OCP E4M3 "fn": 4 significant bits, min normal 2^-6, subnormal spacing 2^-9,
 * largest finite 448; saturating conversion clamps to +-448. */
double orc_round_e4m3(double x) {
    if (isnan(x)) return x;
    if (isinf(x)) return copysign(448.0, x);
    double q = round_to_format(x, 4, -9);
    if (fabs(q) > 448.0) q = copysign(448.0, x);
    return q;
}

uint16_t orc_bf16_code(double v) {
    float f = (float)v; /* exact for a bf16-representable v */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

double orc_bf16_value(uint16_t code) {
    uint32_t u = (uint32_t)code << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

uint8_t orc_e4m3_code(double v) {
    if (isnan(v)) return 0x7F;
    uint8_t s = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a == 0.0) return s;
    if (a < ldexp(1.0, -6)) return (uint8_t)(s | (uint8_t)(a * 512.0)); /* m * 2^-9 */
    int e;
    double m = frexp(a, &e); /* a = (2m) * 2^(e-1), 2m in [1,2) */
    int E = e - 1;
    int mant = (int)((2.0 * m - 1.0) * 8.0);
    return (uint8_t)(s | (uint8_t)(((E + 7) << 3) | mant));
}

double orc_e4m3_value(uint8_t code) {
    int s = code >> 7, E = (code >> 3) & 15, M = code & 7;
    if (E == 15 && M == 7) return NAN;
    double v = (E == 0) ? ldexp((double)M, -9) : ldexp((double)(8 + M), E - 10);
    return s ? -v : v;
}

void orc_bf16_codes_to_e4m3_codes(const uint16_t* in, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_code(orc_round_e4m3(orc_bf16_value(in[i])));
}

void orc_round_bf16_array(const double* in, uint16_t* out_codes, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out_codes[i] = orc_bf16_code(orc_round_bf16(in[i]));
}

/* ------------------------------------------------------------------------------ */
/* NEOX partial rotation.                                                           */
/* ------------------------------------------------------------------------------ */

void orc_rotate_neox(const uint16_t* x, int dim, int rope_dims,
                     const uint16_t* cos_row, const uint16_t* sin_row, double* out) {
    for (int d = 0; d < dim; ++d) out[d] = orc_bf16_value(x[d]);
    if (cos_row == NULL || rope_dims == 0) return;
    int half = rope_dims / 2;
    for (int i = 0; i < half; ++i) {
        double x1 = orc_bf16_value(x[i]);
        double x2 = orc_bf16_value(x[i + half]);
        double c = orc_bf16_value(cos_row[i]);
        double s = orc_bf16_value(sin_row[i]);
        out[i] = orc_round_bf16(x1 * c - x2 * s);
        out[i + half] = orc_round_bf16(x2 * c + x1 * s);
    }
}

/* ------------------------------------------------------------------------------ */
/* Before step 1: the indexer's q and k norms.                                      */
/* ------------------------------------------------------------------------------ */

void orc_rmsnorm_1pw(const uint16_t* x, const uint16_t* w, int dim, double eps, uint16_t* out) {
    double ss = 0.0;
    for (int d = 0; d < dim; ++d) {
        double v = orc_bf16_value(x[d]);
        ss += v * v;
    }
    double rms = sqrt(ss / dim + eps);
    for (int d = 0; d < dim; ++d)
        out[d] = orc_bf16_code(orc_round_bf16(orc_bf16_value(x[d]) / rms * (1.0 + orc_bf16_value(w[d]))));
}

void orc_layernorm(const uint16_t* x, const uint16_t* g, const uint16_t* b, int dim, double eps,
                   uint16_t* out) {
    double mean = 0.0;
    for (int d = 0; d < dim; ++d) mean += orc_bf16_value(x[d]);
    mean /= dim;
    double var = 0.0;
    for (int d = 0; d < dim; ++d) {
        double c = orc_bf16_value(x[d]) - mean;
        var += c * c;
    }
    var /= dim;
    double sd = sqrt(var + eps);
    for (int d = 0; d < dim; ++d)
        out[d] = orc_bf16_code(orc_round_bf16((orc_bf16_value(x[d]) - mean) / sd * orc_bf16_value(g[d]) +
                                              orc_bf16_value(b[d])));
}

/* ------------------------------------------------------------------------------ */
/* Step 1: summary of one completed region.                                         */
/* ------------------------------------------------------------------------------ */

void orc_summarize_region(const uint16_t* k, const uint16_t* z, int region_tokens,
                          int dim, int t0, int rope_dims,
                          const uint16_t* cos_tab, const uint16_t* sin_tab,
                          double* s_out, uint8_t* code_out) {
    int half = rope_dims / 2;
    double* kr = (double*)malloc(sizeof(double) * (size_t)region_tokens * (size_t)dim);
    for (int j = 0; j < region_tokens; ++j) {
        const uint16_t* cr = cos_tab ? cos_tab + (int64_t)(t0 + j) * half : NULL;
        const uint16_t* sr = sin_tab ? sin_tab + (int64_t)(t0 + j) * half : NULL;
        orc_rotate_neox(k + (int64_t)j * dim, dim, rope_dims, cr, sr, kr + (int64_t)j * dim);
    }
    for (int d = 0; d < dim; ++d) {
        double m = -INFINITY;
        for (int j = 0; j < region_tokens; ++j) {
            double zj = orc_bf16_value(z[(int64_t)j * dim + d]);
            if (zj > m) m = zj;
        }
        double den = 0.0, num = 0.0;
        for (int j = 0; j < region_tokens; ++j) {
            double e = exp(orc_bf16_value(z[(int64_t)j * dim + d]) - m);
            den += e;
            num += e * kr[(int64_t)j * dim + d];
        }
        double s = num / den;
        if (s_out) s_out[d] = s;
        if (code_out) code_out[d] = orc_e4m3_code(orc_round_e4m3(orc_round_bf16(s)));
    }
    free(kr);
}

/* ------------------------------------------------------------------------------ */
/* Step 2: index scores for one (row, group).                                       */
/* ------------------------------------------------------------------------------ */

void orc_score_group(const uint16_t* q, const float* w, int hpg, int dim, int pos,
                     int rope_dims, const uint16_t* cos_tab, const uint16_t* sin_tab,
                     const uint8_t* summ, int64_t R, double* out) {
    int half = rope_dims / 2;
    double* qe = (double*)malloc(sizeof(double) * (size_t)hpg * (size_t)dim);
    double* rot = (double*)malloc(sizeof(double) * (size_t)dim);
    const uint16_t* cr = cos_tab ? cos_tab + (int64_t)pos * half : NULL;
    const uint16_t* sr = sin_tab ? sin_tab + (int64_t)pos * half : NULL;
    for (int h = 0; h < hpg; ++h) {
        orc_rotate_neox(q + (int64_t)h * dim, dim, rope_dims, cr, sr, rot);
        for (int d = 0; d < dim; ++d) qe[(int64_t)h * dim + d] = orc_round_e4m3(rot[d]);
    }
    for (int64_t r = 0; r < R; ++r) {
        const uint8_t* s = summ + r * dim;
        double score = 0.0;
        for (int h = 0; h < hpg; ++h) {
            double dot = 0.0;
            for (int d = 0; d < dim; ++d) dot += qe[(int64_t)h * dim + d] * orc_e4m3_value(s[d]);
            double relu = dot > 0.0 ? dot : 0.0;
            score += relu * (double)w[h];
        }
        out[r] = (score == 0.0) ? 0.0 : score; /* -0 -> +0 */
    }
    free(rot);
    free(qe);
}

/* ------------------------------------------------------------------------------ */
/* Step 3: top-K by (-score, id), ascending.                                         */
/* ------------------------------------------------------------------------------ */

typedef struct {
    double neg_score;
    int64_t id;
} orc_key;

static int key_cmp(const void* pa, const void* pb) {
    const orc_key* a = (const orc_key*)pa;
    const orc_key* b = (const orc_key*)pb;
    if (a->neg_score < b->neg_score) return -1;
    if (a->neg_score > b->neg_score) return 1;
    return (a->id < b->id) ? -1 : (a->id > b->id) ? 1 : 0;
}

int orc_select_topk(const double* scores, int64_t R, int K, int32_t* ids_out) {
    if (R <= 0) return 0;
    orc_key* keys = (orc_key*)malloc(sizeof(orc_key) * (size_t)R);
    for (int64_t r = 0; r < R; ++r) {
        double s = scores[r];
        keys[r].neg_score = (s == 0.0) ? 0.0 : -s; /* -0 and +0 compare equal anyway */
        keys[r].id = r;
    }
    qsort(keys, (size_t)R, sizeof(orc_key), key_cmp);
    int cnt = (R < K) ? (int)R : K;
    for (int i = 0; i < cnt; ++i) ids_out[i] = (int32_t)keys[i].id;
    free(keys);
    return cnt;
}

/* ------------------------------------------------------------------------------ */
/* Step 4: attention over the selected regions plus the row's own region.           */
/* ------------------------------------------------------------------------------ */

void orc_attend_group(const uint16_t* q, int hq_g, int head_dim,
                      const uint16_t* kc, const uint16_t* vc,
                      const int32_t* sel, int cnt, int pos, int region_tokens,
                      double scale, double* out) {
    int own = pos / region_tokens;
    int own_len = pos - own * region_tokens + 1;
    int64_t nkeys = (int64_t)cnt * region_tokens + own_len;
    int64_t* tok = (int64_t*)malloc(sizeof(int64_t) * (size_t)nkeys);
    int64_t n = 0;
    for (int i = 0; i < cnt; ++i)
        for (int j = 0; j < region_tokens; ++j) tok[n++] = (int64_t)sel[i] * region_tokens + j;
    for (int j = 0; j < own_len; ++j) tok[n++] = (int64_t)own * region_tokens + j;

    double* logit = (double*)malloc(sizeof(double) * (size_t)nkeys);
    for (int h = 0; h < hq_g; ++h) {
        const uint16_t* qh = q + (int64_t)h * head_dim;
        double m = -INFINITY;
        for (int64_t t = 0; t < nkeys; ++t) {
            const uint16_t* kt = kc + tok[t] * head_dim;
            double dot = 0.0;
            for (int d = 0; d < head_dim; ++d) dot += orc_bf16_value(qh[d]) * orc_bf16_value(kt[d]);
            logit[t] = scale * dot;
            if (logit[t] > m) m = logit[t];
        }
        double l = 0.0;
        for (int64_t t = 0; t < nkeys; ++t) {
            logit[t] = exp(logit[t] - m);
            l += logit[t];
        }
        for (int d = 0; d < head_dim; ++d) {
            double acc = 0.0;
            for (int64_t t = 0; t < nkeys; ++t) acc += logit[t] * orc_bf16_value(vc[tok[t] * head_dim + d]);
            out[(int64_t)h * head_dim + d] = acc / l;
        }
    }
    free(logit);
    free(tok);
}

/* ------------------------------------------------------------------------------ */
/* Sequence-sharded decode: merge of the shards' picks, partial attention, combine.  */
/* ------------------------------------------------------------------------------ */

int orc_merge_topk(int S, int L, int K, const int32_t* ids, const double* scores, const int32_t* counts,
                   int32_t* ids_out) {
    int64_t total = 0;
    for (int s = 0; s < S; ++s) total += counts[s];
    orc_key* keys = (orc_key*)malloc(sizeof(orc_key) * (size_t)(total > 0 ? total : 1));
    int64_t n = 0;
    for (int s = 0; s < S; ++s)
        for (int i = 0; i < counts[s]; ++i) {
            double sc = scores[(int64_t)s * L + i];
            keys[n].neg_score = (sc == 0.0) ? 0.0 : -sc;
            keys[n].id = ids[(int64_t)s * L + i];
            ++n;
        }
    qsort(keys, (size_t)n, sizeof(orc_key), key_cmp);
    int take = n < K ? (int)n : K;
    for (int i = 0; i < take; ++i) ids_out[i] = (int32_t)keys[i].id;
    for (int i = take; i < K; ++i) ids_out[i] = -1;
    free(keys);
    return take;
}

void orc_attend_partial(const uint16_t* q, int hq_g, int head_dim, const uint16_t* kc, const uint16_t* vc,
                        const int32_t* sel, int cnt, int pos, int region_tokens, int64_t tok_lo,
                        int64_t tok_hi, double scale, double* m, double* l, double* o) {
    int own = pos / region_tokens;
    int own_len = pos - own * region_tokens + 1;
    int64_t* tok = (int64_t*)malloc(sizeof(int64_t) * ((size_t)cnt * region_tokens + own_len + 1));
    int64_t n = 0;
    for (int i = 0; i < cnt; ++i)
        for (int j = 0; j < region_tokens; ++j) {
            int64_t t = (int64_t)sel[i] * region_tokens + j;
            if (t >= tok_lo && t < tok_hi) tok[n++] = t;
        }
    for (int j = 0; j < own_len; ++j) {
        int64_t t = (int64_t)own * region_tokens + j;
        if (t >= tok_lo && t < tok_hi) tok[n++] = t;
    }
    double* logit = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int h = 0; h < hq_g; ++h) {
        const uint16_t* qh = q + (int64_t)h * head_dim;
        double mh = -INFINITY;
        for (int64_t t = 0; t < n; ++t) {
            const uint16_t* kt = kc + tok[t] * head_dim;
            double dot = 0.0;
            for (int d = 0; d < head_dim; ++d) dot += orc_bf16_value(qh[d]) * orc_bf16_value(kt[d]);
            logit[t] = scale * dot;
            if (logit[t] > mh) mh = logit[t];
        }
        double lh = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            logit[t] = exp(logit[t] - mh);
            lh += logit[t];
        }
        m[h] = mh;
        l[h] = lh;
        for (int d = 0; d < head_dim; ++d) {
            double acc = 0.0;
            for (int64_t t = 0; t < n; ++t) acc += logit[t] * orc_bf16_value(vc[tok[t] * head_dim + d]);
            o[(int64_t)h * head_dim + d] = acc;
        }
    }
    free(logit);
    free(tok);
}

void orc_attn_combine(int S, int head_dim, const double* m, const double* l, const double* o, double* out) {
    double M = -INFINITY;
    for (int s = 0; s < S; ++s)
        if (m[s] > M) M = m[s];
    double L = 0.0;
    for (int s = 0; s < S; ++s) L += (l[s] > 0.0 ? exp(m[s] - M) * l[s] : 0.0);
    for (int d = 0; d < head_dim; ++d) {
        double acc = 0.0;
        for (int s = 0; s < S; ++s)
            if (l[s] > 0.0) acc += exp(m[s] - M) * o[(int64_t)s * head_dim + d];
        out[d] = acc / L;
    }
}

/* ------------------------------------------------------------------------------ */
/* After step 4: the per-head sigmoid output gate.                                   */
/* ------------------------------------------------------------------------------ */

void orc_sigmoid_gate(double* out, const uint16_t* gate, int64_t rows, int head_dim) {
    for (int64_t r = 0; r < rows; ++r) {
        const double g = orc_bf16_value(gate[r]);
        const double s = 1.0 / (1.0 + exp(-g));
        for (int d = 0; d < head_dim; ++d) out[r * head_dim + d] *= s;
    }
}

/* ------------------------------------------------------------------------------ */
/* Batched drivers: independent items spread over host threads.                     */
/* ------------------------------------------------------------------------------ */

typedef void (*item_fn)(void* ctx, int64_t item);

typedef struct {
    item_fn fn;
    void* ctx;
    int64_t nitems;
    int tid, nthreads;
} worker_arg;

static void* worker_main(void* p) {
    worker_arg* a = (worker_arg*)p;
    for (int64_t i = a->tid; i < a->nitems; i += a->nthreads) a->fn(a->ctx, i);
    return NULL;
}

static int parallel_for(int64_t nitems, int nthreads, item_fn fn, void* ctx) {
    if (nthreads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = c > 0 ? (int)c : 1;
    }
    if ((int64_t)nthreads > nitems) nthreads = nitems > 0 ? (int)nitems : 1;
    if (nthreads == 1) {
        for (int64_t i = 0; i < nitems; ++i) fn(ctx, i);
        return 1;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    worker_arg* args = (worker_arg*)malloc(sizeof(worker_arg) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        args[t].fn = fn;
        args[t].ctx = ctx;
        args[t].nitems = nitems;
        args[t].tid = t;
        args[t].nthreads = nthreads;
        pthread_create(&th[t], NULL, worker_main, &args[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(args);
    free(th);
    return nthreads;
}

/* summarize: one item per (b, g, region) */
typedef struct {
    int B, G, dim, rt, rope_dims;
    int64_t t_cap, r_cap, max_span;
    const uint16_t *k, *z, *cs, *sn;
    const int32_t *rb, *re;
    uint8_t* summ;
    double* s64;
} sum_ctx;

static void sum_item(void* p, int64_t item) {
    sum_ctx* c = (sum_ctx*)p;
    int64_t j = item % c->max_span;
    int64_t bg = item / c->max_span;
    int g = (int)(bg % c->G), b = (int)(bg / c->G);
    int64_t r = c->rb[b] + j;
    if (r >= c->re[b]) return;
    int64_t krow = ((int64_t)b * c->G + g) * c->t_cap + r * c->rt;
    int64_t srow = ((int64_t)b * c->G + g) * c->r_cap + r;
    orc_summarize_region(c->k + krow * c->dim, c->z + krow * c->dim, c->rt, c->dim,
                         (int)(r * c->rt), c->rope_dims, c->cs, c->sn,
                         c->s64 ? c->s64 + srow * c->dim : NULL, c->summ + srow * c->dim);
}

int orc_summarize_batch(int B, int G, int64_t t_cap, int64_t r_cap, int dim,
                        int region_tokens, int rope_dims,
                        const uint16_t* k, const uint16_t* z,
                        const uint16_t* cos_tab, const uint16_t* sin_tab,
                        const int32_t* region_begin, const int32_t* region_end,
                        uint8_t* summ, double* s_f64, int nthreads) {
    int64_t max_span = 1;
    for (int b = 0; b < B; ++b)
        if ((int64_t)region_end[b] - region_begin[b] > max_span)
            max_span = (int64_t)region_end[b] - region_begin[b];
    sum_ctx c = {B, G, dim, region_tokens, rope_dims, t_cap, r_cap, max_span,
                 k, z, cos_tab, sin_tab, region_begin, region_end, summ, s_f64};
    return parallel_for((int64_t)B * G * max_span, nthreads, sum_item, &c);
}

/* score: one item per (n, g, chunk of regions) */
#define ORC_SCORE_CHUNK 4096
typedef struct {
    int N, G, idx_heads, dim, rt, rope_dims;
    int64_t r_cap, nchunks;
    const uint16_t* q;
    const float* w;
    const int32_t *seq, *pos;
    const uint16_t *cs, *sn;
    const uint8_t* summ;
    double* scores;
} score_ctx;

static void score_item(void* p, int64_t item) {
    score_ctx* c = (score_ctx*)p;
    int64_t chunk = item % c->nchunks;
    int64_t ng = item / c->nchunks;
    int g = (int)(ng % c->G), n = (int)(ng / c->G);
    int64_t R = c->pos[n] / c->rt;
    int64_t r0 = chunk * ORC_SCORE_CHUNK;
    if (r0 >= R) return;
    int64_t len = R - r0 < ORC_SCORE_CHUNK ? R - r0 : ORC_SCORE_CHUNK;
    int hpg = c->idx_heads / c->G;
    int b = c->seq[n];
    orc_score_group(c->q + ((int64_t)n * c->idx_heads + (int64_t)g * hpg) * c->dim,
                    c->w + (int64_t)n * c->idx_heads + (int64_t)g * hpg, hpg, c->dim,
                    c->pos[n], c->rope_dims, c->cs, c->sn,
                    c->summ + (((int64_t)b * c->G + g) * c->r_cap + r0) * c->dim, len,
                    c->scores + ((int64_t)n * c->G + g) * c->r_cap + r0);
}

int orc_score_batch(int N, int G, int idx_heads, int dim, int region_tokens,
                    int rope_dims, int64_t r_cap,
                    const uint16_t* q, const float* w,
                    const int32_t* row_seq, const int32_t* row_pos,
                    const uint16_t* cos_tab, const uint16_t* sin_tab,
                    const uint8_t* summ, double* scores, int nthreads) {
    int64_t maxR = 1;
    for (int n = 0; n < N; ++n)
        if ((int64_t)row_pos[n] / region_tokens > maxR) maxR = row_pos[n] / region_tokens;
    int64_t nchunks = (maxR + ORC_SCORE_CHUNK - 1) / ORC_SCORE_CHUNK;
    score_ctx c = {N, G, idx_heads, dim, region_tokens, rope_dims, r_cap, nchunks,
                   q, w, row_seq, row_pos, cos_tab, sin_tab, summ, scores};
    return parallel_for((int64_t)N * G * nchunks, nthreads, score_item, &c);
}

/* select: one item per (n, g) */
typedef struct {
    int G, K, rt;
    int64_t r_cap;
    const int32_t* pos;
    const double* scores;
    int32_t *ids, *cnt;
} sel_ctx;

static void sel_item(void* p, int64_t item) {
    sel_ctx* c = (sel_ctx*)p;
    int n = (int)(item / c->G);
    int64_t R = c->pos[n] / c->rt;
    int32_t* ids = c->ids + item * c->K;
    for (int i = 0; i < c->K; ++i) ids[i] = -1;
    c->cnt[item] = orc_select_topk(c->scores + item * c->r_cap, R, c->K, ids);
}

int orc_select_batch(int N, int G, int K, int region_tokens, int64_t r_cap,
                     const int32_t* row_pos, const double* scores,
                     int32_t* sel_ids, int32_t* sel_count, int nthreads) {
    sel_ctx c = {G, K, region_tokens, r_cap, row_pos, scores, sel_ids, sel_count};
    return parallel_for((int64_t)N * G, nthreads, sel_item, &c);
}

/* attend: one item per (n, g) */
typedef struct {
    int G, hq, D, rt, K;
    int64_t t_cap;
    double scale;
    const uint16_t *q, *kc, *vc;
    const int32_t *seq, *pos, *ids, *cnt;
    double* out;
} att_ctx;

static void att_item(void* p, int64_t item) {
    att_ctx* c = (att_ctx*)p;
    int n = (int)(item / c->G), g = (int)(item % c->G);
    int hq_g = c->hq / c->G;
    int b = c->seq[n];
    int64_t cache = ((int64_t)b * c->G + g) * c->t_cap * c->D;
    orc_attend_group(c->q + ((int64_t)n * c->hq + (int64_t)g * hq_g) * c->D, hq_g, c->D,
                     c->kc + cache, c->vc + cache, c->ids + item * c->K, c->cnt[item],
                     c->pos[n], c->rt, c->scale,
                     c->out + ((int64_t)n * c->hq + (int64_t)g * hq_g) * c->D);
}

int orc_attend_batch(int N, int G, int num_q_heads, int head_dim, int region_tokens,
                     int K, int64_t t_cap, double scale,
                     const uint16_t* q, const uint16_t* kc, const uint16_t* vc,
                     const int32_t* row_seq, const int32_t* row_pos,
                     const int32_t* sel_ids, const int32_t* sel_count,
                     double* out, int nthreads) {
    att_ctx c = {G, num_q_heads, head_dim, region_tokens, K, t_cap, scale,
                 q, kc, vc, row_seq, row_pos, sel_ids, sel_count, out};
    return parallel_for((int64_t)N * G, nthreads, att_item, &c);
}

/* ------------------------------------------------------------------------------ */
/* The decode front end (rows in order).                                            */
/* ------------------------------------------------------------------------------ */

int orc_indexer_front(int N, int G, int idx_heads, int dim, int region_tokens, int rope_dims,
                      int B, int64_t t_cap, int64_t r_cap, double eps,
                      const uint16_t* q_pre, const uint16_t* k_pre, const uint16_t* z_pre,
                      const uint16_t* qw, const uint16_t* kw, const uint16_t* kb,
                      const int32_t* row_seq, const int32_t* row_pos,
                      const uint16_t* cos_tab, const uint16_t* sin_tab,
                      uint16_t* q_out, uint16_t* k_cache, uint16_t* z_cache, uint8_t* summ) {
    int bad = 0;
    for (int n = 0; n < N; ++n) {
        for (int h = 0; h < idx_heads; ++h)
            orc_rmsnorm_1pw(q_pre + ((int64_t)n * idx_heads + h) * dim, qw, dim, eps,
                            q_out + ((int64_t)n * idx_heads + h) * dim);
        int b = row_seq[n], p = row_pos[n];
        if (b < 0 || b >= B || p < 0 || p >= t_cap) {
            bad = -1;
            continue;
        }
        for (int g = 0; g < G; ++g) {
            int64_t row = (((int64_t)b * G + g) * t_cap + p) * dim;
            orc_layernorm(k_pre + ((int64_t)n * G + g) * dim, kw, kb, dim, eps, k_cache + row);
            memcpy(z_cache + row, z_pre + ((int64_t)n * G + g) * dim, sizeof(uint16_t) * (size_t)dim);
        }
        if (p % region_tokens == region_tokens - 1 && p / region_tokens < r_cap) {
            int r = p / region_tokens;
            for (int g = 0; g < G; ++g) {
                int64_t t0 = ((int64_t)b * G + g) * t_cap + (int64_t)r * region_tokens;
                orc_summarize_region(k_cache + t0 * dim, z_cache + t0 * dim, region_tokens, dim,
                                     r * region_tokens, rope_dims, cos_tab, sin_tab, NULL,
                                     summ + (((int64_t)b * G + g) * r_cap + r) * dim);
            }
        }
    }
    return bad;
}
