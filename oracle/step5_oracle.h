/*
 * step5_oracle.h -- plain, slow CPU oracle for the Step-5 sparse-indexer attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this
 * library; only the tests, the smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Source of the method: "Step-5-Preview on one 256 GB Mac" (TensorFold PR #903),
 * the commit that adds the CSA indexer for contexts up to 1M tokens: every completed
 * 8-token region is summarised as a per-dim softmax over z of the indexer k, rounded
 * through bf16 to e4m3; a region's score in a KV group is sum_h relu(e4m3(q_h) . summary)
 * * w_h over the group's indexer heads; the 512 smallest (-score, id) keys are kept in
 * key order; the row attends to those regions and to its own region.  The indexer's q and k take NEOX rotation on their
 * first 32 dims from bf16 cos/sin (same page, the commit on Step-5's glue).
 *
 * Arithmetic: fp64 everywhere except at the rounding points the page fixes
 * (bf16 after rotation, bf16 then e4m3 for summaries, e4m3 for the indexer q).
 * Codes: bf16 values travel as uint16 bit patterns, e4m3 values as uint8 codes
 * (OCP FP8 E4M3 "fn": bias 7, 3 mantissa bits, no infinities, 0x7F/0xFF = NaN).
 */
#ifndef STEP5_ORACLE_H
#define STEP5_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- codecs (format definitions: bfloat16 = IEEE binary32 with 7 stored mantissa
 *      bits; OCP 8-bit floating point, E4M3 with saturation) ---------------------- */
double   orc_round_bf16(double x);      /* nearest bf16 value, ties to even; overflow -> inf */
double   orc_round_e4m3(double x);      /* nearest e4m3 value, ties to even; |x|>448 -> 448 */
uint16_t orc_bf16_code(double v);       /* bit pattern of a bf16-representable value        */
double   orc_bf16_value(uint16_t code);
uint8_t  orc_e4m3_code(double v);       /* code of an e4m3-representable value (or NaN)      */
double   orc_e4m3_value(uint8_t code);
void     orc_bf16_codes_to_e4m3_codes(const uint16_t* in, uint8_t* out, int64_t n);
void     orc_round_bf16_array(const double* in, uint16_t* out_codes, int64_t n);

/* ---- NEOX partial rotation (the page's glue commit: q and k rotated NEOX-style from
 *      bf16 cos/sin tables; the indexer commit: the first 32 dims rotate) -----------
 * x: dim bf16 codes.  Pairs (i, i + rope_dims/2) for i < rope_dims/2 rotate by the
 * angle whose bf16 cosine/sine are cos_row[i]/sin_row[i].  Each rotated element is
 * x1*c - x2*s (first half) or x2*c + x1*s (second half), rounded once to bf16.
 * cos_row == NULL means "already rotated": out = x.  out: dim doubles (bf16 values). */
void orc_rotate_neox(const uint16_t* x, int dim, int rope_dims,
                     const uint16_t* cos_row, const uint16_t* sin_row, double* out);

/* ---- before step 1: the indexer's q and k norms (decode front end) ------------------
 * ("Step-5-Preview on one 256 GB Mac", CSA-indexer commit: the indexer's 16-head q
 * takes an RMSNorm with weight 1 + w, its k a LayerNorm with bias; z is not normalised.)  x, w, g, b: dim bf16 codes; fp64
 * arithmetic, one bf16 rounding of each output.
 *   RMSNorm 1 + w:  y[d] = x[d] / sqrt(mean_d x^2 + eps) * (1 + w[d])
 *   LayerNorm:      y[d] = (x[d] - mean) / sqrt(mean_d (x - mean)^2 + eps) * g[d] + b[d] */
void orc_rmsnorm_1pw(const uint16_t* x, const uint16_t* w, int dim, double eps, uint16_t* out);
void orc_layernorm(const uint16_t* x, const uint16_t* g, const uint16_t* b, int dim, double eps,
                   uint16_t* out);

/* ---- step 1: region summary -------------------------------------------------------
 * k, z: region_tokens rows of dim bf16 codes (row stride dim).  Token j sits at
 * position t0 + j; its rotation row is cos_tab[(t0 + j) * (rope_dims/2)].
 * s_out[d] = sum_j softmax_j(z[., d]) * rot(k)[j][d]   (fp64)
 * code_out[d] = e4m3(bf16(s_out[d])).                                                */
void orc_summarize_region(const uint16_t* k, const uint16_t* z, int region_tokens,
                          int dim, int t0, int rope_dims,
                          const uint16_t* cos_tab, const uint16_t* sin_tab,
                          double* s_out, uint8_t* code_out);

/* ---- step 2: index scores for one (row, KV group) ---------------------------------
 * q: hpg indexer heads x dim bf16 codes (the group's heads), w: hpg floats, row at
 * position pos.  summ: R regions x dim e4m3 codes.
 * out[r] = sum_h relu( sum_d e4m3(bf16(rot(q_h)))[d] * summ[r][d] ) * w_h  (fp64;
 * the inner sum is exact in fp64).  -0 is returned as +0.                           */
void orc_score_group(const uint16_t* q, const float* w, int hpg, int dim, int pos,
                     int rope_dims, const uint16_t* cos_tab, const uint16_t* sin_tab,
                     const uint8_t* summ, int64_t R, double* out);

/* ---- step 3: selection for one (row, KV group) ------------------------------------
 * Sorts the R keys (-score, id) ascending and writes the first min(K, R) ids in that
 * order.  Returns the count.  scores are fp64 (an fp32 score converts exactly).      */
int orc_select_topk(const double* scores, int64_t R, int K, int32_t* ids_out);

/* ---- step 4: attention for one (row, KV group) -------------------------------------
 * q: hq_g query heads x head_dim bf16 codes.  kc, vc: this (sequence, group)'s cache,
 * t_cap rows x head_dim bf16 codes.  Keys: every token of the cnt regions in sel, then
 * the tokens rt*o .. pos of the row's own region o = pos / rt.
 * out[h][d] = sum_t softmax_t(scale * q_h . k_t) v_t[d]   (fp64, max-subtracted).     */
void orc_attend_group(const uint16_t* q, int hq_g, int head_dim,
                      const uint16_t* kc, const uint16_t* vc,
                      const int32_t* sel, int cnt, int pos, int region_tokens,
                      double scale, double* out);

/* ---- sequence-sharded decode (one row's regions split over shards) ------------------
 * Merge: the K smallest keys (-score, id) of the union of S shards' picks (shard s's
 * list: ids[s][0 .. cnt_s) and their scores, rows of L entries), written in key order
 * (ids_out has K entries, -1 padded); returns the count.
 * The pick of the whole row equals this merge of the shards' own top K whenever the
 * shards partition its regions.                                                        */
int orc_merge_topk(int S, int L, int K, const int32_t* ids, const double* scores, const int32_t* counts,
                   int32_t* ids_out);

/* Partial attention of one (row, KV group) over the keys of a shard of its tokens
 * [tok_lo, tok_hi): the picked regions inside it and, when it holds the row's own region,
 * that region's tokens 8o .. pos.  Per head h, with logits x_t = scale * q_h . k_t:
 *   m[h] = max_t x_t,  l[h] = sum_t exp(x_t - m[h]),  o[h][d] = sum_t exp(x_t - m[h]) v_t[d]
 * (m = -inf, l = 0, o = 0 when the shard holds no key).  kc, vc: the whole (sequence,
 * group) cache (t_cap rows, global token index); fp64.                               */
void orc_attend_partial(const uint16_t* q, int hq_g, int head_dim, const uint16_t* kc, const uint16_t* vc,
                        const int32_t* sel, int cnt, int pos, int region_tokens, int64_t tok_lo,
                        int64_t tok_hi, double scale, double* m, double* l, double* o);

/* Combine of S partial states of one head: out[d] = sum_s e^(m_s - M) o_s[d] /
 * sum_s e^(m_s - M) l_s, M = max_s m_s.  m, l: [S]; o: [S][head_dim].                */
void orc_attn_combine(int S, int head_dim, const double* m, const double* l, const double* o, double* out);

/* ---- after step 4: the per-head sigmoid output gate ----------------------------------
 * ("Step-5-Preview on one 256 GB Mac", the native-family commit: Step-5's glue keeps
 * a per-head sigmoid gate among StepFun's rounding points.)  Reading: one gate
 * logit per (row, query head), a bf16 input; every output dim of the head is scaled by
 * sigmoid(logit) before the output's single bf16 rounding.
 * out: [rows][head_dim] fp64, scaled in place; gate: [rows] bf16 codes.              */
void orc_sigmoid_gate(double* out, const uint16_t* gate, int64_t rows, int head_dim);

/* ---- batched drivers: plain loops over independent items, spread over nthreads
 *      host threads (0 = all online cores).  They add no arithmetic of their own. ---- */

/* Summaries for b in [0,B), g in [0,G), r in [region_begin[b], region_end[b]).
 * k, z: [B][G][t_cap][dim].  summ: [B][G][r_cap][dim] codes; s_f64 (nullable) same
 * shape in fp64.  Returns the threads used.                                          */
int orc_summarize_batch(int B, int G, int64_t t_cap, int64_t r_cap, int dim,
                        int region_tokens, int rope_dims,
                        const uint16_t* k, const uint16_t* z,
                        const uint16_t* cos_tab, const uint16_t* sin_tab,
                        const int32_t* region_begin, const int32_t* region_end,
                        uint8_t* summ, double* s_f64, int nthreads);

/* Scores for n in [0,N), g in [0,G), r < row_pos[n] / region_tokens.
 * q: [N][idx_heads][dim], w: [N][idx_heads]; group g owns heads [g*hpg, (g+1)*hpg).
 * summ: [B][G][r_cap][dim].  scores: [N][G][r_cap] fp64 (entries past R untouched). */
int orc_score_batch(int N, int G, int idx_heads, int dim, int region_tokens,
                    int rope_dims, int64_t r_cap,
                    const uint16_t* q, const float* w,
                    const int32_t* row_seq, const int32_t* row_pos,
                    const uint16_t* cos_tab, const uint16_t* sin_tab,
                    const uint8_t* summ, double* scores, int nthreads);

/* Selections for every (n, g) from scores [N][G][r_cap] (fp64), R = row_pos/rt.
 * sel_ids: [N][G][K], padded with -1; sel_count: [N][G].                             */
int orc_select_batch(int N, int G, int K, int region_tokens, int64_t r_cap,
                     const int32_t* row_pos, const double* scores,
                     int32_t* sel_ids, int32_t* sel_count, int nthreads);

/* Attention for every (n, g).  q: [N][num_q_heads][head_dim]; kc, vc:
 * [B][G][t_cap][head_dim]; sel_ids [N][G][K], sel_count [N][G];
 * out: [N][num_q_heads][head_dim] fp64.                                              */
int orc_attend_batch(int N, int G, int num_q_heads, int head_dim, int region_tokens,
                     int K, int64_t t_cap, double scale,
                     const uint16_t* q, const uint16_t* kc, const uint16_t* vc,
                     const int32_t* row_seq, const int32_t* row_pos,
                     const int32_t* sel_ids, const int32_t* sel_count,
                     double* out, int nthreads);

/* The decode front end, rows in order n = 0 .. N-1: the row's indexer q, head by head,
 * through RMSNorm 1 + w into q_out [N][idx_heads][dim]; its k through LayerNorm and its
 * z as they are, written at token row_pos[n] of the caches [B][G][t_cap][dim] of
 * sequence row_seq[n]; when that token completes its region (row_pos % region_tokens
 * == region_tokens - 1), the region's summary codes into summ [B][G][r_cap][dim] (as
 * orc_summarize_region).  q_pre [N][idx_heads][dim], k_pre / z_pre [N][G][dim];
 * qw [dim], kw [dim], kb [dim] bf16 codes.  Returns 0, or -1 for a row out of range. */
int orc_indexer_front(int N, int G, int idx_heads, int dim, int region_tokens, int rope_dims,
                      int B, int64_t t_cap, int64_t r_cap, double eps,
                      const uint16_t* q_pre, const uint16_t* k_pre, const uint16_t* z_pre,
                      const uint16_t* qw, const uint16_t* kw, const uint16_t* kb,
                      const int32_t* row_seq, const int32_t* row_pos,
                      const uint16_t* cos_tab, const uint16_t* sin_tab,
                      uint16_t* q_out, uint16_t* k_cache, uint16_t* z_cache, uint8_t* summ);

#ifdef __cplusplus
}
#endif
#endif
