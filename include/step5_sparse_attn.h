/*
 * step5_sparse_attn.h -- C ABI of libstep5sa.so, the GB300 (sm_103a) implementation of
 * the Step-5 full-attention layer's sparse-indexer attention (DSA/CSA).
 *
 * The method is stated in "Step-5-Preview on one 256 GB Mac" (TensorFold PR #903), in
 * the commit that adds StepFun's CSA indexer so that contexts reach 1M tokens:
 *   (1) every completed 8-token region is summarised, per KV group, as a per-dim
 *       softmax over z of the indexer k, rounded through bf16 to e4m3;
 *   (2) a region's score in KV group g is sum_h relu(e4m3(q_h) . summary) * w_h over
 *       g's indexer heads h;
 *   (3) the 512 regions with the smallest (-score, id) keys are kept, in key order;
 *   (4) the row attends to those regions and to its own region; a row with at most
 *       512 candidate regions keeps them all, so its attention is the dense one.
 * The indexer q and k take NEOX rotation on their first 32 dims from bf16 cos/sin (same
 * page, commit on Step-5's glue).  Geometry rules follow the vLLM Step5 model's DSA
 * validation (`_validate_step5_dsa_parallel_geometry`): indexer provider groups equal
 * the attention KV groups, indexer heads divide into them, and each KV group serves
 * 4, 8 or 16 query heads.
 *
 * Conventions shared by every call
 *  - All pointers named *_bf16, *_e4m3, *_f32, sel_*, row_*, region_*, out and
 *    workspace are DEVICE pointers on the current CUDA device.  bf16 data are raw
 *    16-bit patterns, e4m3 data are OCP FP8 E4M3 ("fn") byte codes.  Every buffer is
 *    dense, row-major, in the layout written beside it.  The caller owns all memory;
 *    the library allocates nothing and never synchronises `stream`: every call only
 *    enqueues kernels on `stream` and returns.
 *  - Arguments are checked on the host before anything is enqueued; a call that
 *    returns anything but STEP5_OK has enqueued nothing.  Values that live in device
 *    memory (positions, ids, ranges) are caller preconditions; the kernels check them
 *    anyway, skip the offending item instead of touching memory out of range, and set
 *    a bit in the device status word (step5_device_status).
 *  - Positions: a query row at position p (0-based) sees keys 0..p.  Its own region is
 *    o = p / region_tokens (tokens region_tokens*o .. p); its candidate regions are
 *    0 .. o-1, so it has R(p) = p / region_tokens of them.
 */
#ifndef STEP5_SPARSE_ATTN_H
#define STEP5_SPARSE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st* step5_stream_t;

typedef enum {
    STEP5_OK = 0,
    STEP5_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, misaligned pointer     */
    STEP5_ERR_UNSUPPORTED = 2,      /* geometry outside what the kernels implement    */
    STEP5_ERR_WORKSPACE = 3,        /* workspace missing or smaller than required     */
    STEP5_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed           */
    STEP5_ERR_TIMEOUT = 5           /* a bounded device wait gave up (device status)  */
} step5_status;

/* Layer geometry.  Supported: num_kv_groups in [1, 16]; idx_heads a multiple of
 * num_kv_groups with idx_heads / num_kv_groups in {1, 2, 4, 8}; num_q_heads a multiple
 * of num_kv_groups with num_q_heads / num_kv_groups in {4, 8, 16}; head_dim 128;
 * idx_dim 64; rope_dims in {0, 16, 32, 48, 64}; region_tokens 8; 1 <= top_k <= 2048;
 * softmax_scale finite and > 0.  Step-5: {32, 4, 128, 16, 64, 32, 8, 512, 1/sqrt(128)}. */
typedef struct {
    int32_t num_q_heads;    /* attention query heads of the layer (all KV groups)     */
    int32_t num_kv_groups;  /* KV groups = indexer provider groups                    */
    int32_t head_dim;       /* attention head dim                                     */
    int32_t idx_heads;      /* indexer query heads; group g owns a contiguous block   */
    int32_t idx_dim;        /* indexer proxy dim                                      */
    int32_t rope_dims;      /* leading indexer dims rotated NEOX-style                */
    int32_t region_tokens;  /* tokens per region                                      */
    int32_t top_k;          /* regions kept per (row, KV group)                       */
    float softmax_scale;    /* attention logit scale                                  */
} step5_geometry;

/* The indexer's decode front end, ahead of step (1) ("Step-5-Preview on one 256 GB Mac",
 * CSA-indexer commit: the indexer's 16-head q takes an RMSNorm with weight 1 + w,
 * its k a LayerNorm with bias, and z stays unnormalised).  For every row n (a device [N] of sequences and positions):
 *   idx_q_out[n][h] = bf16(q_pre[n][h] / sqrt(mean_d q_pre[n][h][d]^2 + eps) * (1 + q_norm_w))
 *   idx_k[b][g][p]  = bf16((k_pre[n][g] - mean) / sqrt(var + eps) * k_norm_w + k_norm_b)
 *   idx_z[b][g][p]  = z_pre[n][g]
 * (fp32 arithmetic, one rounding; b = row_seq[n], p = row_pos[n]; the rotation of q and
 * k is left to steps (2) and (1)), and when p % 8 == 7 the summaries of region p / 8,
 * exactly as step5_region_summarize would write them.
 * q_pre [N][idx_heads][idx_dim], k_pre / z_pre [N][G][idx_dim], norm weights and bias
 * [idx_dim] (bf16, device); caches [B][G][t_cap][idx_dim], summaries
 * [B][G][r_cap][idx_dim]; rope tables as step5_region_summarize (both NULL: the
 * cache holds rotated k).  Up to 4 KV groups.  A row whose region completes reads
 * that region's other 7 tokens from the caches: rows of one call must not write into
 * one another's completing regions (decode: one row per sequence).  Out-of-range rows
 * set STEP5_DEV_RANGE and write nothing but their normalised q. */
step5_status step5_indexer_front(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap,
                                 int32_t r_cap, const void* q_pre_bf16, const void* k_pre_bf16,
                                 const void* z_pre_bf16, const void* q_norm_w_bf16,
                                 const void* k_norm_w_bf16, const void* k_norm_b_bf16, float eps,
                                 const int32_t* row_seq, const int32_t* row_pos,
                                 const void* rope_cos_bf16, const void* rope_sin_bf16,
                                 void* idx_q_out_bf16, void* idx_k_bf16, void* idx_z_bf16,
                                 uint8_t* summaries_e4m3, step5_stream_t stream);

/* Step (1): region summaries.
 * For every sequence b < B, KV group g and region r in [region_begin[b], region_end[b]):
 *   kr[t][d] = bf16(NEOX-rotated idx_k at position 8r+t) for d < rope_dims, else idx_k;
 *   s[d]     = sum_t softmax_t(idx_z[.][d]) * kr[t][d]        (fp32, t = 8r .. 8r+7)
 *   summaries_e4m3[b][g][r][d] = e4m3(bf16(s[d]))              (round to nearest even,
 *                                                                saturate at +-448)
 *   summaries_f32_or_null[b][g][r][d] = s[d]                   (if not NULL)
 * idx_k_bf16, idx_z_bf16: [B][G][t_cap][idx_dim].  rope_cos_bf16, rope_sin_bf16:
 * [t_cap][rope_dims/2], the cosine/sine of pair i at each position; both NULL means the
 * indexer k is already rotated.  region_begin, region_end: device int32 [B].
 * max_regions_per_seq: host upper bound on region_end[b] - region_begin[b] (sizes the
 * grid; regions beyond it are not summarised and set the status range bit).
 * Preconditions: 0 <= region_begin[b] <= region_end[b], region_end[b] <= r_cap,
 * 8 * region_end[b] <= t_cap.  t_cap must be a multiple of region_tokens.
 * Pointers must be 16-byte aligned. */
step5_status step5_region_summarize(const step5_geometry* geom, int32_t B, int32_t t_cap,
                                    int32_t r_cap, int32_t max_regions_per_seq,
                                    const void* idx_k_bf16, const void* idx_z_bf16,
                                    const void* rope_cos_bf16, const void* rope_sin_bf16,
                                    const int32_t* region_begin, const int32_t* region_end,
                                    uint8_t* summaries_e4m3, float* summaries_f32_or_null,
                                    step5_stream_t stream);

/* Steps (2) and (3): index scores and top-k selection, fused.
 * For every row n < N (sequence b = row_seq[n], position p = row_pos[n]) and KV group g,
 * with H = idx_heads / G heads h = g*H .. g*H+H-1:
 *   qe[h]   = e4m3(bf16(NEOX-rotated idx_q[n][h] at position p))
 *   score_r = sum_h relu( sum_d qe[h][d] * summaries[b][g][r][d] ) * w[n][h]
 *             (fp32; r < R(p); -0 is stored as +0)
 *   sel_ids[n][g][0..k) = the k = min(top_k, R(p)) region ids with the smallest keys
 *             (-score, id), in ascending key order; entries k..top_k-1 are -1.
 *   sel_count[n][g] = k.
 * idx_q_bf16: [N][idx_heads][idx_dim]; w: [N][idx_heads] fp32; row_seq, row_pos: [N].
 * rope_cos/sin: [t_cap][rope_dims/2] or both NULL (idx_q already rotated); t_cap is the
 * table length (positions must be < t_cap).  summaries_e4m3: [B][G][r_cap][idx_dim].
 * sel_ids: [N][G][top_k]; sel_count: [N][G].
 * scores_or_null: [N][G][r_cap] fp32, receives every score (entries past R(p) are not
 * written).  sel_scores_or_null: [N][G][top_k] fp32, the picked scores (-inf padding).
 * workspace: see step5_workspace_bytes / step5_workspace_init. */
step5_status step5_index_score_topk(const step5_geometry* geom, int32_t N, int32_t B,
                                    int32_t t_cap, int32_t r_cap,
                                    const void* idx_q_bf16, const float* w,
                                    const int32_t* row_seq, const int32_t* row_pos,
                                    const void* rope_cos_bf16, const void* rope_sin_bf16,
                                    const uint8_t* summaries_e4m3,
                                    int32_t* sel_ids, int32_t* sel_count,
                                    float* scores_or_null, float* sel_scores_or_null,
                                    void* workspace, size_t workspace_bytes,
                                    step5_stream_t stream);

/* Steps (2) and (3) without a caller-provided workspace (the paper has no counterpart:
 * this is a deployment variant).  For callers that cannot allocate device memory -- code
 * whose device allocations all belong to a host framework, or a path where no allocator
 * is reachable or allocating would synchronise the device -- this call takes the same
 * inputs and outputs as step5_index_score_topk and keeps its scratch in a fixed array
 * of static device memory inside the library (about 6 MiB: 4 MiB for this call's own
 * scratch after the ~2 MiB any workspace keeps for step5_sparse_attn; one array per
 * device that loads the library, held until the process exits).  It allocates nothing.
 *  - Limit: step5_workspace_bytes(geom, N, r_cap) must fit the array (for Step-5's
 *    geometry: one row up to ~322,000 summary slots, four up to ~74,000 each, sixteen up
 *    to ~12,400 each; e.g. one row at 1M tokens or four at 128K);
 *    larger problems return STEP5_ERR_WORKSPACE before anything is enqueued.
 *  - Every call looks up the array's address on the current device (a cheap lookup,
 *    so no stale address survives a device reset); the first call on a device may
 *    also load the library's device code there, so make it before any stream capture.
 *  - Each call clears the part of the array it uses (an enqueued memset), since the
 *    array keeps the previous call's contents.  All calls share the one array: calls
 *    whose executions overlap on the GPU (other streams, other threads) race. */
step5_status step5_index_score_topk_noalloc(const step5_geometry* geom, int32_t N, int32_t B,
                                            int32_t t_cap, int32_t r_cap,
                                            const void* idx_q_bf16, const float* w,
                                            const int32_t* row_seq, const int32_t* row_pos,
                                            const void* rope_cos_bf16, const void* rope_sin_bf16,
                                            const uint8_t* summaries_e4m3,
                                            int32_t* sel_ids, int32_t* sel_count,
                                            float* scores_or_null, float* sel_scores_or_null,
                                            step5_stream_t stream);

/* Step (4): attention over the picked regions plus the row's own region.
 * For every row n, query head h of KV group g = h / (num_q_heads / G):
 *   keys  = tokens 8r .. 8r+7 of every r in sel_ids[n][g][0 .. sel_count[n][g]),
 *           then the own-region tokens 8o .. p (o = p / 8)
 *   out[n][h] = softmax(softmax_scale * q[n][h] . K^T) V   (bf16 products, fp32
 *           accumulation, rounded once to bf16)
 * q_bf16: [N][num_q_heads][head_dim]; k_cache_bf16, v_cache_bf16: [B][G][t_cap][head_dim]
 * (post-rotation keys); sel_ids [N][G][top_k], sel_count [N][G] as written by
 * step5_index_score_topk (ids must be distinct candidates of the row, < o);
 * out_bf16: [N][num_q_heads][head_dim].  Cache rows past p are never read into the
 * result (they may hold anything).  t_cap must be a multiple of region_tokens; pointers
 * 16-byte aligned.
 * workspace / workspace_bytes: a workspace of step5_workspace_bytes(geom, N, any r_cap)
 * bytes, zeroed once (step5_workspace_init), or NULL / 0.  With fewer (row, group) pairs
 * than half the SMs, the call splits each pair's key list over several blocks, which
 * exchange their partial softmax states through the workspace's first part (an epoch
 * word per pair, a flag per block and ~8 KB of state per block, at most ~2.1 MiB) and
 * merge them in a fixed order; the result does not depend on timing.  NULL / 0: one
 * block per pair (slower when the pairs are few; the fp32 merge order differs, so the
 * bf16 outputs may differ in the last bit).  A non-NULL workspace smaller than that
 * part returns STEP5_ERR_WORKSPACE.  A bounded wait that gives up raises
 * STEP5_DEV_TIMEOUT (re-zero the workspace before the next call). */
step5_status step5_sparse_attn(const step5_geometry* geom, int32_t N, int32_t B,
                               int32_t t_cap, const void* q_bf16,
                               const void* k_cache_bf16, const void* v_cache_bf16,
                               const int32_t* row_seq, const int32_t* row_pos,
                               const int32_t* sel_ids, const int32_t* sel_count,
                               void* out_bf16, void* workspace, size_t workspace_bytes,
                               step5_stream_t stream);

/* Step (4) followed by the per-head sigmoid output gate ("Step-5-Preview on one 256 GB
 * Mac", native-family commit: Step-5's glue lists a per-head sigmoid gate among
 * StepFun's rounding points).  As step5_sparse_attn, except that every output dim of
 * query head h of row n is scaled by sigmoid(gate[n][h]) before the output's single
 * bf16 rounding:  out[n][h] = bf16(sigmoid(gate[n][h]) * softmax(...) V).
 * gate_bf16: [N][num_q_heads] bf16 logits (device, required; NULL returns
 * STEP5_ERR_INVALID_ARGUMENT).  Everything else as step5_sparse_attn. */
step5_status step5_sparse_attn_gated(const step5_geometry* geom, int32_t N, int32_t B,
                                     int32_t t_cap, const void* q_bf16,
                                     const void* k_cache_bf16, const void* v_cache_bf16,
                                     const int32_t* row_seq, const int32_t* row_pos,
                                     const int32_t* sel_ids, const int32_t* sel_count,
                                     const void* gate_bf16, void* out_bf16,
                                     void* workspace, size_t workspace_bytes,
                                     step5_stream_t stream);

/* Sequence-sharded decode ("Step-5-Preview on one 256 GB Mac", CSA-indexer commit:
 * the indexer is what takes Step-5 to contexts of 1M tokens; with a row's regions and
 * KV cache split over S shards (one per GPU, or processed one after another) the
 * method's result is unchanged, since:
 *  - a region among the row's top_k by (-score, id) is among its own shard's top_k, so
 *    the row's pick is the top_k of the union of the shards' picks (step5_merge_topk);
 *  - softmax attention over a union of disjoint key sets is the combine of each set's
 *    (max m, sum l, weighted sum o) state (step5_attn_combine).)
 * Every call below takes the geometry and conventions of the whole-row calls.
 *
 * Step (2)+(3) on one shard: the shard holds the summaries of regions region_lo ..
 * region_lo + r_cap_local - 1 of every sequence, summaries_e4m3 [B][G][r_cap_local][64];
 * row n's candidates in it are those below its own region, o = p / 8.  Writes that
 * shard's pick as step5_index_score_topk does, with ids the row's region ids (region_lo
 * added) and sel_scores (required) their scores.  t_cap is the rows' token capacity
 * (the rope tables' rows; positions must be below it).  region_lo >= 0.  Other
 * arguments as step5_index_score_topk (scores are not exported). */
step5_status step5_index_score_topk_shard(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap,
                                          int32_t r_cap_local, int32_t region_lo, const void* idx_q_bf16,
                                          const float* w, const int32_t* row_seq, const int32_t* row_pos,
                                          const void* rope_cos_bf16, const void* rope_sin_bf16,
                                          const uint8_t* summaries_e4m3, int32_t* sel_ids, int32_t* sel_count,
                                          float* sel_scores, void* workspace, size_t workspace_bytes,
                                          step5_stream_t stream);

/* The row's pick from S shards' picks: for each (n, g), the min(top_k, sum_s count)
 * smallest (-score, id) keys of the union of shard_ids[s][n][g][0 .. shard_counts[s][n][g])
 * (each shard's list in ascending key order, as step5_index_score_topk_shard writes
 * it; ids distinct across shards), in ascending key order; the rest of sel_ids is -1
 * (sel_scores -inf).  shard_ids, shard_scores: [S][N][G][top_k]; shard_counts [S][N][G];
 * sel_ids [N][G][top_k]; sel_count [N][G]; sel_scores_or_null [N][G][top_k] or NULL.
 * 1 <= S <= 32, S * top_k <= 16384 and N * G <= 65535, else STEP5_ERR_UNSUPPORTED.  A
 * count outside [0, top_k] raises STEP5_DEV_RANGE and is clamped. */
step5_status step5_merge_topk(const step5_geometry* geom, int32_t S, int32_t N, const int32_t* shard_ids,
                              const float* shard_scores, const int32_t* shard_counts, int32_t* sel_ids,
                              int32_t* sel_count, float* sel_scores_or_null, step5_stream_t stream);

/* step5_merge_topk, then step5_sparse_attn_shard on the merged pick, in one call (no
 * counterpart in the pages: the composition a shard runs once the shards' picks have
 * been exchanged): sel_ids [N][G][top_k] and sel_count [N][G] receive the row's pick
 * (as step5_merge_topk writes them; no picked-score export), and states_f32 this
 * shard's attention states (as step5_sparse_attn_shard writes them).  The attention
 * launch starts while the merge runs and waits for it on the device.  Every argument of
 * both calls is checked before anything is enqueued; layouts, limits and errors are
 * those of the two calls. */
step5_status step5_merge_attend_shard(const step5_geometry* geom, int32_t S, int32_t N, int32_t B,
                                      int32_t t_cap_local, int32_t token_lo, const int32_t* shard_ids,
                                      const float* shard_scores, const int32_t* shard_counts, const void* q_bf16,
                                      const void* k_cache_bf16, const void* v_cache_bf16, const int32_t* row_seq,
                                      const int32_t* row_pos, int32_t* sel_ids, int32_t* sel_count,
                                      float* states_f32, void* workspace, size_t workspace_bytes,
                                      step5_stream_t stream);

/* Step (4) on one shard: the shard's caches k_cache_bf16, v_cache_bf16
 * [B][G][t_cap_local][head_dim] hold tokens token_lo .. token_lo + t_cap_local - 1 of
 * every sequence (token_lo and t_cap_local multiples of region_tokens).  Of row n's keys
 * (the regions sel_ids picked for the whole row, then its own region) those inside the
 * shard are attended; instead of an output, the call writes per query head the state
 * (m, l, o[128]) with m the largest scaled score softmax_scale * log2(e) * q . k
 * (-inf when the shard holds none of the row's keys), l = sum 2^(s - m), o = sum
 * 2^(s - m) v (fp32; the P V product takes P in bf16 as step5_sparse_attn does):
 * states_f32 [N][num_q_heads][130], 16-byte aligned.  Positions may lie past the
 * shard.  workspace as for step5_sparse_attn. */
step5_status step5_sparse_attn_shard(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap_local,
                                     int32_t token_lo, const void* q_bf16, const void* k_cache_bf16,
                                     const void* v_cache_bf16, const int32_t* row_seq, const int32_t* row_pos,
                                     const int32_t* sel_ids, const int32_t* sel_count, float* states_f32,
                                     void* workspace, size_t workspace_bytes, step5_stream_t stream);

/* The output from S shards' states: states_f32 [S][N][num_q_heads][130] (shard s's
 * states at s * N * num_q_heads * 130); per head row, M = max_s m_s and
 *   out = bf16( sigmoid(gate) * (sum_s 2^(m_s - M) o_s) / (sum_s 2^(m_s - M) l_s) )
 * summed in shard order, with the gate factor 1 when gate_bf16_or_null is NULL
 * (gate [N][num_q_heads] bf16 logits); 0 where no shard holds a key.
 * out_bf16 [N][num_q_heads][head_dim], 16-byte aligned.  1 <= S <= 32. */
step5_status step5_attn_combine(const step5_geometry* geom, int32_t S, int32_t N, const float* states_f32,
                                const void* gate_bf16_or_null, void* out_bf16, step5_stream_t stream);

/* One whole step: step5_region_summarize, then step5_index_score_topk, then
 * step5_sparse_attn, on one stream, with the same arguments and the same results as the
 * three calls (no counterpart in the pages: a composition for serving loops).  Every
 * argument is checked before anything is enqueued; then:
 *  - summaries of regions [region_begin[b], region_end[b]) are written (skipped when
 *    max_regions_per_seq is 0; the summary inputs must still be valid pointers);
 *  - the scoring kernel reads its non-summary inputs, and the summaries of regions
 *    outside [region_begin[b], region_end[b]), before waiting for the summary kernel
 *    (that kernel writes nothing else, so the step5_set_prologue_overlap contract holds
 *    by construction here).
 * Layouts, ownership and errors are those of the three calls (scores and picked scores
 * are not exported).  workspace: as for step5_index_score_topk. */
step5_status step5_decode_step(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap, int32_t r_cap,
                               int32_t max_regions_per_seq, const void* idx_k_bf16, const void* idx_z_bf16,
                               const void* rope_cos_bf16, const void* rope_sin_bf16,
                               const int32_t* region_begin, const int32_t* region_end,
                               uint8_t* summaries_e4m3, const void* idx_q_bf16, const float* w,
                               const int32_t* row_seq, const int32_t* row_pos, const void* q_bf16,
                               const void* k_cache_bf16, const void* v_cache_bf16, int32_t* sel_ids,
                               int32_t* sel_count, void* out_bf16, void* workspace, size_t workspace_bytes,
                               step5_stream_t stream);

/* Byte offsets of a decode step's per-row inputs packed in one buffer (no counterpart in
 * the pages: the host-side form of step5_decode_step's inputs, so that a step needs one
 * host-to-device copy).  Each array starts on a 256-byte boundary, in this order:
 *   q [N][num_q_heads][head_dim] bf16, idx_q [N][idx_heads][idx_dim] bf16,
 *   w [N][idx_heads] fp32, row_seq [N] int32, row_pos [N] int32,
 *   region_begin [B] int32, region_end [B] int32;
 * total = the buffer's size in bytes. */
typedef struct {
    size_t q, idx_q, w, row_seq, row_pos, region_begin, region_end, total;
} step5_rows_layout;

/* Fills *layout for N rows and B sequences.  STEP5_ERR_INVALID_ARGUMENT for N or B <= 0
 * or a NULL layout; geometry errors as elsewhere. */
step5_status step5_rows_layout_for(const step5_geometry* geom, int32_t N, int32_t B, step5_rows_layout* layout);

/* step5_decode_step with its per-row inputs and its output in HOST memory: rows_host
 * (laid out by step5_rows_layout_for, layout.total bytes) holds the step's per-row
 * inputs and out_host ([N][num_q_heads][head_dim] bf16) receives its output.
 *  - When the device can address both (cudaHostGetDevicePointer accepts them:
 *    cudaHostAlloc / cudaMallocHost memory under unified addressing, and on Grace, where
 *    NVLink-C2C is coherent and the GPU uses the CPU's page tables, pageable memory too),
 *    the step's kernels read the inputs from rows_host and write the output into
 *    out_host in place: no copy operation is enqueued and rows_dev / out_dev are not
 *    touched.
 *  - Otherwise (or after step5_set_host_copies(1)) the call enqueues the copy of
 *    rows_host into rows_dev, the step over rows_dev's arrays and the copy of out_dev into
 *    out_host (pageable host memory works, under the runtime's synchronous-copy rules).
 * rows_dev (16-byte aligned, layout.total bytes) and out_dev are device buffers owned by
 * the caller, required in both cases.  The caches, rope tables, summaries, sel_ids,
 * sel_count and the workspace are device-resident as for step5_decode_step.  Every
 * argument is checked before anything is enqueued; results and errors are
 * step5_decode_step's, bit for bit the same in both modes.  rows_host must stay
 * unchanged, and out_host is valid, once `stream` has reached the end of the call's
 * work. */
step5_status step5_decode_step_host(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap, int32_t r_cap,
                                    int32_t max_regions_per_seq, const void* idx_k_bf16, const void* idx_z_bf16,
                                    const void* rope_cos_bf16, const void* rope_sin_bf16, uint8_t* summaries_e4m3,
                                    const void* k_cache_bf16, const void* v_cache_bf16, const void* rows_host,
                                    void* rows_dev, void* out_host, void* out_dev, int32_t* sel_ids,
                                    int32_t* sel_count, void* workspace, size_t workspace_bytes,
                                    step5_stream_t stream);

/* Bytes of device workspace that step5_index_score_topk and step5_sparse_attn need for
 * N rows and r_cap summary slots (one buffer serves both: step (4)'s part comes first
 * and depends on the geometry and N only).  Returns 0 for an unsupported geometry. */
size_t step5_workspace_bytes(const step5_geometry* geom, int32_t N, int32_t r_cap);

/* Zero-fills a workspace (enqueued on stream).  A zeroed workspace is ready for a call,
 * and every call that completes leaves it ready for the next one with the same N,
 * geometry and r_cap (its synchronisation words carry generation numbers, so they are
 * not cleared).  Zero it once after allocating it, again whenever N, the geometry or
 * r_cap change between calls on it, and after any call whose device status reported an
 * error (a bounded wait that gave up leaves the counters inconsistent). */
step5_status step5_workspace_init(void* workspace, size_t workspace_bytes, step5_stream_t stream);

/* Reads and clears the device status word of the current device: a bit mask of
 * STEP5_DEV_* flags raised by kernels since the last read.  Synchronises `stream`. */
#define STEP5_DEV_RANGE   1u  /* a position, id, range or sequence index out of bounds */
#define STEP5_DEV_TIMEOUT 2u  /* a bounded wait on an in-flight copy gave up           */
step5_status step5_device_status(uint32_t* flags_out, step5_stream_t stream);

/* Poll limit of the split selection path's waits on other blocks (the threshold word
 * and the per-(row, group) barrier of step5_index_score_topk; no counterpart in the
 * pages: a testing and tuning switch).  A wait that polls `polls` times without seeing
 * the other blocks gives up: the kernel raises STEP5_DEV_TIMEOUT, returns without
 * writing the (row, group)'s selection, and the workspace must be zeroed
 * (step5_workspace_init) before its next use.  0 restores the default (2^22 polls,
 * seconds).  Process-wide, read when a call is enqueued.  Returns the previous limit. */
uint32_t step5_set_wait_polls(uint32_t polls);

/* Kernels of step5_sparse_attn (and the gated call): 0 = automatic: with few
 * (row, group) pairs and a workspace, each pair's keys split over up to 16 blocks of one
 * thread-block cluster that merge their softmax states through distributed shared
 * memory (the workspace area is not used); otherwise one tcgen05 tensor-core CTA per
 * pair.  1 = the warp-level MMA kernel throughout, its splits (up to 64 blocks per pair)
 * merged through the workspace.  2 = one tensor-core CTA per pair, never split.  The
 * outputs agree within rounding (the fp32 sums run in different orders); each path is
 * deterministic.  A testing and tuning switch; process-wide; other values are ignored.
 * Returns the previous value. */
int32_t step5_set_attention_path(int32_t mode);

/* Selection path of step5_index_score_topk: 0 = automatic, 1 = one block per
 * (row, group) scoring on the CUDA cores and selecting in shared memory, 2 = many blocks
 * per (row, group) with a histogram threshold pass, 3 = tcgen05 tensor-core scoring of
 * blocks of rows that share a sequence (the scores go to the workspace or the caller's
 * export, and without either path 1 runs), then one selecting block per (row, group).
 * Paths 1 and 2 give identical results; path 3's scores differ from theirs only by the
 * fp32 summation order of each dot product (the e4m3 products are exact in both), so
 * its picks are the same but at near-equal scores.  A tuning and testing switch.
 * Returns the previous value. */
int32_t step5_set_select_path(int32_t mode);

/* Opt-in overlap of the scoring prologue with the launch before it (no counterpart in
 * the pages: a launch-scheduling contract of this library).  With enable = 1,
 * step5_index_score_topk's split-path kernel reads idx_q, w, row_seq, row_pos and the
 * rope tables before waiting for the kernel launched just before it on the stream
 * (programmatic dependent launch); only the summaries are read after the wait.  The
 * caller must then guarantee that this preceding kernel writes none of those inputs,
 * as step5_region_summarize does (it writes only summaries).  Default 0: every read
 * waits.  Process-wide, read when a call is enqueued; values other than 0 and 1 are
 * ignored.  Returns the previous value. */
int32_t step5_set_prologue_overlap(int32_t enable);

/* step5_decode_step_host's host-buffer access: 0 (default) = in place when the host
 * buffers are device-addressable page-locked memory, else through copies; 1 = always
 * through copies.  Process-wide; other values are ignored.  Returns the previous value. */
int32_t step5_set_host_copies(int32_t always);

/* The selection path step5_index_score_topk takes for this geometry, N rows, B sequences
 * and r_cap under the current step5_set_select_path setting (1, 2 or 3 as above; path 3
 * falls back to 1 at the call when neither a workspace nor a score export is passed); 0
 * for an unsupported geometry or non-positive sizes. */
int32_t step5_select_path_for(const step5_geometry* geom, int32_t N, int32_t B, int32_t r_cap);

/* Human-readable name of a status code (static string). */
const char* step5_status_string(step5_status status);

/* e4m3(bf16 value) for n bf16 inputs with the same device conversion the summaries use
 * (round to nearest even, saturate at +-448); in_bf16 [n] -> out_e4m3 [n]. */
step5_status step5_convert_bf16_to_e4m3(const void* in_bf16, uint8_t* out_e4m3, int64_t n,
                                        step5_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* STEP5_SPARSE_ATTN_H */
