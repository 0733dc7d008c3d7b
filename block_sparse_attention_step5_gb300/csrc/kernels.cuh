// kernels.cuh -- parameter blocks and launchers of the libstep5sa kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include <atomic>

#include "common.cuh"

namespace step5 {

// Runs set() once per CUDA device: kernel attributes belong to a device's context, so a
// process driving several GPUs sets them on each.  `done` holds a bit per device ordinal
// below 64 (others run set() on every call).
template <class F>
cudaError_t once_per_device(std::atomic<uint64_t>& done, F&& set) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = set();
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// ----------------------------------------------------------------- step (1)
struct SummarizeParams {
    const uint16_t* idx_k;   // [B][G][t_cap][64]
    const uint16_t* idx_z;   // [B][G][t_cap][64]
    const uint16_t* cos;     // [t_cap][rope_dims/2] or null
    const uint16_t* sin;
    const int32_t* region_begin;  // [B]
    const int32_t* region_end;    // [B]
    uint8_t* summ;           // [B][G][r_cap][64]
    float* summ_f32;         // [B][G][r_cap][64] or null
    uint32_t* status;
    int G, t_cap, r_cap, max_span, rope_dims;
};
cudaError_t launch_summarize(const SummarizeParams& p, int B, cudaStream_t stream);

// Summary value of dim d of the region whose first cache row is row0 (element offset of
// token 0, dim 0 in [B][G][t_cap][64]) and whose first token is position t0: the
// per-dim softmax over z of the NEOX-rotated k, in fp32 with tokens in order (not yet
// rounded).  CG: read through L2 (data written earlier in the same launch).
template <bool CG>
__device__ __forceinline__ float region_summary_dim(const uint16_t* idx_k, const uint16_t* idx_z,
                                                    const uint16_t* cos, const uint16_t* sin, int rope_dims,
                                                    int64_t row0, int t0, int d) {
    auto ld = [](const uint16_t* a) -> uint16_t { return CG ? __ldcg(a) : __ldg(a); };
    const int half = rope_dims >> 1;
    const bool rotated = cos != nullptr && d < rope_dims;
    const bool first = d < half;
    const int pd = first ? d + half : d - half;  // NEOX partner dim
    const int pi = first ? d : d - half;         // NEOX pair index
    // every load of the region is issued before any arithmetic
    uint16_t zv[8], kv[8], pv[8], cv[8], sv[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        zv[t] = ld(idx_z + row0 + t * 64 + d);
        kv[t] = ld(idx_k + row0 + t * 64 + d);
    }
    if (rotated) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int64_t tab = (int64_t)(t0 + t) * half + pi;
            pv[t] = ld(idx_k + row0 + t * 64 + pd);
            cv[t] = ld(cos + tab);
            sv[t] = ld(sin + tab);
        }
    }
    float m = -INFINITY;
#pragma unroll
    for (int t = 0; t < 8; ++t) m = fmaxf(m, bf16_to_f32(zv[t]));
    // weights and weighted sum (fp32, tokens in order)
    float den = 0.0f, num = 0.0f;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        float kr = bf16_to_f32(kv[t]);
        if (rotated)
            kr = bf16_to_f32(neox_rotate(kr, bf16_to_f32(pv[t]), bf16_to_f32(cv[t]), bf16_to_f32(sv[t]), first));
        const float e = expf(bf16_to_f32(zv[t]) - m);
        den += e;
        num = fmaf(e, kr, num);
    }
    return num / den;
}

// Decode front end: the indexer's q RMSNorm (1 + w), k LayerNorm with bias, the k/z
// cache write of the row's token and, when it completes its region, that summary.
struct FrontParams {
    const uint16_t* q_pre;   // [N][idx_heads][64]
    const uint16_t* k_pre;   // [N][G][64]
    const uint16_t* z_pre;   // [N][G][64]
    const uint16_t* q_w;     // [64]
    const uint16_t* k_w;     // [64]
    const uint16_t* k_b;     // [64]
    const int32_t* row_seq;
    const int32_t* row_pos;
    const uint16_t* cos;     // [t_cap][rope_dims/2] or null
    const uint16_t* sin;
    uint16_t* q_out;         // [N][idx_heads][64]
    uint16_t* idx_k;         // [B][G][t_cap][64]
    uint16_t* idx_z;
    uint8_t* summ;           // [B][G][r_cap][64]
    uint32_t* status;
    int N, B, G, idx_heads, t_cap, r_cap, rope_dims;
    float eps;
};
cudaError_t launch_front(const FrontParams& p, cudaStream_t stream);
cudaError_t launch_convert(const uint16_t* in, uint8_t* out, int64_t n, cudaStream_t stream);

// ----------------------------------------------------------------- steps (2) + (3)
constexpr int kHistBits = 12;
constexpr int kHistBins = 1 << kHistBits;
constexpr int kCandCap = 2048;          // candidates per (row, group) on the split path
constexpr int kFusedMaxRegions = 16384; // regions a fused block keeps in shared memory
constexpr int kMaxTopK = 2048;
constexpr int kSplitTileRegions = 1024;  // regions of one split-path scoring tile

struct ScoreParams {
    const uint16_t* idx_q;   // [N][idx_heads][64]
    const float* w;          // [N][idx_heads]
    const int32_t* row_seq;  // [N]
    const int32_t* row_pos;  // [N]
    const uint16_t* cos;     // [t_cap][rope_dims/2] or null
    const uint16_t* sin;
    const uint8_t* summ;     // [B][G][r_cap][64]
    int32_t* sel_ids;        // [N][G][top_k]
    int32_t* sel_count;      // [N][G]
    float* sel_scores;       // [N][G][top_k] or null
    float* scores;           // [N][G][r_cap]: caller's export or workspace (split path)
    uint32_t* hist;          // [N][G][kHistBins]   (split path, left zero by every call)
    uint32_t* cand_count;    // [N][G]              (split path)
    uint64_t* cand;          // [N][G][kCandCap]    (split path)
    uint32_t* arrive1;       // [N][G] histogram arrivals   (split path, left zero by every call)
    uint32_t* thr;           // [N][G] generation | threshold bin (split path)
    uint32_t* bar2;          // [N][G] generation | arrivals      (split path)
    uint32_t* status;
    int N, B, G, idx_heads, hpg, t_cap, r_cap, rope_dims, top_k;
    int region_lo;           // the summaries' first region (a shard of the rows' regions), else 0
    int shard;               // 1: a shard's call (regions past the summaries belong to other shards)
    int num_sms;             // split path: persistent blocks (one per SM)
    int overlap_prologue;    // split path: read the non-summary inputs before the launch wait
    uint32_t wait_polls;     // split path: polls of a wait on other blocks before it gives up
    // split path with overlap_prologue: the launch before writes only the summaries of
    // regions [defer_begin[b], defer_end[b]) of each sequence b; tiles clear of those
    // ranges are fetched before the launch wait (null: wait before the first tile)
    const int32_t* defer_begin;
    const int32_t* defer_end;
};
// Validated (sequence, R) of row n, or R = -1 when the row is out of range.
// Candidate regions of row n in this call's summaries: region_lo + [0, R).  A whole-row
// call needs a slot for every candidate; a shard takes those of its slots.
__device__ __forceinline__ int row_regions(const ScoreParams& p, int n, int& b, int& pos) {
    b = p.row_seq[n];
    pos = p.row_pos[n];
    if (b < 0 || b >= p.B || pos < 0 || pos >= p.t_cap) return -1;
    const int R = pos / 8 - p.region_lo;
    if (!p.shard) return R > p.r_cap ? -1 : R;
    return R < 0 ? 0 : (R > p.r_cap ? p.r_cap : R);
}

cudaError_t launch_score_fused(const ScoreParams& p, cudaStream_t stream, bool pdl);
// The selection of every (row, group) from the scores already in p.scores (one block
// each, as the fused path selects).
cudaError_t launch_select_scores(const ScoreParams& p, cudaStream_t stream, bool pdl);
// Tensor-core scoring (tcgen05, e4m3 x e4m3 into fp32 TMEM) of every candidate region of
// every row into p.scores, for launches with many rows: one CTA per (block of 128 / HPG
// rows, group).  smap: the summaries' 2-D tensor map (box 64 bytes x 256 rows, 64-byte
// swizzle).
cudaError_t launch_score_tc(const ScoreParams& p, const CUtensorMap& smap, cudaStream_t stream, bool pdl);
// Split path: one persistent launch (score, candidates, ranks) with grid barriers.
// smap: 2-D tensor map of the summaries, [B*G*r_cap rows][64 bytes], box 64 x 256,
// 64-byte swizzle (used when idx_heads / G == 4).
cudaError_t launch_score_split(const ScoreParams& p, const CUtensorMap& smap, cudaStream_t stream, bool pdl);

// ----------------------------------------------------------------- step (4)
constexpr int kAttnWarps = 8;
constexpr int kAttnStages = 2;          // pair buffers per warp (warp 0: one more)
constexpr int kAttnMaxSplits = 64;      // blocks per (row, group)
constexpr int kAttnMaxBlocks = 256;     // blocks of one launch that share a (row, group) with others
constexpr int kAttnSlotFloats = 130;    // m, l, o[128] of one head row
// upper bound of step (4)'s workspace area (epochs and flags of <= 128 pairs, 256 slots of 16 heads)
constexpr size_t kAttnAreaMaxBytes = 512 + (size_t)(kAttnMaxBlocks / 2) * kAttnMaxSplits * 4 +
                                     (size_t)kAttnMaxBlocks * 16 * kAttnSlotFloats * 4;

struct AttnParams {
    const uint16_t* q;       // [N][Hq][128]
    const int32_t* row_seq;
    const int32_t* row_pos;
    const int32_t* sel_ids;  // [N][G][top_k]
    const int32_t* sel_count;
    union {
        uint16_t* out;       // the whole row: [N][Hq][128] bf16
        float* states;       // a shard of the rows' tokens: [N][Hq][130] (m, l, o)
    };
    const uint16_t* gate;    // [N][Hq] bf16 logits of the per-head sigmoid output gate, or null
    float* part;             // splits > 1: [N*G][splits][hq_g][130] block states
    uint32_t* bar;           // splits > 1: [N*G] epoch of each (row, group)'s state exchange
    uint32_t* flags;         // splits > 1: [N*G][kAttnMaxSplits] epoch + 1 once a block's state is out
    uint32_t* status;
    int tok_lo;              // a shard: the cache's first token (else 0); the grid covers the N rows
    int B, G, Hq, hq_g, t_cap, top_k;
    int splits, entries_per_split;  // blocks per (row, group) and the entries each takes
    float scale_log2;        // softmax_scale * log2(e)
};
// (kept at 128 bytes: a larger block measurably slows the prefill launches)
static_assert(sizeof(AttnParams) == 128, "attention parameter block");
cudaError_t launch_attention(const AttnParams& p, int N, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream, bool pdl);
// the split blocks of a (row, group) as one thread-block cluster (p.splits <= 16), their
// states merged through distributed shared memory (no workspace area used)
cudaError_t launch_attention_cluster(const AttnParams& p, int N, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                     cudaStream_t stream, bool pdl);
constexpr int kAttnMaxCluster = 16;
int attention_max_clusters(int splits);  // clusters of this many blocks the GPU holds at once
// the shard instantiation (p.states in place of p.out)
cudaError_t launch_attention_shard(const AttnParams& p, int N, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                   cudaStream_t stream, bool pdl);
size_t attention_smem_bytes();  // dynamic part
// The tcgen05 kernel: one 128-thread CTA per (row, group), no split (p.splits == 1), the
// whole-row output only (no shard states).
cudaError_t launch_attention_tc(const AttnParams& p, int N, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                cudaStream_t stream, bool pdl);
size_t attention_tc_smem_bytes(int top_k);
constexpr size_t kAttnStaticSmem = (kMaxTopK + 2) * 4 + 16384;  // picked ids + merge scratch

// ----------------------------------------------------------------- sequence shards
constexpr int kMaxShards = 32;        // shards of one row (a warp's lanes in the combine)
constexpr int kMaxShardKeys = 16384;  // S * top_k keys a merge block stages (128 KB)

// The row's top K from the shards' own top K lists (each in key order).
struct MergeParams {
    const int32_t* ids;      // [S][NG][top_k] region ids of the row (global)
    const float* scores;     // [S][NG][top_k]
    const int32_t* counts;   // [S][NG]
    int32_t* sel_ids;        // [NG][top_k]
    int32_t* sel_count;      // [NG]
    float* sel_scores;       // [NG][top_k] or null
    uint32_t* status;
    int S, NG, top_k;
};
cudaError_t launch_merge(const MergeParams& p, int num_sms, cudaStream_t stream, bool pdl);

// out = (sum_s 2^(m_s - M) o_s) / (sum_s 2^(m_s - M) l_s), M = max_s m_s, per head row.
struct CombineParams {
    const float* states;     // [S][N][Hq][130] (m, l, o[128]) of each shard
    const uint16_t* gate;    // [N][Hq] bf16 gate logits or null
    uint16_t* out;           // [N][Hq][128]
    int S, N, Hq;
};
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);

}  // namespace step5
