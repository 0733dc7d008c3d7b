// step5_api.cu -- the C ABI of libstep5sa: host-side validation, workspace layout,
// TMA descriptors and kernel launches.  Declared in include/step5_sparse_attn.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "kernels.cuh"
#include "step5_sparse_attn.h"

namespace step5 {
namespace {

__device__ uint32_t g_status_word;

int32_t g_select_path = 0;  // 0 auto, 1 fused, 2 split
int32_t g_overlap_prologue = 0;
int32_t g_host_copies = 0;  // step5_decode_step_host: 1 = always through copies
uint32_t g_wait_polls = 0;  // split path's waits on other blocks: 0 = kBarrierPolls
int32_t g_attn_path = 0;    // step (4): 0 auto (split: cluster; one block per pair: tensor cores), 1 warp MMA kernel, 2 tensor cores

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Geometry check after the vLLM Step5 DSA validation (provider groups = KV groups,
// indexer heads divisible into them, 4/8/16 query heads per KV group) plus the shapes
// the kernels implement.
step5_status check_geometry(const step5_geometry* g) {
    if (g == nullptr) return STEP5_ERR_INVALID_ARGUMENT;
    if (g->num_q_heads <= 0 || g->num_kv_groups <= 0 || g->idx_heads <= 0) return STEP5_ERR_INVALID_ARGUMENT;
    if (g->num_kv_groups > 16) return STEP5_ERR_UNSUPPORTED;
    if (g->idx_heads % g->num_kv_groups) return STEP5_ERR_UNSUPPORTED;
    const int hpg = g->idx_heads / g->num_kv_groups;
    if (hpg != 1 && hpg != 2 && hpg != 4 && hpg != 8) return STEP5_ERR_UNSUPPORTED;
    if (g->num_q_heads % g->num_kv_groups) return STEP5_ERR_UNSUPPORTED;
    const int hq = g->num_q_heads / g->num_kv_groups;
    if (hq != 4 && hq != 8 && hq != 16) return STEP5_ERR_UNSUPPORTED;
    if (g->head_dim != 128 || g->idx_dim != 64 || g->region_tokens != 8) return STEP5_ERR_UNSUPPORTED;
    if (g->rope_dims < 0 || g->rope_dims > g->idx_dim || (g->rope_dims % 16) != 0) return STEP5_ERR_UNSUPPORTED;
    if (g->top_k < 1 || g->top_k > kMaxTopK) return STEP5_ERR_UNSUPPORTED;
    if (!(g->softmax_scale > 0.0f) || !isfinite(g->softmax_scale)) return STEP5_ERR_INVALID_ARGUMENT;
    return STEP5_OK;
}

uint32_t* status_ptr() {
    static uint32_t* ptr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        ptr[dev] = static_cast<uint32_t*>(p);
    }
    return ptr[dev];
}

int num_sms() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        cached[dev] = v;
    }
    return cached[dev];
}

// ------------------------------------------------------------------ workspace layout
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Step (4)'s part of the workspace: with fewer (row, group) pairs than half the SMs, a
// pair's key list is split over several blocks, which need an epoch word per pair, a
// flag per (pair, block) and one state slot (m, l, o of each head) per block.  Sized from the geometry and N alone
// (step5_sparse_attn has no r_cap); zero when no pair can be split.
struct AttnArea {
    size_t bar, flags, part, end;
    int max_blocks;
};

AttnArea attn_area(const step5_geometry* g, int N) {
    AttnArea A{0, 0, 0, 0, 0};
    const int64_t items = (int64_t)N * g->num_kv_groups;
    const int hq_g = g->num_q_heads / g->num_kv_groups;
    if (2 * items > kAttnMaxBlocks) return A;
    const int64_t blocks = std::min<int64_t>(items * kAttnMaxSplits, kAttnMaxBlocks);
    A.max_blocks = (int)blocks;
    A.bar = 0;
    A.flags = align256((size_t)items * 4);
    A.part = align256(A.flags + (size_t)items * kAttnMaxSplits * 4);
    A.end = align256(A.part + (size_t)blocks * hq_g * kAttnSlotFloats * 4);
    return A;
}

// How step (4) splits a row's (top_k + 1)-entry key list: S blocks per (row, group),
// as many as the SMs allow with one block per SM for the whole launch (the gather of
// each block runs at a per-SM rate, so the more SMs the better), at most 64 and at least
// 16 outputs of the final merge per block; S = 1 without a workspace area.  Each block
// takes `eps` entries (whole pairs).
void attn_plan(const step5_geometry* g, int N, bool split_area, int* splits_out, int* eps_out, bool query_device) {
    const int E = g->top_k + 1;
    const int64_t items = (int64_t)N * g->num_kv_groups;
    const int hq_g = g->num_q_heads / g->num_kv_groups;
    const int sms = query_device ? num_sms() : 152;
    int64_t S = 1;
    if (split_area) {
        const AttnArea A = attn_area(g, N);
        S = std::min<int64_t>({(int64_t)kAttnMaxSplits, sms / items, (int64_t)(hq_g * 128 + 15) / 16,
                               (int64_t)A.max_blocks / items});
        if (S < 1) S = 1;
    }
    int eps = (int)((E + S - 1) / S);
    eps = (eps + 1) / 2 * 2;
    *splits_out = (int)S;
    *eps_out = eps;
}

// Workspace: step (4)'s area first (its offset depends on the geometry and N only),
// then step (2)-(3)'s, whose zero-maintained parts (histograms and counters) come first.
struct Layout {
    size_t hist, cand_count, arrive1, thr, bar2, scores, cand, end;
};

Layout layout(const step5_geometry* g, int N, int r_cap) {
    Layout L;
    const int G = g->num_kv_groups;
    const size_t ng = (size_t)N * G;
    L.hist = attn_area(g, N).end;
    L.cand_count = align256(L.hist + ng * kHistBins * 4);
    L.arrive1 = align256(L.cand_count + ng * 4);
    L.thr = align256(L.arrive1 + ng * 4);
    L.bar2 = align256(L.thr + ng * 4);
    L.scores = align256(L.bar2 + ng * 4);
    L.cand = align256(L.scores + ng * (size_t)(r_cap > 0 ? r_cap : 0) * 4);
    L.end = align256(L.cand + ng * kCandCap * 8);
    return L;
}

// ------------------------------------------------------------------ TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D view of a [B][G][t_cap][128] bf16 cache as (64 dims, rows, 2 halves of a row):
// one box (64 x 8 x 2) is a whole 8-token region, landing in shared memory as two
// 1 KB half tiles [half][token][64 dims] with 128-byte swizzle.
bool encode_cache_map(CUtensorMap* map, const void* base, uint64_t rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, rows, 2};
    cuuint64_t strides[2] = {256, 128};  // bytes: next row, next half
    cuuint32_t box[3] = {64, 8, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D view [rows][64] bytes of the e4m3 summaries; box 64 bytes x 256 rows, 64-byte
// swizzle.
bool encode_summary_map(CUtensorMap* map, const void* base, uint64_t rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {64, rows};
    cuuint64_t strides[1] = {64};
    cuuint32_t box[2] = {64, 256};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct SummaryMapCache {
    std::mutex mu;
    const void* ptr = nullptr;
    uint64_t rows = 0;
    CUtensorMap map;
};
SummaryMapCache g_smap;

bool cache_summary_map(const void* ptr, uint64_t rows, CUtensorMap* out) {
    std::lock_guard<std::mutex> lock(g_smap.mu);
    if (g_smap.ptr != ptr || g_smap.rows != rows) {
        if (!encode_summary_map(&g_smap.map, ptr, rows)) {
            g_smap.ptr = nullptr;
            return false;
        }
        g_smap.ptr = ptr;
        g_smap.rows = rows;
    }
    *out = g_smap.map;
    return true;
}

struct MapCache {
    std::mutex mu;
    const void* kptr = nullptr;
    const void* vptr = nullptr;
    uint64_t rows = 0;
    CUtensorMap k, v;
};
MapCache g_maps;

bool cache_maps(const void* kptr, const void* vptr, uint64_t rows, CUtensorMap* k, CUtensorMap* v) {
    std::lock_guard<std::mutex> lock(g_maps.mu);
    if (g_maps.kptr != kptr || g_maps.vptr != vptr || g_maps.rows != rows) {
        if (!encode_cache_map(&g_maps.k, kptr, rows) || !encode_cache_map(&g_maps.v, vptr, rows)) {
            g_maps.kptr = g_maps.vptr = nullptr;
            return false;
        }
        g_maps.kptr = kptr;
        g_maps.vptr = vptr;
        g_maps.rows = rows;
    }
    *k = g_maps.k;
    *v = g_maps.v;
    return true;
}

bool use_pdl() { return true; }



// Selection paths of steps (2)-(3): 1 = fused (one block per (row, group) scores on the
// CUDA cores and selects in shared memory), 2 = split (one persistent launch whose blocks
// share each (row, group)'s regions), 3 = tensor-core scoring of blocks of rows that share
// a sequence, then one selecting block per (row, group).
// Fused vs split was measured on GB300 (eager calls after an L2 flush, summaries built
// from k and z): the split path's time grows with the (row, group) count NG (23-25 us at
// NG = 4, 33 at 16, 37 at 32, 42 at 64), the fused path's with the regions per row (25 us
// at 2,050, 31 at 4,000, 41 at 6,000); the crossover moves from ~3,000 regions at NG = 4
// to past 3,842 at NG = 64.  The tensor-core path needs rows that share their sequence's
// summaries (it scores a block of rows against one sequence's summaries at a time): taken
// for many rows (NG >= 128) with at least 8 rows per sequence on average.
int choose_path(const step5_geometry* geom, int N, int B, int r_cap) {
    const int G = geom->num_kv_groups;
    const int hpg = geom->idx_heads / G;
    int P2 = 1;
    while (P2 < geom->top_k) P2 <<= 1;
    const int fused_need = (P2 + (P2 > 512 ? P2 : 512)) * 8 + ((r_cap + 3) & ~3) * 4 + hpg * 64 * 4;
    const bool fused_fits = r_cap <= kFusedMaxRegions && fused_need <= 200 * 1024;
    int path;
    if (g_select_path == 1 || g_select_path == 2 || g_select_path == 3)
        path = g_select_path;
    else if ((int64_t)N * G >= 128 && (int64_t)N >= 8 * (int64_t)B)
        path = 3;
    else
        path = ((int64_t)N * G >= 128 || r_cap <= 2800 + 45 * N * G) ? 1 : 2;
    if (path != 2 && !fused_fits) path = 2;  // the selecting block keeps a row's keys on chip
    return path;
}

}  // namespace
}  // namespace step5

#ifdef STEP5_TRACE
__device__ unsigned long long* step5::g_trace = nullptr;
#endif

using namespace step5;

extern "C" {

#ifdef STEP5_TRACE
// Trace builds only: registers the device buffer the phase stamps go to (NULL stops).
int step5_trace_buffer(void* device_buffer) {
    return (int)cudaMemcpyToSymbol(g_trace, &device_buffer, sizeof(device_buffer));
}
#endif

const char* step5_status_string(step5_status s) {
    switch (s) {
        case STEP5_OK: return "ok";
        case STEP5_ERR_INVALID_ARGUMENT: return "invalid argument";
        case STEP5_ERR_UNSUPPORTED: return "unsupported geometry";
        case STEP5_ERR_WORKSPACE: return "workspace missing or too small";
        case STEP5_ERR_CUDA: return "CUDA error";
        case STEP5_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

int32_t step5_set_host_copies(int32_t always) {
    const int32_t prev = g_host_copies;
    if (always == 0 || always == 1) g_host_copies = always;
    return prev;
}

int32_t step5_set_prologue_overlap(int32_t enable) {
    const int32_t prev = g_overlap_prologue;
    if (enable == 0 || enable == 1) g_overlap_prologue = enable;
    return prev;
}

uint32_t step5_set_wait_polls(uint32_t polls) {
    const uint32_t prev = g_wait_polls ? g_wait_polls : kBarrierPolls;
    g_wait_polls = polls;
    return prev;
}

int32_t step5_set_attention_path(int32_t mode) {
    const int32_t prev = g_attn_path;
    if (mode >= 0 && mode <= 2) g_attn_path = mode;
    return prev;
}

int32_t step5_set_select_path(int32_t mode) {
    const int32_t prev = g_select_path;
    if (mode >= 0 && mode <= 3) g_select_path = mode;
    return prev;
}

int32_t step5_select_path_for(const step5_geometry* geom, int32_t N, int32_t B, int32_t r_cap) {
    if (check_geometry(geom) != STEP5_OK || N <= 0 || B <= 0 || r_cap <= 0) return 0;
    return choose_path(geom, N, B, r_cap);
}

size_t step5_workspace_bytes(const step5_geometry* geom, int32_t N, int32_t r_cap) {
    if (check_geometry(geom) != STEP5_OK || N <= 0 || r_cap <= 0) return 0;
    return layout(geom, N, r_cap).end;
}

step5_status step5_workspace_init(void* workspace, size_t workspace_bytes, step5_stream_t stream) {
    if (workspace == nullptr || workspace_bytes == 0) return STEP5_ERR_INVALID_ARGUMENT;
    if (cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream) != cudaSuccess) return STEP5_ERR_CUDA;
    return STEP5_OK;
}

step5_status step5_device_status(uint32_t* flags_out, step5_stream_t stream) {
    if (flags_out == nullptr) return STEP5_ERR_INVALID_ARGUMENT;
    uint32_t* st = status_ptr();
    if (!st) return STEP5_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, st, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess) return STEP5_ERR_CUDA;
    if (cudaMemsetAsync(st, 0, 4, (cudaStream_t)stream) != cudaSuccess) return STEP5_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return STEP5_ERR_CUDA;
    *flags_out = v;
    return (v & STEP5_DEV_TIMEOUT) ? STEP5_ERR_TIMEOUT : STEP5_OK;
}

step5_status step5_convert_bf16_to_e4m3(const void* in_bf16, uint8_t* out_e4m3, int64_t n, step5_stream_t stream) {
    if (n < 0 || (n > 0 && (in_bf16 == nullptr || out_e4m3 == nullptr))) return STEP5_ERR_INVALID_ARGUMENT;
    if (n == 0) return STEP5_OK;
    if (launch_convert(static_cast<const uint16_t*>(in_bf16), out_e4m3, n, (cudaStream_t)stream) != cudaSuccess)
        return STEP5_ERR_CUDA;
    return STEP5_OK;
}

}  // extern "C"

namespace {

// The three calls, each as validation (launch = false: returns the status the call would
// return for its arguments, enqueues nothing) or validation + launch.
step5_status summarize_impl(const step5_geometry* geom, int32_t B, int32_t t_cap, int32_t r_cap,
                            int32_t max_regions_per_seq, const void* idx_k_bf16, const void* idx_z_bf16,
                            const void* rope_cos_bf16, const void* rope_sin_bf16, const int32_t* region_begin,
                            const int32_t* region_end, uint8_t* summaries_e4m3, float* summaries_f32_or_null,
                            step5_stream_t stream, bool launch) {
    step5_status s = check_geometry(geom);
    if (s != STEP5_OK) return s;
    if (B <= 0 || t_cap <= 0 || r_cap <= 0 || max_regions_per_seq < 0) return STEP5_ERR_INVALID_ARGUMENT;
    if (t_cap % geom->region_tokens) return STEP5_ERR_INVALID_ARGUMENT;
    if (!idx_k_bf16 || !idx_z_bf16 || !region_begin || !region_end || !summaries_e4m3)
        return STEP5_ERR_INVALID_ARGUMENT;
    if ((rope_cos_bf16 == nullptr) != (rope_sin_bf16 == nullptr)) return STEP5_ERR_INVALID_ARGUMENT;
    if (!aligned16(idx_k_bf16) || !aligned16(idx_z_bf16) || !aligned16(summaries_e4m3) ||
        !aligned16(summaries_f32_or_null) || !aligned16(rope_cos_bf16) || !aligned16(rope_sin_bf16))
        return STEP5_ERR_INVALID_ARGUMENT;
    if ((int64_t)B * geom->num_kv_groups * t_cap > INT32_MAX) return STEP5_ERR_INVALID_ARGUMENT;
    if (max_regions_per_seq == 0 || !launch) return STEP5_OK;
    uint32_t* st = status_ptr();
    if (!st) return STEP5_ERR_CUDA;
    SummarizeParams p;
    p.idx_k = static_cast<const uint16_t*>(idx_k_bf16);
    p.idx_z = static_cast<const uint16_t*>(idx_z_bf16);
    p.cos = static_cast<const uint16_t*>(rope_cos_bf16);
    p.sin = static_cast<const uint16_t*>(rope_sin_bf16);
    p.region_begin = region_begin;
    p.region_end = region_end;
    p.summ = summaries_e4m3;
    p.summ_f32 = summaries_f32_or_null;
    p.status = st;
    p.G = geom->num_kv_groups;
    p.t_cap = t_cap;
    p.r_cap = r_cap;
    p.max_span = max_regions_per_seq;
    p.rope_dims = rope_cos_bf16 ? geom->rope_dims : 0;
    if (launch_summarize(p, B, (cudaStream_t)stream) != cudaSuccess) return STEP5_ERR_CUDA;
    return STEP5_OK;
}

step5_status score_impl(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap, int32_t r_cap,
                        const void* idx_q_bf16, const float* w, const int32_t* row_seq, const int32_t* row_pos,
                        const void* rope_cos_bf16, const void* rope_sin_bf16, const uint8_t* summaries_e4m3,
                        int32_t* sel_ids, int32_t* sel_count, float* scores_or_null, float* sel_scores_or_null,
                        void* workspace, size_t workspace_bytes, step5_stream_t stream, int overlap,
                        const int32_t* defer_begin, const int32_t* defer_end, bool launch,
                        int32_t region_lo = 0, bool shard = false) {
    step5_status s = check_geometry(geom);
    if (s != STEP5_OK) return s;
    if (N <= 0 || B <= 0 || t_cap <= 0 || r_cap <= 0) return STEP5_ERR_INVALID_ARGUMENT;
    if (N > 65535) return STEP5_ERR_UNSUPPORTED;
    if (!idx_q_bf16 || !w || !row_seq || !row_pos || !summaries_e4m3 || !sel_ids || !sel_count)
        return STEP5_ERR_INVALID_ARGUMENT;
    if ((rope_cos_bf16 == nullptr) != (rope_sin_bf16 == nullptr)) return STEP5_ERR_INVALID_ARGUMENT;
    if (!aligned16(summaries_e4m3) || !aligned16(idx_q_bf16)) return STEP5_ERR_INVALID_ARGUMENT;
    const int G = geom->num_kv_groups;
    const int hpg = geom->idx_heads / G;
    int path = choose_path(geom, N, B, r_cap);
    const Layout L = layout(geom, N, r_cap);
    // the tensor-core path keeps every score in the workspace (or the caller's export);
    // without either, the fused path runs
    if (path == 3 && scores_or_null == nullptr && (workspace == nullptr || workspace_bytes < L.end)) path = 1;
    const bool fused = path == 1;
    if (path == 2) {
        if (workspace == nullptr) return STEP5_ERR_WORKSPACE;
        if (workspace_bytes < L.end) return STEP5_ERR_WORKSPACE;
    }
    if (path != 1 && (uint64_t)B * G * r_cap > (uint64_t)INT32_MAX - kSplitTileRegions)
        return STEP5_ERR_INVALID_ARGUMENT;
    if (!launch) return STEP5_OK;
    uint32_t* st = status_ptr();
    if (!st) return STEP5_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    ScoreParams p;
    p.idx_q = static_cast<const uint16_t*>(idx_q_bf16);
    p.w = w;
    p.row_seq = row_seq;
    p.row_pos = row_pos;
    p.cos = static_cast<const uint16_t*>(rope_cos_bf16);
    p.sin = static_cast<const uint16_t*>(rope_sin_bf16);
    p.summ = summaries_e4m3;
    p.sel_ids = sel_ids;
    p.sel_count = sel_count;
    p.sel_scores = sel_scores_or_null;
    const bool split = path == 2;
    p.scores = scores_or_null ? scores_or_null : (fused ? nullptr : reinterpret_cast<float*>(ws + L.scores));
    p.hist = split ? reinterpret_cast<uint32_t*>(ws + L.hist) : nullptr;
    p.cand_count = split ? reinterpret_cast<uint32_t*>(ws + L.cand_count) : nullptr;
    p.cand = split ? reinterpret_cast<uint64_t*>(ws + L.cand) : nullptr;
    p.arrive1 = split ? reinterpret_cast<uint32_t*>(ws + L.arrive1) : nullptr;
    p.thr = split ? reinterpret_cast<uint32_t*>(ws + L.thr) : nullptr;
    p.bar2 = split ? reinterpret_cast<uint32_t*>(ws + L.bar2) : nullptr;
    p.num_sms = num_sms();
    p.overlap_prologue = overlap;
    p.wait_polls = g_wait_polls ? g_wait_polls : kBarrierPolls;
    p.defer_begin = overlap ? defer_begin : nullptr;
    p.defer_end = overlap ? defer_end : nullptr;
    p.status = st;
    p.N = N;
    p.B = B;
    p.G = G;
    p.idx_heads = geom->idx_heads;
    p.hpg = hpg;
    p.t_cap = t_cap;
    p.r_cap = r_cap;
    p.rope_dims = rope_cos_bf16 ? geom->rope_dims : 0;
    p.region_lo = region_lo;
    p.shard = shard ? 1 : 0;
    p.top_k = geom->top_k;
    cudaError_t e;
    if (fused) {
        e = launch_score_fused(p, (cudaStream_t)stream, use_pdl());
    } else {
        CUtensorMap smap;
        const uint64_t srows = (uint64_t)B * G * r_cap;
        if (!cache_summary_map(summaries_e4m3, srows, &smap)) return STEP5_ERR_CUDA;
        if (split) {
            e = launch_score_split(p, smap, (cudaStream_t)stream, use_pdl());
        } else {
            e = launch_score_tc(p, smap, (cudaStream_t)stream, use_pdl());
            if (e == cudaSuccess) e = launch_select_scores(p, (cudaStream_t)stream, true);
        }
    }
    return e == cudaSuccess ? STEP5_OK : STEP5_ERR_CUDA;
}

step5_status attn_impl(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap, const void* q_bf16,
                       const void* k_cache_bf16, const void* v_cache_bf16, const int32_t* row_seq,
                       const int32_t* row_pos, const int32_t* sel_ids, const int32_t* sel_count, void* out_bf16,
                       void* workspace, size_t workspace_bytes, step5_stream_t stream, bool launch,
                       const void* gate_bf16 = nullptr, float* states = nullptr, int32_t tok_lo = 0) {
    step5_status s = check_geometry(geom);
    if (s != STEP5_OK) return s;
    if (N <= 0 || B <= 0 || t_cap <= 0 || (t_cap % geom->region_tokens)) return STEP5_ERR_INVALID_ARGUMENT;
    if (N > 65535) return STEP5_ERR_UNSUPPORTED;
    if (!q_bf16 || !k_cache_bf16 || !v_cache_bf16 || !row_seq || !row_pos || !sel_ids || !sel_count ||
        (out_bf16 == nullptr) == (states == nullptr))
        return STEP5_ERR_INVALID_ARGUMENT;
    if (!aligned16(q_bf16) || !aligned16(k_cache_bf16) || !aligned16(v_cache_bf16) ||
        (out_bf16 && !aligned16(out_bf16)) || (states && !aligned16(states)))
        return STEP5_ERR_INVALID_ARGUMENT;
    if (tok_lo < 0 || tok_lo % geom->region_tokens || (int64_t)tok_lo + t_cap > INT32_MAX)
        return STEP5_ERR_INVALID_ARGUMENT;
    const int G = geom->num_kv_groups;
    const uint64_t rows = (uint64_t)B * G * t_cap;
    if (rows > (uint64_t)INT32_MAX) return STEP5_ERR_INVALID_ARGUMENT;
    const AttnArea A = attn_area(geom, N);
    const bool use_area = workspace != nullptr && workspace_bytes > 0 && A.end > 0;
    if (use_area && workspace_bytes < A.end) return STEP5_ERR_WORKSPACE;
    if (!launch) return STEP5_OK;

    uint32_t* st = status_ptr();
    if (!st) return STEP5_ERR_CUDA;
    int splits, eps;
    attn_plan(geom, N, use_area, &splits, &eps, true);
    // the split blocks of a (row, group) as one cluster merging through distributed
    // shared memory (whole rows, automatic path): the largest cluster of at most 16
    // blocks whose clusters for every pair fit the GPCs at once (a cluster must sit in
    // one GPC; a second wave of clusters would cost more than the merge saves)
    bool cluster = false;
    if (states == nullptr && g_attn_path == 0 && splits > 1) {
        const int64_t pairs = (int64_t)N * geom->num_kv_groups;
        for (int cs = splits < kAttnMaxCluster ? splits : kAttnMaxCluster; cs >= 2; --cs) {
            if (attention_max_clusters(cs) >= pairs) {
                cluster = true;
                splits = cs;
                eps = (geom->top_k + 1 + splits - 1) / splits;
                eps = (eps + 1) / 2 * 2;
                break;
            }
        }
    }
    CUtensorMap kmap, vmap;
    if (!cache_maps(k_cache_bf16, v_cache_bf16, rows, &kmap, &vmap)) return STEP5_ERR_CUDA;
    AttnParams p;
    p.q = static_cast<const uint16_t*>(q_bf16);
    p.row_seq = row_seq;
    p.row_pos = row_pos;
    p.sel_ids = sel_ids;
    p.sel_count = sel_count;
    if (states != nullptr)
        p.states = states;
    else
        p.out = static_cast<uint16_t*>(out_bf16);
    p.gate = static_cast<const uint16_t*>(gate_bf16);
    p.tok_lo = tok_lo;
    p.status = st;
    p.B = B;
    p.G = G;
    p.Hq = geom->num_q_heads;
    p.hq_g = geom->num_q_heads / G;
    p.t_cap = t_cap;
    p.top_k = geom->top_k;
    p.splits = splits;
    p.entries_per_split = eps;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.bar = splits > 1 ? reinterpret_cast<uint32_t*>(ws + A.bar) : nullptr;
    p.flags = splits > 1 ? reinterpret_cast<uint32_t*>(ws + A.flags) : nullptr;
    p.part = splits > 1 ? reinterpret_cast<float*>(ws + A.part) : nullptr;
    p.scale_log2 = geom->softmax_scale * 1.4426950408889634f;
    cudaError_t e;
    if (states != nullptr)
        e = launch_attention_shard(p, N, kmap, vmap, (cudaStream_t)stream, use_pdl());
    else if (cluster)
        e = launch_attention_cluster(p, N, kmap, vmap, (cudaStream_t)stream, use_pdl());
    else if (splits == 1 && g_attn_path != 1)
        e = launch_attention_tc(p, N, kmap, vmap, (cudaStream_t)stream, use_pdl());
    else
        e = launch_attention(p, N, kmap, vmap, (cudaStream_t)stream, use_pdl());
    return e == cudaSuccess ? STEP5_OK : STEP5_ERR_CUDA;
}

}  // namespace

extern "C" {

step5_status step5_region_summarize(const step5_geometry* geom, int32_t B, int32_t t_cap, int32_t r_cap,
                                    int32_t max_regions_per_seq, const void* idx_k_bf16, const void* idx_z_bf16,
                                    const void* rope_cos_bf16, const void* rope_sin_bf16,
                                    const int32_t* region_begin, const int32_t* region_end,
                                    uint8_t* summaries_e4m3, float* summaries_f32_or_null, step5_stream_t stream) {
    return summarize_impl(geom, B, t_cap, r_cap, max_regions_per_seq, idx_k_bf16, idx_z_bf16, rope_cos_bf16,
                          rope_sin_bf16, region_begin, region_end, summaries_e4m3, summaries_f32_or_null, stream,
                          true);
}

step5_status step5_index_score_topk(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap, int32_t r_cap,
                                    const void* idx_q_bf16, const float* w, const int32_t* row_seq,
                                    const int32_t* row_pos, const void* rope_cos_bf16, const void* rope_sin_bf16,
                                    const uint8_t* summaries_e4m3, int32_t* sel_ids, int32_t* sel_count,
                                    float* scores_or_null, float* sel_scores_or_null, void* workspace,
                                    size_t workspace_bytes, step5_stream_t stream) {
    return score_impl(geom, N, B, t_cap, r_cap, idx_q_bf16, w, row_seq, row_pos, rope_cos_bf16, rope_sin_bf16,
                      summaries_e4m3, sel_ids, sel_count, scores_or_null, sel_scores_or_null, workspace,
                      workspace_bytes, stream, g_overlap_prologue, nullptr, nullptr, true);
}

step5_status step5_index_score_topk_shard(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap,
                                          int32_t r_cap_local, int32_t region_lo, const void* idx_q_bf16,
                                          const float* w, const int32_t* row_seq, const int32_t* row_pos,
                                          const void* rope_cos_bf16, const void* rope_sin_bf16,
                                          const uint8_t* summaries_e4m3, int32_t* sel_ids, int32_t* sel_count,
                                          float* sel_scores, void* workspace, size_t workspace_bytes,
                                          step5_stream_t stream) {
    if (region_lo < 0 || sel_scores == nullptr) return STEP5_ERR_INVALID_ARGUMENT;
    if ((int64_t)region_lo + r_cap_local > INT32_MAX / 8) return STEP5_ERR_INVALID_ARGUMENT;
    return score_impl(geom, N, B, t_cap, r_cap_local, idx_q_bf16, w, row_seq, row_pos, rope_cos_bf16,
                      rope_sin_bf16, summaries_e4m3, sel_ids, sel_count, nullptr, sel_scores, workspace,
                      workspace_bytes, stream, g_overlap_prologue, nullptr, nullptr, true, region_lo, true);
}

step5_status step5_sparse_attn(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap, const void* q_bf16,
                               const void* k_cache_bf16, const void* v_cache_bf16, const int32_t* row_seq,
                               const int32_t* row_pos, const int32_t* sel_ids, const int32_t* sel_count,
                               void* out_bf16, void* workspace, size_t workspace_bytes, step5_stream_t stream) {
    return attn_impl(geom, N, B, t_cap, q_bf16, k_cache_bf16, v_cache_bf16, row_seq, row_pos, sel_ids, sel_count,
                     out_bf16, workspace, workspace_bytes, stream, true);
}

step5_status step5_sparse_attn_gated(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap,
                                     const void* q_bf16, const void* k_cache_bf16, const void* v_cache_bf16,
                                     const int32_t* row_seq, const int32_t* row_pos, const int32_t* sel_ids,
                                     const int32_t* sel_count, const void* gate_bf16, void* out_bf16,
                                     void* workspace, size_t workspace_bytes, step5_stream_t stream) {
    if (gate_bf16 == nullptr) return STEP5_ERR_INVALID_ARGUMENT;
    return attn_impl(geom, N, B, t_cap, q_bf16, k_cache_bf16, v_cache_bf16, row_seq, row_pos, sel_ids, sel_count,
                     out_bf16, workspace, workspace_bytes, stream, true, gate_bf16);
}

step5_status step5_sparse_attn_shard(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap_local,
                                     int32_t token_lo, const void* q_bf16, const void* k_cache_bf16,
                                     const void* v_cache_bf16, const int32_t* row_seq, const int32_t* row_pos,
                                     const int32_t* sel_ids, const int32_t* sel_count, float* states_f32,
                                     void* workspace, size_t workspace_bytes, step5_stream_t stream) {
    if (states_f32 == nullptr) return STEP5_ERR_INVALID_ARGUMENT;
    return attn_impl(geom, N, B, t_cap_local, q_bf16, k_cache_bf16, v_cache_bf16, row_seq, row_pos, sel_ids,
                     sel_count, nullptr, workspace, workspace_bytes, stream, true, nullptr, states_f32, token_lo);
}

}  // extern "C"

namespace {

step5_status merge_impl(const step5_geometry* geom, int32_t S, int32_t N, const int32_t* shard_ids,
                        const float* shard_scores, const int32_t* shard_counts, int32_t* sel_ids, int32_t* sel_count,
                        float* sel_scores_or_null, step5_stream_t stream, bool launch) {
    step5_status s = check_geometry(geom);
    if (s != STEP5_OK) return s;
    if (S <= 0 || N <= 0) return STEP5_ERR_INVALID_ARGUMENT;
    if (!shard_ids || !shard_scores || !shard_counts || !sel_ids || !sel_count) return STEP5_ERR_INVALID_ARGUMENT;
    const int64_t NG = (int64_t)N * geom->num_kv_groups;
    if (NG > 65535) return STEP5_ERR_UNSUPPORTED;
    if (S > kMaxShards || (int64_t)S * geom->top_k > kMaxShardKeys) return STEP5_ERR_UNSUPPORTED;
    if (!launch) return STEP5_OK;
    uint32_t* st = status_ptr();
    if (!st) return STEP5_ERR_CUDA;
    MergeParams p;
    p.ids = shard_ids;
    p.scores = shard_scores;
    p.counts = shard_counts;
    p.sel_ids = sel_ids;
    p.sel_count = sel_count;
    p.sel_scores = sel_scores_or_null;
    p.status = st;
    p.S = S;
    p.NG = (int)NG;
    p.top_k = geom->top_k;
    return launch_merge(p, num_sms(), (cudaStream_t)stream, use_pdl()) == cudaSuccess ? STEP5_OK : STEP5_ERR_CUDA;
}

}  // namespace

extern "C" {

step5_status step5_merge_topk(const step5_geometry* geom, int32_t S, int32_t N, const int32_t* shard_ids,
                              const float* shard_scores, const int32_t* shard_counts, int32_t* sel_ids,
                              int32_t* sel_count, float* sel_scores_or_null, step5_stream_t stream) {
    return merge_impl(geom, S, N, shard_ids, shard_scores, shard_counts, sel_ids, sel_count, sel_scores_or_null,
                      stream, true);
}

step5_status step5_merge_attend_shard(const step5_geometry* geom, int32_t S, int32_t N, int32_t B,
                                      int32_t t_cap_local, int32_t token_lo, const int32_t* shard_ids,
                                      const float* shard_scores, const int32_t* shard_counts, const void* q_bf16,
                                      const void* k_cache_bf16, const void* v_cache_bf16, const int32_t* row_seq,
                                      const int32_t* row_pos, int32_t* sel_ids, int32_t* sel_count,
                                      float* states_f32, void* workspace, size_t workspace_bytes,
                                      step5_stream_t stream) {
    // every argument is checked before anything is enqueued
    step5_status s = merge_impl(geom, S, N, shard_ids, shard_scores, shard_counts, sel_ids, sel_count, nullptr,
                                stream, false);
    if (s != STEP5_OK) return s;
    if (states_f32 == nullptr) return STEP5_ERR_INVALID_ARGUMENT;
    s = attn_impl(geom, N, B, t_cap_local, q_bf16, k_cache_bf16, v_cache_bf16, row_seq, row_pos, sel_ids, sel_count,
                  nullptr, workspace, workspace_bytes, stream, false, nullptr, states_f32, token_lo);
    if (s != STEP5_OK) return s;
    s = merge_impl(geom, S, N, shard_ids, shard_scores, shard_counts, sel_ids, sel_count, nullptr, stream, true);
    if (s != STEP5_OK) return s;
    // the attention launch waits for the merge through its programmatic-launch wait
    return attn_impl(geom, N, B, t_cap_local, q_bf16, k_cache_bf16, v_cache_bf16, row_seq, row_pos, sel_ids,
                     sel_count, nullptr, workspace, workspace_bytes, stream, true, nullptr, states_f32, token_lo);
}

step5_status step5_attn_combine(const step5_geometry* geom, int32_t S, int32_t N, const float* states_f32,
                                const void* gate_bf16_or_null, void* out_bf16, step5_stream_t stream) {
    step5_status s = check_geometry(geom);
    if (s != STEP5_OK) return s;
    if (S <= 0 || N <= 0 || !states_f32 || !out_bf16 || !aligned16(out_bf16)) return STEP5_ERR_INVALID_ARGUMENT;
    if (S > kMaxShards) return STEP5_ERR_UNSUPPORTED;
    if ((int64_t)N * geom->num_q_heads * kAttnSlotFloats * S > ((int64_t)1 << 40)) return STEP5_ERR_INVALID_ARGUMENT;
    CombineParams p;
    p.states = states_f32;
    p.gate = static_cast<const uint16_t*>(gate_bf16_or_null);
    p.out = static_cast<uint16_t*>(out_bf16);
    p.S = S;
    p.N = N;
    p.Hq = geom->num_q_heads;
    return launch_combine(p, (cudaStream_t)stream) == cudaSuccess ? STEP5_OK : STEP5_ERR_CUDA;
}

step5_status step5_indexer_front(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap, int32_t r_cap,
                                 const void* q_pre_bf16, const void* k_pre_bf16, const void* z_pre_bf16,
                                 const void* q_norm_w_bf16, const void* k_norm_w_bf16, const void* k_norm_b_bf16,
                                 float eps, const int32_t* row_seq, const int32_t* row_pos,
                                 const void* rope_cos_bf16, const void* rope_sin_bf16, void* idx_q_out_bf16,
                                 void* idx_k_bf16, void* idx_z_bf16, uint8_t* summaries_e4m3,
                                 step5_stream_t stream) {
    step5_status s = check_geometry(geom);
    if (s != STEP5_OK) return s;
    if (geom->num_kv_groups > 4) return STEP5_ERR_UNSUPPORTED;  // one thread per (group, dim)
    if (N <= 0 || B <= 0 || t_cap <= 0 || r_cap <= 0 || (t_cap % geom->region_tokens)) return STEP5_ERR_INVALID_ARGUMENT;
    if (!(eps >= 0.0f) || eps > 1.0f) return STEP5_ERR_INVALID_ARGUMENT;
    if (!q_pre_bf16 || !k_pre_bf16 || !z_pre_bf16 || !q_norm_w_bf16 || !k_norm_w_bf16 || !k_norm_b_bf16 ||
        !row_seq || !row_pos || !idx_q_out_bf16 || !idx_k_bf16 || !idx_z_bf16 || !summaries_e4m3)
        return STEP5_ERR_INVALID_ARGUMENT;
    if ((rope_cos_bf16 == nullptr) != (rope_sin_bf16 == nullptr)) return STEP5_ERR_INVALID_ARGUMENT;
    if (!aligned16(q_pre_bf16) || !aligned16(idx_q_out_bf16) || !aligned16(idx_k_bf16) || !aligned16(idx_z_bf16))
        return STEP5_ERR_INVALID_ARGUMENT;
    if ((int64_t)B * geom->num_kv_groups * t_cap > INT32_MAX) return STEP5_ERR_INVALID_ARGUMENT;
    uint32_t* st = status_ptr();
    if (!st) return STEP5_ERR_CUDA;
    FrontParams p;
    p.q_pre = static_cast<const uint16_t*>(q_pre_bf16);
    p.k_pre = static_cast<const uint16_t*>(k_pre_bf16);
    p.z_pre = static_cast<const uint16_t*>(z_pre_bf16);
    p.q_w = static_cast<const uint16_t*>(q_norm_w_bf16);
    p.k_w = static_cast<const uint16_t*>(k_norm_w_bf16);
    p.k_b = static_cast<const uint16_t*>(k_norm_b_bf16);
    p.row_seq = row_seq;
    p.row_pos = row_pos;
    p.cos = static_cast<const uint16_t*>(rope_cos_bf16);
    p.sin = static_cast<const uint16_t*>(rope_sin_bf16);
    p.q_out = static_cast<uint16_t*>(idx_q_out_bf16);
    p.idx_k = static_cast<uint16_t*>(idx_k_bf16);
    p.idx_z = static_cast<uint16_t*>(idx_z_bf16);
    p.summ = summaries_e4m3;
    p.status = st;
    p.N = N;
    p.B = B;
    p.G = geom->num_kv_groups;
    p.idx_heads = geom->idx_heads;
    p.t_cap = t_cap;
    p.r_cap = r_cap;
    p.rope_dims = rope_cos_bf16 ? geom->rope_dims : 0;
    p.eps = eps;
    return launch_front(p, (cudaStream_t)stream) == cudaSuccess ? STEP5_OK : STEP5_ERR_CUDA;
}

step5_status step5_decode_step(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap, int32_t r_cap,
                               int32_t max_regions_per_seq, const void* idx_k_bf16, const void* idx_z_bf16,
                               const void* rope_cos_bf16, const void* rope_sin_bf16, const int32_t* region_begin,
                               const int32_t* region_end, uint8_t* summaries_e4m3, const void* idx_q_bf16,
                               const float* w, const int32_t* row_seq, const int32_t* row_pos, const void* q_bf16,
                               const void* k_cache_bf16, const void* v_cache_bf16, int32_t* sel_ids,
                               int32_t* sel_count, void* out_bf16, void* workspace, size_t workspace_bytes,
                               step5_stream_t stream) {
    // every argument is checked before anything is enqueued
    step5_status s = summarize_impl(geom, B, t_cap, r_cap, max_regions_per_seq, idx_k_bf16, idx_z_bf16,
                                    rope_cos_bf16, rope_sin_bf16, region_begin, region_end, summaries_e4m3,
                                    nullptr, stream, false);
    if (s != STEP5_OK) return s;
    s = score_impl(geom, N, B, t_cap, r_cap, idx_q_bf16, w, row_seq, row_pos, rope_cos_bf16, rope_sin_bf16,
                   summaries_e4m3, sel_ids, sel_count, nullptr, nullptr, workspace, workspace_bytes, stream, 0,
                   nullptr, nullptr, false);
    if (s != STEP5_OK) return s;
    s = attn_impl(geom, N, B, t_cap, q_bf16, k_cache_bf16, v_cache_bf16, row_seq, row_pos, sel_ids, sel_count,
                  out_bf16, workspace, workspace_bytes, stream, false);
    if (s != STEP5_OK) return s;
    s = summarize_impl(geom, B, t_cap, r_cap, max_regions_per_seq, idx_k_bf16, idx_z_bf16, rope_cos_bf16,
                       rope_sin_bf16, region_begin, region_end, summaries_e4m3, nullptr, stream, true);
    if (s != STEP5_OK) return s;
    // the summary kernel (when launched) writes only the summaries of regions
    // [region_begin[b], region_end[b]): the scoring kernel reads its other inputs, and
    // the summary tiles clear of those ranges, before waiting for it
    const bool sum_launched = max_regions_per_seq > 0;
    s = score_impl(geom, N, B, t_cap, r_cap, idx_q_bf16, w, row_seq, row_pos, rope_cos_bf16, rope_sin_bf16,
                   summaries_e4m3, sel_ids, sel_count, nullptr, nullptr, workspace, workspace_bytes, stream,
                   sum_launched ? 1 : 0, sum_launched ? region_begin : nullptr,
                   sum_launched ? region_end : nullptr, true);
    if (s != STEP5_OK) return s;
    return attn_impl(geom, N, B, t_cap, q_bf16, k_cache_bf16, v_cache_bf16, row_seq, row_pos, sel_ids, sel_count,
                     out_bf16, workspace, workspace_bytes, stream, true);
}

step5_status step5_rows_layout_for(const step5_geometry* geom, int32_t N, int32_t B, step5_rows_layout* layout) {
    step5_status s = check_geometry(geom);
    if (s != STEP5_OK) return s;
    if (N <= 0 || B <= 0 || layout == nullptr) return STEP5_ERR_INVALID_ARGUMENT;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    size_t at = 0;
    auto take = [&](size_t bytes) {
        const size_t o = at;
        at += up(bytes);
        return o;
    };
    layout->q = take((size_t)N * geom->num_q_heads * geom->head_dim * 2);
    layout->idx_q = take((size_t)N * geom->idx_heads * geom->idx_dim * 2);
    layout->w = take((size_t)N * geom->idx_heads * 4);
    layout->row_seq = take((size_t)N * 4);
    layout->row_pos = take((size_t)N * 4);
    layout->region_begin = take((size_t)B * 4);
    layout->region_end = take((size_t)B * 4);
    layout->total = at;
    return STEP5_OK;
}

step5_status step5_decode_step_host(const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap, int32_t r_cap,
                                    int32_t max_regions_per_seq, const void* idx_k_bf16, const void* idx_z_bf16,
                                    const void* rope_cos_bf16, const void* rope_sin_bf16, uint8_t* summaries_e4m3,
                                    const void* k_cache_bf16, const void* v_cache_bf16, const void* rows_host,
                                    void* rows_dev, void* out_host, void* out_dev, int32_t* sel_ids,
                                    int32_t* sel_count, void* workspace, size_t workspace_bytes,
                                    step5_stream_t stream) {
    step5_rows_layout L;
    step5_status s = step5_rows_layout_for(geom, N, B, &L);
    if (s != STEP5_OK) return s;
    if (!rows_host || !rows_dev || !out_host || !out_dev || !aligned16(rows_dev)) return STEP5_ERR_INVALID_ARGUMENT;
    // Page-locked host buffers that the device can address (unified addressing; on
    // Grace, over NVLink-C2C) are read and written by the step's kernels in place: no
    // copy operations.  Otherwise (or with step5_set_host_copies(1)) the inputs are
    // copied into rows_dev and the output out of out_dev.
    void* rows_map = nullptr;
    void* out_map = nullptr;
    bool mapped = false;
    if (!g_host_copies) {
        mapped = cudaHostGetDevicePointer(&rows_map, const_cast<void*>(rows_host), 0) == cudaSuccess &&
                 cudaHostGetDevicePointer(&out_map, out_host, 0) == cudaSuccess && aligned16(rows_map) &&
                 aligned16(out_map);
        if (!mapped) (void)cudaGetLastError();  // a refused lookup leaves no error behind
    }
    uint8_t* d = static_cast<uint8_t*>(mapped ? rows_map : rows_dev);
    void* out = mapped ? out_map : out_dev;
    const void* q = d + L.q;
    const void* idx_q = d + L.idx_q;
    const float* w = reinterpret_cast<const float*>(d + L.w);
    const int32_t* row_seq = reinterpret_cast<const int32_t*>(d + L.row_seq);
    const int32_t* row_pos = reinterpret_cast<const int32_t*>(d + L.row_pos);
    const int32_t* rb = reinterpret_cast<const int32_t*>(d + L.region_begin);
    const int32_t* re = reinterpret_cast<const int32_t*>(d + L.region_end);
    // every argument is checked before anything is enqueued
    s = summarize_impl(geom, B, t_cap, r_cap, max_regions_per_seq, idx_k_bf16, idx_z_bf16, rope_cos_bf16,
                       rope_sin_bf16, rb, re, summaries_e4m3, nullptr, stream, false);
    if (s != STEP5_OK) return s;
    s = score_impl(geom, N, B, t_cap, r_cap, idx_q, w, row_seq, row_pos, rope_cos_bf16, rope_sin_bf16,
                   summaries_e4m3, sel_ids, sel_count, nullptr, nullptr, workspace, workspace_bytes, stream, 0,
                   nullptr, nullptr, false);
    if (s != STEP5_OK) return s;
    s = attn_impl(geom, N, B, t_cap, q, k_cache_bf16, v_cache_bf16, row_seq, row_pos, sel_ids, sel_count, out,
                  workspace, workspace_bytes, stream, false);
    if (s != STEP5_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    if (!mapped && cudaMemcpyAsync(rows_dev, rows_host, L.total, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return STEP5_ERR_CUDA;
    s = step5_decode_step(geom, N, B, t_cap, r_cap, max_regions_per_seq, idx_k_bf16, idx_z_bf16, rope_cos_bf16,
                          rope_sin_bf16, rb, re, summaries_e4m3, idx_q, w, row_seq, row_pos, q, k_cache_bf16,
                          v_cache_bf16, sel_ids, sel_count, out, workspace, workspace_bytes, stream);
    if (s != STEP5_OK || mapped) return s;
    const size_t out_bytes = (size_t)N * geom->num_q_heads * geom->head_dim * 2;
    return cudaMemcpyAsync(out_host, out_dev, out_bytes, cudaMemcpyDeviceToHost, st) == cudaSuccess ? STEP5_OK
                                                                                                   : STEP5_ERR_CUDA;
}

}  // extern "C"
