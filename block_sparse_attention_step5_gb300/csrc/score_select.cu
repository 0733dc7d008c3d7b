// score_select.cu -- steps (2) and (3): FP8 index scores and top-k by (-score, id).
//
// "Step-5-Preview on one 256 GB Mac" (TensorFold PR #903), CSA-indexer commit: scores
// sum_h relu(e4m3(q_h) . summary) * w_h per KV group; the top 512 by (-score, id),
// ascending.  Provider groups own contiguous blocks of indexer heads (vLLM Step5 DSA
// geometry: "the sparse indexer reduces scores within provider groups").
//
// Scoring runs on the CUDA cores: each region is read as four 16-byte vectors, one per
// thread, every e4m3 pair is widened to fp32 (exact) and multiplied with the thread's
// 16 query dims per head using packed fp32x2 FMAs; a two-step butterfly completes the
// 64-dim dot products.  Selection works on 64-bit keys (desc(score) << 32 | id), which
// are unique, so any exact selection yields the same ordered ids.
//
// Two selection paths with identical results:
//  * fused: one block per (row, group) scores every region into shared memory, then
//    runs an 8-bit radix descent over the keys and a bitonic sort of the k winners.
//  * split: many blocks per (row, group) score a slice each and add a 12-bit histogram
//    of the keys into global memory; a filter pass copies every key in or above the
//    bin holding the k-th key into a candidate list; one block per (row, group) then
//    runs the same radix descent + sort over the candidates.  Used when there are few
//    rows and many regions (decode at 128K-1M tokens).
#include "kernels.cuh"

namespace step5 {

namespace {

// ----------------------------------------------------------------- query fragment

template <int HPG>
struct QFrag {
    float2 q[HPG][8];  // e4m3 query of head h at dims 16*qd + 2i, 16*qd + 2i + 1
    float w[HPG];      // w of every head (HPG == 4: w[0] holds head qd's weight)
};

// e4m3(bf16(NEOX(q))) of the group's HPG heads, as floats, into s_q[h * 64 + d].  Ends
// with a __syncthreads.
template <int HPG>
__device__ void stage_query(const ScoreParams& p, int n, int g, int pos, float* s_q) {
    const int half = p.rope_dims >> 1;
    for (int i = threadIdx.x; i < HPG * 64; i += blockDim.x) {
        const int h = i >> 6, d = i & 63;
        const uint16_t* qrow = p.idx_q + ((int64_t)n * p.idx_heads + (int64_t)g * HPG + h) * 64;
        uint16_t rb = qrow[d];
        if (p.cos != nullptr && d < p.rope_dims) {
            const bool first = d < half;
            const int pd = first ? d + half : d - half;
            const int pi = first ? d : d - half;
            const float c = bf16_to_f32(p.cos[(int64_t)pos * half + pi]);
            const float s = bf16_to_f32(p.sin[(int64_t)pos * half + pi]);
            rb = neox_rotate(bf16_to_f32(rb), bf16_to_f32(qrow[pd]), c, s, first);
        }
        s_q[i] = e4m3x2_to_f32x2(f32_to_e4m3(bf16_to_f32(rb))).x;
    }
    __syncthreads();
}

// The staged query into registers for the 4-lanes-per-region layout: each thread keeps
// the 16 dims it multiplies (qd = lane & 3).
template <int HPG>
__device__ void load_qfrag(const ScoreParams& p, int n, int g, int pos, float* s_q, QFrag<HPG>& f) {
    const int qd = threadIdx.x & 3;
#pragma unroll
    for (int h = 0; h < HPG; ++h) f.w[h] = p.w[(int64_t)n * p.idx_heads + (int64_t)g * HPG + h];
    if constexpr (HPG == 4) f.w[0] = p.w[(int64_t)n * p.idx_heads + (int64_t)g * HPG + qd];
    stage_query<HPG>(p, n, g, pos, s_q);
#pragma unroll
    for (int h = 0; h < HPG; ++h) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            f.q[h][i] = make_float2(s_q[h * 64 + 16 * qd + 2 * i], s_q[h * 64 + 16 * qd + 2 * i + 1]);
    }
}

// ----------------------------------------------------------------- one thread per region
//
// For 4 indexer heads per group: a thread scores whole regions (64 dims, 4 heads), two at
// a time, so no cross-lane reduction is needed.  The query lives in shared memory as
// q4[2 * pair + hp] = (q_{2hp}[2 pair], q_{2hp}[2 pair + 1], q_{2hp+1}[2 pair],
// q_{2hp+1}[2 pair + 1]); every lane reads the same element (broadcast) and one query
// load serves both regions.

// Rearranges s_q [4][64] into q4 [64]; ends with a __syncthreads.
__device__ __forceinline__ void build_q4(const float* s_q, float4* q4) {
    if (threadIdx.x < 64) {
        const int pr = threadIdx.x >> 1, hp = threadIdx.x & 1;
        q4[threadIdx.x] = make_float4(s_q[(2 * hp) * 64 + 2 * pr], s_q[(2 * hp) * 64 + 2 * pr + 1],
                                      s_q[(2 * hp + 1) * 64 + 2 * pr], s_q[(2 * hp + 1) * 64 + 2 * pr + 1]);
    }
    __syncthreads();
}

__device__ __forceinline__ float finish_score4(const float2 (&acc)[4], const float (&w)[4]) {
    float sc = 0.0f;
#pragma unroll
    for (int h = 0; h < 4; ++h) sc = fmaf(fmaxf(__fadd_rn(acc[h].x, acc[h].y), 0.0f), w[h], sc);
    return __fadd_rn(sc, 0.0f);  // -0 -> +0
}

// Scores of two regions whose 64 summary bytes are a[0..3] and b[0..3] (dims 16k..16k+15
// in chunk k).  Each head's dot product is the sum of an even-dim and an odd-dim partial
// sum, accumulated in dim order.
__device__ __forceinline__ void score_rows2(const uint4 (&a)[4], const uint4 (&b)[4], const float4* q4,
                                            const float (&w)[4], float& sa, float& sb) {
    float2 A[4], Bc[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) A[h] = Bc[h] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t wa[4] = {a[k].x, a[k].y, a[k].z, a[k].w};
        const uint32_t wb[4] = {b[k].x, b[k].y, b[k].z, b[k].w};
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            const int p0 = 8 * k + 2 * qq;
#pragma unroll
            for (int hw = 0; hw < 2; ++hw) {  // low / high 16 bits: pair p0 / p0 + 1
                const float2 xa = e4m3x2_to_f32x2((uint16_t)(hw ? wa[qq] >> 16 : wa[qq] & 0xffffu));
                const float2 xb = e4m3x2_to_f32x2((uint16_t)(hw ? wb[qq] >> 16 : wb[qq] & 0xffffu));
                const float4 q01 = q4[2 * (p0 + hw)], q23 = q4[2 * (p0 + hw) + 1];
                const float2 q0 = make_float2(q01.x, q01.y), q1 = make_float2(q01.z, q01.w);
                const float2 q2 = make_float2(q23.x, q23.y), q3 = make_float2(q23.z, q23.w);
                A[0] = __ffma2_rn(q0, xa, A[0]);
                A[1] = __ffma2_rn(q1, xa, A[1]);
                A[2] = __ffma2_rn(q2, xa, A[2]);
                A[3] = __ffma2_rn(q3, xa, A[3]);
                Bc[0] = __ffma2_rn(q0, xb, Bc[0]);
                Bc[1] = __ffma2_rn(q1, xb, Bc[1]);
                Bc[2] = __ffma2_rn(q2, xb, Bc[2]);
                Bc[3] = __ffma2_rn(q3, xb, Bc[3]);
            }
        }
    }
    sa = finish_score4(A, w);
    sb = finish_score4(Bc, w);
}

// Score of the region whose 16 dims [16*qd, 16*qd + 16) this thread holds in v.  All
// four threads of the region (lanes 4k..4k+3) must call it together; all get the same
// bits back.
template <int HPG>
__device__ __forceinline__ float score_from_vec(const QFrag<HPG>& f, uint4 v) {
    float2 acc[HPG];
#pragma unroll
    for (int h = 0; h < HPG; ++h) acc[h] = make_float2(0.0f, 0.0f);
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 s0 = e4m3x2_to_f32x2((uint16_t)(w4[q] & 0xffffu));
        const float2 s1 = e4m3x2_to_f32x2((uint16_t)(w4[q] >> 16));
#pragma unroll
        for (int h = 0; h < HPG; ++h) {
            acc[h] = __ffma2_rn(f.q[h][2 * q], s0, acc[h]);
            acc[h] = __ffma2_rn(f.q[h][2 * q + 1], s1, acc[h]);
        }
    }
    if constexpr (HPG == 4) {
        // transpose-reduce over the region's 4 lanes: afterwards lane qd holds head qd's
        // full dot product; then relu * w and a sum over the 4 lanes
        const int qd = threadIdx.x & 3;
        float d0 = __fadd_rn(acc[0].x, acc[0].y), d1 = __fadd_rn(acc[1].x, acc[1].y);
        float d2 = __fadd_rn(acc[2].x, acc[2].y), d3 = __fadd_rn(acc[3].x, acc[3].y);
        const bool lo2 = qd < 2;
        const float send0 = lo2 ? d2 : d0, send1 = lo2 ? d3 : d1;
        float k0 = lo2 ? d0 : d2, k1 = lo2 ? d1 : d3;
        k0 = __fadd_rn(k0, __shfl_xor_sync(0xffffffffu, send0, 2));
        k1 = __fadd_rn(k1, __shfl_xor_sync(0xffffffffu, send1, 2));
        const bool odd = qd & 1;
        const float send = odd ? k0 : k1;
        float dot = __fadd_rn(odd ? k1 : k0, __shfl_xor_sync(0xffffffffu, send, 1));
        float v = __fmul_rn(fmaxf(dot, 0.0f), f.w[0]);
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
        return __fadd_rn(v, 0.0f);  // -0 -> +0
    } else {
        float sc = 0.0f;
#pragma unroll
        for (int h = 0; h < HPG; ++h) {
            float dot = __fadd_rn(acc[h].x, acc[h].y);
            dot = __fadd_rn(dot, __shfl_xor_sync(0xffffffffu, dot, 1));
            dot = __fadd_rn(dot, __shfl_xor_sync(0xffffffffu, dot, 2));
            sc = fmaf(fmaxf(dot, 0.0f), f.w[h], sc);
        }
        return __fadd_rn(sc, 0.0f);  // -0 -> +0
    }
}

// ----------------------------------------------------------------- block top-k

constexpr int kRadixBits = 11;
constexpr int kRadixBins = 1 << kRadixBits;

struct TopkSmem {
    uint32_t hist[kRadixBins];
    uint32_t wsum[32];
    uint32_t count;
    uint32_t v, before, inbin;
};

// Bitonic sort, ascending, of P2 (a power of two >= 32) keys in shared memory.  Stages
// whose partner distance is below 32 run in registers with warp shuffles; the others
// exchange through shared memory.
template <int NT>
__device__ void block_bitonic_sort(uint64_t* s, int P2) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NW = NT / 32;
    for (int k = 2; k <= P2; k <<= 1) {
        int j = k >> 1;
        for (; j >= 32; j >>= 1) {
            for (int i = tid; i < P2; i += NT) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const uint64_t a = s[i], b = s[ixj];
                    const bool asc = (i & k) == 0;
                    if ((a > b) == asc) {
                        s[i] = b;
                        s[ixj] = a;
                    }
                }
            }
            __syncthreads();
        }
        // remaining distances j < 32: within aligned chunks of 32 keys, one per lane
        for (int c = warp; c < P2 / 32; c += NW) {
            const int i = c * 32 + lane;
            uint64_t v = s[i];
            for (int jj = j; jj > 0; jj >>= 1) {
                const uint64_t o = __shfl_xor_sync(0xffffffffu, v, jj);
                const bool asc = (i & k) == 0;
                const bool lower = (i & jj) == 0;
                v = (lower == asc) ? (v < o ? v : o) : (v > o ? v : o);
            }
            s[i] = v;
        }
        __syncthreads();
    }
}

// Gathers the K smallest of cnt unique 64-bit keys (all of them if cnt <= K) into
// s_sel[0..min(cnt, K)) in no particular order, pads s_sel up to P2 (a power of two >=
// max(K, 32)) with ~0, returns min(cnt, K).  A radix descent over 11-bit digits (most
// significant first) finds the K-th key; every key at or below it is gathered.  get(i)
// returns key i.  Must be called by all NT threads of the block.
template <int NT, class Get>
__device__ int block_select_set(Get get, int cnt, int K, int P2, uint64_t* s_sel, TopkSmem& ts) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint64_t bound = ~0ull;
    if (cnt > K) {
        uint64_t prefix = 0;
        int need = K;
        int hi = 64;  // key bits at and above `hi` are fixed by `prefix`
        while (hi > 0) {
            const int width = hi >= kRadixBits ? kRadixBits : hi;
            const int shift = hi - width;
            const uint32_t dmask = (1u << width) - 1u;
            for (int i = tid; i < kRadixBins; i += NT) ts.hist[i] = 0;
            __syncthreads();
            const uint64_t mask = (hi == 64) ? 0ull : (~0ull << hi);
            for (int i = tid; i < cnt; i += NT) {
                const uint64_t k = get(i);
                if ((k & mask) == prefix) atomicAdd(&ts.hist[(uint32_t)(k >> shift) & dmask], 1u);
            }
            __syncthreads();
            {
                // block-wide scan: each thread owns PER consecutive bins
                constexpr int PER = kRadixBins / NT;
                constexpr int NW = NT / 32;
                uint32_t loc[PER];
                uint32_t sum = 0;
#pragma unroll
                for (int q = 0; q < PER; ++q) {
                    loc[q] = ts.hist[tid * PER + q];
                    sum += loc[q];
                }
                uint32_t incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                if (lane == 31) ts.wsum[warp] = incl;
                __syncthreads();
                if (warp == 0) {
                    uint32_t w = lane < NW ? ts.wsum[lane] : 0u;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t t = __shfl_up_sync(0xffffffffu, w, o);
                        if (lane >= o) w += t;
                    }
                    if (lane < NW) ts.wsum[lane] = w;  // inclusive warp prefix
                }
                __syncthreads();
                incl += warp ? ts.wsum[warp - 1] : 0u;
                const uint32_t excl = incl - sum;
                if (excl < (uint32_t)need && (uint32_t)need <= incl) {
                    uint32_t c = excl;
#pragma unroll
                    for (int q = 0; q < PER; ++q) {
                        if (c + loc[q] >= (uint32_t)need) {
                            ts.v = tid * PER + q;
                            ts.before = c;
                            ts.inbin = loc[q];
                            break;
                        }
                        c += loc[q];
                    }
                }
            }
            __syncthreads();
            const uint32_t v = ts.v, before = ts.before, inbin = ts.inbin;
            __syncthreads();
            prefix |= (uint64_t)v << shift;
            need -= (int)before;
            if ((int)inbin == need) {
                bound = prefix | ((shift == 0) ? 0ull : ((1ull << shift) - 1ull));
                break;
            }
            hi = shift;
        }
    }
    if (tid == 0) ts.count = 0;
    for (int i = tid; i < P2; i += NT) s_sel[i] = ~0ull;
    __syncthreads();
    for (int base = 0; base < cnt; base += NT) {
        const int i = base + tid;
        bool act = false;
        uint64_t k = 0;
        if (i < cnt) {
            k = get(i);
            act = k <= bound;
        }
        const uint32_t am = __ballot_sync(0xffffffffu, act);
        uint32_t slot = 0;
        if (lane == 0 && am) slot = atomicAdd(&ts.count, (uint32_t)__popc(am));
        slot = __shfl_sync(0xffffffffu, slot, 0);
        if (act) {
            const uint32_t idx = slot + __popc(am & ((1u << lane) - 1u));
            if (idx < (uint32_t)P2) s_sel[idx] = k;
        }
    }
    __syncthreads();
    return cnt < K ? cnt : K;
}

// block_select_set followed by an ascending sort of the gathered keys.
template <int NT, class Get>
__device__ int block_topk(Get get, int cnt, int K, int P2, uint64_t* s_sel, TopkSmem& ts) {
    const int take = block_select_set<NT>(get, cnt, K, P2, s_sel, ts);
    block_bitonic_sort<NT>(s_sel, P2);
    return take;
}

// Key getters for block_topk.
struct SmemKeys {  // keys indexed by region id: desc(score) << 32 | id
    const uint32_t* key;
    __device__ __forceinline__ uint64_t operator()(int i) const {
        return ((uint64_t)key[i] << 32) | (uint32_t)i;
    }
};
struct CandKeys {  // explicit candidate list
    const uint64_t* cand;
    __device__ __forceinline__ uint64_t operator()(int i) const { return cand[i]; }
};
struct ScoreKeys {  // every score of the row, from global memory
    const float* scores;
    __device__ __forceinline__ uint64_t operator()(int i) const {
        return ((uint64_t)desc_key(scores[i]) << 32) | (uint32_t)i;
    }
};

template <int NT>
__device__ void write_selection(const ScoreParams& p, int n, int g, int take, const uint64_t* s_sel) {
    const int64_t ng = (int64_t)n * p.G + g;
    int32_t* ids = p.sel_ids + ng * p.top_k;
    float* ss = p.sel_scores ? p.sel_scores + ng * p.top_k : nullptr;
    for (int i = threadIdx.x; i < p.top_k; i += NT) {
        if (i < take) {
            const uint64_t key = s_sel[i];
            ids[i] = (int32_t)(uint32_t)(key & 0xffffffffu);
            if (ss) ss[i] = score_of_desc_key((uint32_t)(key >> 32));
        } else {
            ids[i] = -1;
            if (ss) ss[i] = -INFINITY;
        }
    }
    if (threadIdx.x == 0) p.sel_count[ng] = take;
}

// Validated (sequence, R) of row n, or R = -1 when the row is out of range.
__device__ __forceinline__ int row_regions(const ScoreParams& p, int n, int& b, int& pos) {
    b = p.row_seq[n];
    pos = p.row_pos[n];
    if (b < 0 || b >= p.B || pos < 0 || pos >= p.t_cap || pos / 8 > p.r_cap) return -1;
    return pos / 8;
}

// ----------------------------------------------------------------- fused path

constexpr int kFusedThreads = 256;

template <int HPG>
__global__ void __launch_bounds__(kFusedThreads) score_fused_kernel(ScoreParams p, int P2, int key_cap) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint64_t* s_sel = reinterpret_cast<uint64_t*>(smem);                 // P2
    uint32_t* s_key = reinterpret_cast<uint32_t*>(s_sel + P2);           // key_cap
    float* s_q = reinterpret_cast<float*>(s_key + key_cap);              // HPG * 64
    __shared__ TopkSmem ts;

    const int g = blockIdx.x, n = blockIdx.y;
    pdl_wait();
    pdl_launch_dependents();
    int b, pos;
    int R = row_regions(p, n, b, pos);
    if (R < 0 || R > key_cap) {
        if (threadIdx.x == 0) raise_status(p.status, kDevRange);
        R = 0;
        b = 0;
        pos = 0;
    }
    const uint4* base = reinterpret_cast<const uint4*>(p.summ + ((int64_t)b * p.G + g) * p.r_cap * 64);
    float* exp_scores = p.scores ? p.scores + ((int64_t)n * p.G + g) * p.r_cap : nullptr;
    if constexpr (HPG == 4) {
        __shared__ float4 s_q4[64];
        float w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) w[h] = p.w[(int64_t)n * p.idx_heads + (int64_t)g * 4 + h];
        stage_query<4>(p, n, g, pos, s_q);
        build_q4(s_q, s_q4);
        for (int r0 = 0; r0 < R; r0 += 2 * kFusedThreads) {
            const int ra = r0 + threadIdx.x, rb = ra + kFusedThreads;
            uint4 va[4], vb[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                va[k] = ra < R ? __ldg(base + (int64_t)ra * 4 + k) : make_uint4(0, 0, 0, 0);
                vb[k] = rb < R ? __ldg(base + (int64_t)rb * 4 + k) : make_uint4(0, 0, 0, 0);
            }
            float sa, sb;
            score_rows2(va, vb, s_q4, w, sa, sb);
            if (ra < R) {
                s_key[ra] = desc_key(sa);
                if (exp_scores) exp_scores[ra] = sa;
            }
            if (rb < R) {
                s_key[rb] = desc_key(sb);
                if (exp_scores) exp_scores[rb] = sb;
            }
        }
    } else {
        QFrag<HPG> f;
        load_qfrag<HPG>(p, n, g, pos, s_q, f);
        const int qd = threadIdx.x & 3;
        const int slot = threadIdx.x >> 2;  // 64 regions per pass
        constexpr int U = 4;
        for (int r0 = 0; r0 < R; r0 += 64 * U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int r = r0 + u * 64 + slot;
                v[u] = (r < R) ? __ldg(base + (int64_t)r * 4 + qd) : make_uint4(0, 0, 0, 0);
            }
            float sc[U];
#pragma unroll
            for (int u = 0; u < U; ++u) sc[u] = score_from_vec<HPG>(f, v[u]);
            // lane qd keeps the bookkeeping of region u = qd
            const float mysc = qd == 0 ? sc[0] : qd == 1 ? sc[1] : qd == 2 ? sc[2] : sc[3];
            const int r = r0 + qd * 64 + slot;
            if (r < R) {
                s_key[r] = desc_key(mysc);
                if (exp_scores) exp_scores[r] = mysc;
            }
        }
    }
    __syncthreads();
    const int take = block_topk<kFusedThreads>(SmemKeys{s_key}, R, p.top_k, P2, s_sel, ts);
    write_selection<kFusedThreads>(p, n, g, take, s_sel);
}

// ----------------------------------------------------------------- split path

constexpr int kSplitThreads = 256;

// ----------------------------------------------------------------- split path scoring
//
// Persistent blocks (two per SM) walk a contiguous run of tiles; a tile is kTileRegions
// consecutive regions of one (row, group), contiguous in the summary store, fetched with
// one bulk copy into a 2-stage shared-memory ring while the previous tile is scored.
// Each run of tiles of one (row, group) adds its shared-memory histogram to the global
// one and takes a ticket; the block holding the last ticket publishes the bin of the
// k-th key for the filter pass.

constexpr int kTileRegions = 512;                 // 32 KB of summaries
constexpr int kTileBytes = kTileRegions * 64;
constexpr int kTileU = kTileRegions / 64;         // regions per thread per tile (8)
constexpr int kScoreStages = 2;
constexpr size_t kScoreSmem = kScoreStages * kTileBytes + 1024;

struct Tile {
    int valid, ng, n, g, b, pos, R, c0, c1;
};

// The next tile of this block's range [x, hi) of the flattened (row, group, region)
// space (r_cap regions per (row, group)): at most kTileRegions consecutive candidate
// regions of one (row, group).  Regions past a row's R, and rows out of range, are
// skipped.  Advances x past the tile.
__device__ __forceinline__ Tile next_tile(const ScoreParams& p, int64_t& x, int64_t hi) {
    Tile t;
    t.valid = 0;
    while (x < hi) {
        const int ng = (int)(x / p.r_cap);
        const int r = (int)(x - (int64_t)ng * p.r_cap);
        const int n = ng / p.G;
        int b, pos;
        const int R = row_regions(p, n, b, pos);
        if (R < 0) {
            if (threadIdx.x == 0) raise_status(p.status, kDevRange);
            x = (int64_t)(ng + 1) * p.r_cap;
            continue;
        }
        if (r >= R) {
            x = (int64_t)(ng + 1) * p.r_cap;
            continue;
        }
        int c1 = min(R, r + kTileRegions);
        const int64_t lim = hi - (int64_t)ng * p.r_cap;
        if ((int64_t)c1 > lim) c1 = (int)lim;
        t.valid = 1;
        t.ng = ng;
        t.n = n;
        t.g = ng - n * p.G;
        t.b = b;
        t.pos = pos;
        t.R = R;
        t.c0 = r;
        t.c1 = c1;
        x = (int64_t)ng * p.r_cap + c1;
        return t;
    }
    return t;
}

// Scores one staged tile: thread (slot, qd) covers regions u * 64 + slot, u < kTileU;
// lane qd of each region quad keeps the score and histogram update of every fourth
// region.  FULL: the tile holds kTileRegions regions (no bounds checks).
template <int HPG, bool FULL>
__device__ __forceinline__ void score_tile(const QFrag<HPG>& f, const uint4* tile, int nreg, float* scores,
                                           uint32_t* s_hist, int qd, int slot) {
#pragma unroll
    for (int u4 = 0; u4 < kTileU; u4 += 4) {
        float sc[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int lr = (u4 + u) * 64 + slot;
            const uint4 v = (FULL || lr < nreg) ? tile[lr * 4 + qd] : make_uint4(0, 0, 0, 0);
            sc[u] = score_from_vec<HPG>(f, v);
        }
        const float mysc = qd == 0 ? sc[0] : qd == 1 ? sc[1] : qd == 2 ? sc[2] : sc[3];
        const int lr = (u4 + qd) * 64 + slot;
        if (FULL || lr < nreg) {
            scores[lr] = mysc;
            atomicAdd(&s_hist[desc_key(mysc) >> (32 - kHistBits)], 1u);
        }
    }
}

// One thread per region (HPG == 4): thread t scores rows t and t + 256 of a tile that
// arrived as two 256-row boxes through the summaries' tensor map with 64-byte swizzle
// (16-byte chunk k of row r sits at chunk k ^ ((r >> 1) & 3)), so the 8 rows a quarter
// warp reads at once fall in 8 different bank groups.
__device__ __forceinline__ void score_tile_rows(const uint8_t* tile, int nreg, const float4* q4,
                                                const float (&w)[4], float* scores, uint32_t* s_hist) {
    const int t = threadIdx.x;  // 0..255
    const int sw = (t >> 1) & 3;
    const uint4* ra = reinterpret_cast<const uint4*>(tile + t * 64);
    const uint4* rb = reinterpret_cast<const uint4*>(tile + 16384 + t * 64);
    uint4 a[4], b[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        a[k] = ra[k ^ sw];
        b[k] = rb[k ^ sw];
    }
    float sa, sb;
    score_rows2(a, b, q4, w, sa, sb);
    if (t < nreg) {
        scores[t] = sa;
        atomicAdd(&s_hist[desc_key(sa) >> (32 - kHistBits)], 1u);
    }
    if (t + 256 < nreg) {
        scores[t + 256] = sb;
        atomicAdd(&s_hist[desc_key(sb) >> (32 - kHistBits)], 1u);
    }
}

template <int HPG>
__global__ void __launch_bounds__(kSplitThreads, 2) score_hist_kernel(const __grid_constant__ CUtensorMap smap,
                                                                      ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint32_t s_hist[kHistBins];
    __shared__ float s_q[HPG * 64];
    __shared__ __align__(8) uint64_t s_bar[kScoreStages];
    const int tid = threadIdx.x;
    const int qd = tid & 3, slot = tid >> 2;

    if (tid == 0) {
        for (int st = 0; st < kScoreStages; ++st) mbar_init(&s_bar[st], 1);
        fence_mbar_init();
    }
    STEP5_STAMP(1, 0);
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();
    STEP5_STAMP(1, 1);
    // this block's even share of the flattened (row, group, region) space
    const int64_t total = (int64_t)p.N * p.G * p.r_cap;
    int64_t xpos = total * blockIdx.x / gridDim.x;
    const int64_t xend = total * (blockIdx.x + 1) / gridDim.x;
    auto next_valid = [&]() -> Tile { return next_tile(p, xpos, xend); };
    auto issue = [&](const Tile& x, int st) {
        if (tid == 0) {
            if constexpr (HPG == 4) {
                // two full boxes (rows past the tensor end arrive as zeros)
                const int y = (int)(((int64_t)x.b * p.G + x.g) * p.r_cap + x.c0);
                mbar_arrive_expect_tx(&s_bar[st], (uint32_t)kTileBytes);
                tma_load_2d(ring + st * kTileBytes, &smap, &s_bar[st], 0, y);
                tma_load_2d(ring + st * kTileBytes + kTileBytes / 2, &smap, &s_bar[st], 0, y + kTileRegions / 2);
            } else {
                const uint32_t bytes = (uint32_t)(x.c1 - x.c0) * 64u;
                mbar_arrive_expect_tx(&s_bar[st], bytes);
                bulk_load(ring + st * kTileBytes, p.summ + (((int64_t)x.b * p.G + x.g) * p.r_cap + x.c0) * 64,
                          bytes, &s_bar[st]);
            }
        }
    };
    // two tiles in flight: `cur` in stage st, `nxt` in stage st ^ 1
    Tile cur = next_valid();
    if (cur.valid) issue(cur, 0);
    Tile nxt = next_valid();
    if (nxt.valid) issue(nxt, 1);
    STEP5_STAMP(1, 2);

    int seg_ng = -1;
    int ntile = 0;
    QFrag<HPG> f;
    __shared__ float4 s_q4[64];
    float w4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    auto finish = [&](int ng) {
        __syncthreads();
        uint32_t* gh = p.hist + (int64_t)ng * kHistBins;
        uint32_t coarse = 0;
        // each thread flushes kHistBins / 256 = 16 consecutive fine bins; 4 threads make
        // one coarse bin of 64
        for (int i = 0; i < kHistBins / kSplitThreads; ++i) {
            const int bin = tid * (kHistBins / kSplitThreads) + i;
            const uint32_t c = s_hist[bin];
            coarse += c;
            if (c) atomicAdd(gh + bin, c);
        }
        coarse += __shfl_xor_sync(0xffffffffu, coarse, 1);
        coarse += __shfl_xor_sync(0xffffffffu, coarse, 2);
        if ((tid & 3) == 0 && coarse) atomicAdd(p.coarse + (int64_t)ng * kCoarseBins + (tid >> 2), coarse);
    };

    uint32_t ph0 = 0, ph1 = 0;
    int st = 0;
    bool timed_out = false;
    while (cur.valid) {
        if (cur.ng != seg_ng) {
            if (seg_ng >= 0) finish(seg_ng);
            seg_ng = cur.ng;
            for (int i = tid; i < kHistBins; i += kSplitThreads) s_hist[i] = 0;
            if constexpr (HPG == 4) {
#pragma unroll
                for (int h = 0; h < 4; ++h) w4[h] = p.w[(int64_t)cur.n * p.idx_heads + (int64_t)cur.g * 4 + h];
                stage_query<4>(p, cur.n, cur.g, cur.pos, s_q);
                build_q4(s_q, s_q4);
            } else {
                load_qfrag<HPG>(p, cur.n, cur.g, cur.pos, s_q, f);  // has a __syncthreads
            }
        }
        if (ntile < 4) STEP5_STAMP(1, 3 + 2 * ntile);
        if (!mbar_wait(&s_bar[st], st ? ph1 : ph0)) {
            timed_out = true;
            break;
        }
        if (ntile < 4) STEP5_STAMP(1, 4 + 2 * ntile);
        ++ntile;
        if (st) ph1 ^= 1u; else ph0 ^= 1u;
        float* scores = p.scores + (int64_t)cur.ng * p.r_cap + cur.c0;
        const int nreg = cur.c1 - cur.c0;
        if constexpr (HPG == 4) {
            score_tile_rows(ring + st * kTileBytes, nreg, s_q4, w4, scores, s_hist);
        } else {
            const uint4* tile = reinterpret_cast<const uint4*>(ring + st * kTileBytes);
            if (nreg == kTileRegions)
                score_tile<HPG, true>(f, tile, nreg, scores, s_hist, qd, slot);
            else
                score_tile<HPG, false>(f, tile, nreg, scores, s_hist, qd, slot);
        }
        __syncthreads();  // every thread is done with this stage before it is refilled
        cur = nxt;
        nxt = next_valid();
        if (nxt.valid) {
            if (tid == 0) fence_proxy_async();
            issue(nxt, st);
        }
        st ^= 1;
    }
    if (timed_out) {
        if (tid == 0) raise_status(p.status, kDevTimeout);
        // give copies still in flight a bounded chance to land before the block exits
        if (cur.valid) mbar_wait(&s_bar[st], st ? ph1 : ph0);
        if (nxt.valid) mbar_wait(&s_bar[st ^ 1], st ? ph0 : ph1);
    }
    STEP5_STAMP(1, 11);
    if (seg_ng >= 0 && !timed_out) finish(seg_ng);
    STEP5_STAMP(1, 12);
}

// Bin holding the K-th smallest key of (row, group) from the coarse (64-bin) and fine
// (4096-bin) histograms; all bins when the row has at most K regions.  Two small reads
// (256 bytes each) instead of the whole fine histogram.
__device__ int threshold_bin2(const uint32_t* coarse, const uint32_t* fine, int R, int K, int* s_out) {
    if (R <= K) return kHistBins - 1;
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid < 32) {
        const uint32_t c0 = __ldcg(coarse + 2 * lane), c1 = __ldcg(coarse + 2 * lane + 1);
        uint32_t incl = c0 + c1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const uint32_t excl = incl - c0 - c1;
        // the coarse bin holding the K-th key
        int cb = -1;
        uint32_t before = 0;
        if (excl < (uint32_t)K && (uint32_t)K <= excl + c0) {
            cb = 2 * lane;
            before = excl;
        } else if (excl + c0 < (uint32_t)K && (uint32_t)K <= incl) {
            cb = 2 * lane + 1;
            before = excl + c0;
        }
        const uint32_t found = __ballot_sync(0xffffffffu, cb >= 0);
        const int src = found ? __ffs(found) - 1 : 0;
        cb = __shfl_sync(0xffffffffu, cb, src);
        before = __shfl_sync(0xffffffffu, before, src);
        if (!found) cb = kCoarseBins - 1, before = 0;
        // the fine bins of that coarse bin
        const uint32_t f0 = __ldcg(fine + cb * 64 + 2 * lane), f1 = __ldcg(fine + cb * 64 + 2 * lane + 1);
        uint32_t fin = f0 + f1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, fin, o);
            if (lane >= o) fin += t;
        }
        const uint32_t fex = before + fin - f0 - f1;
        int fb = -1;
        if (fex < (uint32_t)K && (uint32_t)K <= fex + f0)
            fb = cb * 64 + 2 * lane;
        else if (fex + f0 < (uint32_t)K && (uint32_t)K <= before + fin)
            fb = cb * 64 + 2 * lane + 1;
        const uint32_t ff = __ballot_sync(0xffffffffu, fb >= 0);
        fb = __shfl_sync(0xffffffffu, fb, ff ? __ffs(ff) - 1 : 0);
        if (lane == 0) *s_out = ff ? fb : kHistBins - 1;
    }
    __syncthreads();
    return *s_out;
}

constexpr int kFilterPerThread = 4;  // scores per thread (regions_per_cta = 1024)

__global__ void __launch_bounds__(kSplitThreads) filter_kernel(ScoreParams p) {
    __shared__ uint32_t s_wcnt[kSplitThreads / 32];
    __shared__ uint32_t s_base;
    __shared__ int s_bin;
    const int g = blockIdx.y, n = blockIdx.z;
    STEP5_STAMP(2, 0);
    pdl_wait();
    pdl_launch_dependents();
    STEP5_STAMP(2, 1);
    int b, pos;
    const int R = row_regions(p, n, b, pos);
    if (R < 0) return;
    const int c0 = blockIdx.x * p.regions_per_cta;
    const int c1 = min(R, c0 + p.regions_per_cta);
    if (c0 >= c1) return;
    const int64_t ng = (int64_t)n * p.G + g;
    const float* scores = p.scores + ng * p.r_cap;
    // every score of the block is requested at once
    float sc[kFilterPerThread];
#pragma unroll
    for (int u = 0; u < kFilterPerThread; ++u) {
        const int r = c0 + u * kSplitThreads + threadIdx.x;
        sc[u] = r < c1 ? __ldcg(scores + r) : 0.0f;
    }
    const int b1 = threshold_bin2(p.coarse + ng * kCoarseBins, p.hist + ng * kHistBins, R, p.top_k, &s_bin);
    STEP5_STAMP(2, 2);
    uint32_t mine = 0, keys[kFilterPerThread];
#pragma unroll
    for (int u = 0; u < kFilterPerThread; ++u) {
        const int r = c0 + u * kSplitThreads + threadIdx.x;
        keys[u] = desc_key(sc[u]);
        if (r < c1 && (int)(keys[u] >> (32 - kHistBits)) <= b1) ++mine;
    }
    // one atomic per block: block-wide exclusive scan of the per-thread counts
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_wcnt[warp] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t tot = 0;
        for (int w = 0; w < kSplitThreads / 32; ++w) {
            const uint32_t c = s_wcnt[w];
            s_wcnt[w] = tot;
            tot += c;
        }
        s_base = tot ? atomicAdd(p.cand_count + ng, tot) : 0u;
    }
    __syncthreads();
    STEP5_STAMP(2, 3);
    uint32_t slot = s_base + s_wcnt[warp] + incl - mine;
    uint64_t* cand = p.cand + ng * kCandCap;
#pragma unroll
    for (int u = 0; u < kFilterPerThread; ++u) {
        const int r = c0 + u * kSplitThreads + threadIdx.x;
        if (r < c1 && (int)(keys[u] >> (32 - kHistBits)) <= b1) {
            if (slot < (uint32_t)kCandCap) cand[slot] = ((uint64_t)keys[u] << 32) | (uint32_t)r;
            ++slot;
        }
    }
}

constexpr int kFinalThreads = 512;
constexpr int kFinalSlices = 8;  // blocks per (row, group) in the final select

// Final select of the split path: kFinalSlices blocks per (row, group) each gather the
// same k winners from the candidate list (radix descent in shared memory), then each
// places only the winners whose id falls in its slice (id mod kFinalSlices), at the rank
// it counts among all winners.  The last slice to finish reading the candidates leaves
// the histogram, candidate counter and ticket of its (row, group) zero for the next call.
__global__ void __launch_bounds__(kFinalThreads) final_select_kernel(ScoreParams p, int P2, int /*unused*/) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint64_t* s_sel = reinterpret_cast<uint64_t*>(smem);
    uint64_t* s_cand = s_sel + P2;  // kCandCap
    __shared__ TopkSmem ts;
    __shared__ int s_last;
    const int slice = blockIdx.x, g = blockIdx.y, n = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    STEP5_STAMP(3, 0);
    pdl_wait();
    pdl_launch_dependents();
    STEP5_STAMP(3, 1);
    int b, pos;
    int R = row_regions(p, n, b, pos);
    if (R < 0) R = 0;
    const int64_t ng = (int64_t)n * p.G + g;
    // the whole candidate buffer is requested together with its count
    const uint64_t* cand = p.cand + ng * kCandCap;
    uint64_t cv[kCandCap / kFinalThreads];
#pragma unroll
    for (int k = 0; k < kCandCap / kFinalThreads; ++k) cv[k] = __ldcg(cand + k * kFinalThreads + tid);
    const int c = (int)__ldcg(p.cand_count + ng);
    const bool from_cand = c <= kCandCap;
#pragma unroll
    for (int k = 0; k < kCandCap / kFinalThreads; ++k)
        if (k * kFinalThreads + tid < c) s_cand[k * kFinalThreads + tid] = cv[k];
    __syncthreads();
    if (tid == 0) {
        const uint32_t t = atomicAdd(p.ticket + ng, 1u);
        s_last = (t == (uint32_t)(kFinalSlices - 1));
    }
    __syncthreads();
    if (s_last) {
        uint32_t* gh = p.hist + ng * kHistBins;
        for (int i = tid; i < kHistBins; i += kFinalThreads) gh[i] = 0;
        if (tid < kCoarseBins) p.coarse[ng * kCoarseBins + tid] = 0;
        if (tid == 0) {
            p.cand_count[ng] = 0;
            p.ticket[ng] = 0;
        }
    }
    STEP5_STAMP(3, 2);
    const int take = from_cand
                         ? block_select_set<kFinalThreads>(CandKeys{s_cand}, c, p.top_k, P2, s_sel, ts)
                         : block_select_set<kFinalThreads>(ScoreKeys{p.scores + ng * p.r_cap}, R, p.top_k, P2,
                                                           s_sel, ts);
    STEP5_STAMP(3, 3);
    // rank by counting: one warp per winner of this slice, lanes split the comparisons
    int32_t* ids = p.sel_ids + ng * p.top_k;
    float* ss = p.sel_scores ? p.sel_scores + ng * p.top_k : nullptr;
    for (int i = warp; i < take; i += kFinalThreads / 32) {
        const uint64_t key = s_sel[i];
        if ((int)((uint32_t)key % kFinalSlices) != slice) continue;
        uint32_t cnt_less = 0;
        for (int j = lane; j < take; j += 32) cnt_less += s_sel[j] < key ? 1u : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cnt_less += __shfl_xor_sync(0xffffffffu, cnt_less, o);
        if (lane == 0) {
            ids[cnt_less] = (int32_t)(uint32_t)(key & 0xffffffffu);
            if (ss) ss[cnt_less] = score_of_desc_key((uint32_t)(key >> 32));
        }
    }
    STEP5_STAMP(3, 4);
    if (slice == 0) {
        for (int i = take + tid; i < p.top_k; i += kFinalThreads) {
            ids[i] = -1;
            if (ss) ss[i] = -INFINITY;
        }
        if (tid == 0) p.sel_count[ng] = take;
    }
}

int pow2_at_least(int x) {
    int p2 = 32;
    while (p2 < x) p2 <<= 1;
    return p2;
}

template <class K>
cudaError_t launch_ex(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                      const ScoreParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <class K>
cudaError_t launch_ex2(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                       const ScoreParams& p, int a, int b) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, p, a, b);
}

template <int HPG>
cudaError_t fused_for(const ScoreParams& p, cudaStream_t stream, bool pdl) {
    const int P2 = pow2_at_least(p.top_k);
    const int key_cap = (p.r_cap < kFusedMaxRegions ? p.r_cap : kFusedMaxRegions);
    const size_t smem = (size_t)P2 * 8 + (size_t)((key_cap + 3) & ~3) * 4 + HPG * 64 * 4;
    auto kern = score_fused_kernel<HPG>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_ex2(kern, dim3(p.G, p.N), dim3(kFusedThreads), smem, stream, pdl, p, P2,
                      (key_cap + 3) & ~3);
}

template <class K>
cudaError_t launch_map(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                       const CUtensorMap& map, const ScoreParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, map, p);
}

template <int HPG>
cudaError_t split_for(const ScoreParams& p_in, const CUtensorMap& smap, cudaStream_t stream, bool pdl) {
    ScoreParams p = p_in;
    // two persistent blocks per SM, each an even share of the regions
    const int64_t tiles = ((int64_t)p.N * p.G * p.r_cap + kTileRegions - 1) / kTileRegions;
    int64_t grid = 2 * (int64_t)p.num_sms;
    if (grid > tiles) grid = tiles;
    static bool attr = false;
    if (!attr) {
        cudaError_t e0 = cudaFuncSetAttribute(score_hist_kernel<HPG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)kScoreSmem);
        if (e0 != cudaSuccess) return e0;
        attr = true;
    }
    cudaError_t e = launch_map(score_hist_kernel<HPG>, dim3((unsigned)grid), dim3(kSplitThreads), kScoreSmem,
                               stream, pdl, smap, p);
    if (e != cudaSuccess) return e;
    const int fchunks = (p.r_cap + p.regions_per_cta - 1) / p.regions_per_cta;
    e = launch_ex(filter_kernel, dim3(fchunks, p.G, p.N), dim3(kSplitThreads), 0, stream, true, p);
    if (e != cudaSuccess) return e;
    const int P2 = pow2_at_least(p.top_k);
    const size_t smem = (size_t)P2 * 8 + (size_t)kCandCap * 8;
    e = cudaFuncSetAttribute(final_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_ex2(final_select_kernel, dim3(kFinalSlices, p.G, p.N), dim3(kFinalThreads), smem, stream, true,
                      p, P2, 0);
}

}  // namespace

cudaError_t launch_score_fused(const ScoreParams& p, cudaStream_t stream, bool pdl) {
    switch (p.hpg) {
        case 1: return fused_for<1>(p, stream, pdl);
        case 2: return fused_for<2>(p, stream, pdl);
        case 4: return fused_for<4>(p, stream, pdl);
        case 8: return fused_for<8>(p, stream, pdl);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_score_split(const ScoreParams& p, const CUtensorMap& smap, cudaStream_t stream, bool pdl) {
    switch (p.hpg) {
        case 1: return split_for<1>(p, smap, stream, pdl);
        case 2: return split_for<2>(p, smap, stream, pdl);
        case 4: return split_for<4>(p, smap, stream, pdl);
        case 8: return split_for<8>(p, smap, stream, pdl);
    }
    return cudaErrorInvalidValue;
}

}  // namespace step5
