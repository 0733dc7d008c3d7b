// score_select.cu -- steps (2) and (3): FP8 index scores and top-k by (-score, id).
//
// "Step-5-Preview on one 256 GB Mac" (TensorFold PR #903), CSA-indexer commit: a
// region's score in a KV group is sum_h relu(e4m3(q_h) . summary) * w_h over the group's
// indexer heads; the 512 smallest (-score, id) keys are kept, in key order.  Provider groups own contiguous blocks of indexer heads (vLLM Step5 DSA
// geometry: the indexer's scores are summed within each provider group).
//
// Scoring: on the CUDA cores for the fused path (with 4 indexer heads per group a thread
// scores whole regions, two at a time against a shared-memory query broadcast; otherwise
// each region is read as four 16-byte vectors, one per thread, and a butterfly completes
// the 64-dim dot products; every e4m3 pair is widened to an f16 pair, exact, and
// multiplied by the mixed-precision fma, f16 products into an fp32 addend, which gives
// the bits of an fp32 fma on the decoded values), and on the tensor cores (e4m3 MMAs into
// TMEM) in the split path with 4 heads per group and in score_tc.cu.
// Selection orders 64-bit keys (desc(score) << 32 | id), which are unique, so any exact
// selection yields the same ordered ids.
//
// Selection paths with identical picks from the same scores:
//  * fused (and path 3's selection from stored scores): one block per (row, group)
//    keeps the row's 32-bit score keys in shared memory and runs the block top-k: the
//    keys' range, 11-bit digits below the bits the range fixes until the k-th key's bin
//    is small, the keys below it taken, the bin's keys ranked on chip, then a counting
//    sort of the picks.
//  * split: one persistent launch for few rows with many regions (decode at 128K-1M
//    tokens).  Blocks score an even share each and add a 12-bit histogram of the keys
//    into global memory; after a grid barrier each block copies its keys in or above
//    the bin holding the k-th key into a candidate list; after a second barrier the
//    blocks place every candidate at its rank (a count of the smaller candidates).
#include "kernels.cuh"
#include "tcgen05.cuh"

namespace step5 {

namespace {

// ----------------------------------------------------------------- query fragment

template <int HPG>
struct QFrag {
    uint32_t q[HPG][8];  // e4m3 query of head h at dims 16*qd + 2i, 16*qd + 2i + 1 (f16 pair)
    float w[HPG];        // w of every head (HPG == 4: w[0] holds head qd's weight)
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
            f.q[h][i] = pack_f16x2(s_q[h * 64 + 16 * qd + 2 * i], s_q[h * 64 + 16 * qd + 2 * i + 1]);
    }
}

// ----------------------------------------------------------------- one thread per region
//
// For 4 indexer heads per group: a thread scores whole regions (64 dims, 4 heads), two at
// a time, so no cross-lane reduction is needed.  Both operands of every product are e4m3
// values, which f16 holds exactly, so the summaries are widened only to f16 (one cvt per
// two dims) and the products accumulate in fp32 through the mixed-precision fma (f16
// inputs, fp32 addend and result, one rounding): the same bits as an fp32 fma on the
// decoded values, at fewer instructions per product than widening every value to fp32.
// The query lives in shared memory as qh[pair] = 4 words, word h = the f16 pair
// (q_h[2 pair], q_h[2 pair + 1]); every lane reads the same words (broadcast) and one
// load serves both regions.

// Packs s_q [4][64] (e4m3-valued floats) into qh [32] uint4; ends with a __syncthreads.
__device__ __forceinline__ void build_qh(const float* s_q, uint32_t* qh) {
    if (threadIdx.x < 128) {
        const int pr = threadIdx.x >> 2, h = threadIdx.x & 3;
        qh[threadIdx.x] = pack_f16x2(s_q[h * 64 + 2 * pr], s_q[h * 64 + 2 * pr + 1]);
    }
    __syncthreads();
}

// Two f16 pairs of e4m3-valued elements, widened from two e4m3 bytes.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
    return h2;
}

// lo += q.lo * x.lo and hi += q.hi * x.hi (f16 pairs q and x, fp32 accumulators).
__device__ __forceinline__ void fma_f16x2_f32(float& lo, float& hi, uint32_t q, uint32_t x) {
    asm("{.reg .f16 q0, q1, x0, x1;\n\t"
        "mov.b32 {q0, q1}, %2;\n\t"
        "mov.b32 {x0, x1}, %3;\n\t"
        "fma.rn.f32.f16 %0, q0, x0, %0;\n\t"
        "fma.rn.f32.f16 %1, q1, x1, %1;}"
        : "+f"(lo), "+f"(hi)
        : "r"(q), "r"(x));
}

__device__ __forceinline__ float finish_score4(const float (&ev)[4], const float (&od)[4], const float (&w)[4]) {
    float sc = 0.0f;
#pragma unroll
    for (int h = 0; h < 4; ++h) sc = fmaf(fmaxf(__fadd_rn(ev[h], od[h]), 0.0f), w[h], sc);
    return __fadd_rn(sc, 0.0f);  // -0 -> +0
}

// Scores of two regions whose 64 summary bytes are a[0..3] and b[0..3] (dims 16k..16k+15
// in chunk k).  Each head's dot product is the sum of an even-dim and an odd-dim partial
// sum, each accumulated in dim order.
__device__ __forceinline__ void score_rows2(const uint4 (&a)[4], const uint4 (&b)[4], const uint4* qh,
                                            const float (&w)[4], float& sa, float& sb) {
    float ae[4], ao[4], be[4], bo[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) ae[h] = ao[h] = be[h] = bo[h] = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t wa[4] = {a[k].x, a[k].y, a[k].z, a[k].w};
        const uint32_t wb[4] = {b[k].x, b[k].y, b[k].z, b[k].w};
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
#pragma unroll
            for (int hw = 0; hw < 2; ++hw) {  // low / high 16 bits: pair 8k + 2qq + hw
                const uint32_t xa = e4m3x2_to_f16x2((uint16_t)(hw ? wa[qq] >> 16 : wa[qq] & 0xffffu));
                const uint32_t xb = e4m3x2_to_f16x2((uint16_t)(hw ? wb[qq] >> 16 : wb[qq] & 0xffffu));
                const uint4 q = qh[8 * k + 2 * qq + hw];
                const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    fma_f16x2_f32(ae[h], ao[h], qw[h], xa);
                    fma_f16x2_f32(be[h], bo[h], qw[h], xb);
                }
            }
        }
    }
    sa = finish_score4(ae, ao, w);
    sb = finish_score4(be, bo, w);
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
        const uint32_t s0 = e4m3x2_to_f16x2((uint16_t)(w4[q] & 0xffffu));
        const uint32_t s1 = e4m3x2_to_f16x2((uint16_t)(w4[q] >> 16));
#pragma unroll
        for (int h = 0; h < HPG; ++h) {
            fma_f16x2_f32(acc[h].x, acc[h].y, f.q[h][2 * q], s0);
            fma_f16x2_f32(acc[h].x, acc[h].y, f.q[h][2 * q + 1], s1);
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

// The candidates (the K-th key's bin, once it holds at most kSelCands keys) live in the
// first half of hist, and the counts of their own descent (kCandBits digits) after them.
constexpr int kCandBits = 8;
constexpr int kCandBins = 1 << kCandBits;
constexpr int kSelCands = 512;
constexpr int kSelRankMax = 24;  // a bin or a sort segment this small is ranked pairwise
static_assert(kSelCands * 2 + kCandBins <= kRadixBins, "candidates and their counts fit the histogram");

struct TopkSmem {
    uint32_t hist[kRadixBins];
    uint32_t wsum[32];
    uint32_t count, ncand, nmem;
    uint32_t v, before, inbin;
    uint32_t kmin, kmax;  // range of the score keys
    uint32_t segmax;      // longest segment of the counting sort
};

// Scratch of the selection and its sort, in 64-bit keys.
__host__ __device__ constexpr int sel_aux_slots(int P2) { return P2 > kSelCands ? P2 : kSelCands; }

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

// The bin holding the need-th smallest key (need >= 1) of the NB digit counts in hist:
// ts.v = the bin, ts.before = keys in lower bins, ts.inbin = keys in the bin.  Called by
// all NT threads once the counts are complete; ends with a barrier.
template <int NT, int NB>
__device__ void block_find_bin(const uint32_t* hist, uint32_t need, TopkSmem& ts) {
    constexpr int PER = NB >= NT ? NB / NT : 1;  // bins per thread (threads past NB own none)
    constexpr int NW = NT / 32;
    static_assert(NB % NT == 0 || NT % NB == 0, "bins divide among the threads");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t loc[PER];
    uint32_t sum = 0;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        loc[q] = tid * PER < NB ? hist[tid * PER + q] : 0u;
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
    if (excl < need && need <= incl) {
        uint32_t c = excl;
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            if (c + loc[q] >= need) {
                ts.v = tid * PER + q;
                ts.before = c;
                ts.inbin = loc[q];
                break;
            }
            c += loc[q];
        }
    }
    __syncthreads();
}

// Exclusive scan, in place, of the NB counts in hist; the largest count goes to
// ts.segmax (set to 0 beforehand).  Called by all NT threads; ends with a barrier.
template <int NT, int NB>
__device__ void block_excl_scan_bins(uint32_t* hist, TopkSmem& ts) {
    constexpr int PER = NB / NT;
    constexpr int NW = NT / 32;
    static_assert(NB % NT == 0 && PER >= 1, "bins divide among the threads");  // NB >= NT here
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t loc[PER];
    uint32_t sum = 0, mx = 0;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        loc[q] = hist[tid * PER + q];
        sum += loc[q];
        mx = max(mx, loc[q]);
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) atomicMax(&ts.segmax, mx);
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
        if (lane < NW) ts.wsum[lane] = w;
    }
    __syncthreads();
    uint32_t c = incl - sum + (warp ? ts.wsum[warp - 1] : 0u);
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        hist[tid * PER + q] = c;
        c += loc[q];
    }
    __syncthreads();
}

// Appends the keys of the lanes with `act` set to list[*ctr ...] (slots past cap dropped).
__device__ __forceinline__ void warp_append(bool act, uint64_t key, uint64_t* list, uint32_t* ctr, uint32_t cap) {
    const int lane = threadIdx.x & 31;
    const uint32_t am = __ballot_sync(0xffffffffu, act);
    uint32_t slot = 0;
    if (lane == 0 && am) slot = atomicAdd(ctr, (uint32_t)__popc(am));
    slot = __shfl_sync(0xffffffffu, slot, 0);
    if (act) {
        const uint32_t idx = slot + __popc(am & ((1u << lane) - 1u));
        if (idx < cap) list[idx] = key;
    }
}

// Gathers the K smallest keys (desc(score) << 32 | id, i.e. by score key and then by id)
// of ids 0..cnt-1 (all of them if cnt <= K) into s_sel[0..min(cnt, K)) in no particular
// order, pads s_sel up to P2 (a power of two >= max(K, 32)) with ~0, returns min(cnt, K).
// src(i) returns the 32-bit score key of id i and src.get4(j, cnt) those of ids 4j..4j+3
// (entries past cnt undefined); s_aux holds sel_aux_slots(P2) keys of scratch.
// A radix descent over 11-bit digits, one pass over all keys each (four per thread per
// 16-byte shared load), until the K-th key's bin is taken whole, holds at most kSelCands
// keys, or is one key value.  The first digit is either the keys' top bits, counted by
// the caller as it wrote the keys (first_given: ts.hist holds those counts), or the 11
// bits below those that the range [smallest, largest] of the keys fixes (a pass for the
// range first: scores of one row mostly share sign and exponent).  Then a pass counts
// each thread's keys below the bin and in it and one writes them (every key below the
// bin taken, the bin's keys kept as candidates), with one slot reservation per thread in
// between.  The candidates descend by 8-bit digits until their bin is taken whole or
// holds at most kSelRankMax keys, which are ranked against each other by (key, id).  A
// single key value shared by more than kSelCands keys is resolved by one warp taking the
// smallest ids in id order.  Must be called by all NT threads of the block.
template <int NT, class Src>
__device__ int block_select_set(const Src& src, int cnt, int K, int P2, uint64_t* s_sel, uint64_t* s_aux,
                                TopkSmem& ts, bool first_given = false) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n4 = (cnt + 3) >> 2;
    uint64_t lo = 1ull << 32, hi_excl = 1ull << 32;  // keys below lo taken; [lo, hi_excl) the bin
    int need = 0;                                   // keys still needed from the bin
    int hi = 0;                                     // bits of the bin's keys at and above hi agree
    int mode = 0;                                   // 0 bin taken whole, 1 candidates, 2 ties
    // first_given: ts.hist already holds the counts of the keys' top kRadixBits bits (taken
    // by the caller's pass that wrote the keys): they are the descent's first level, and
    // no pass for the keys' range is needed
    bool given = first_given;
    if (cnt > K && given) {
        need = K;
        hi = 32;
    }
    if (cnt > K && !given) {
        if (tid == 0) {
            ts.kmin = ~0u;
            ts.kmax = 0u;
        }
        uint32_t mn = ~0u, mx = 0u;
        for (int j = tid; j < n4; j += NT) {
            const uint4 k = src.get4(j, cnt);
            const int i0 = 4 * j;
            mn = min(mn, k.x);
            mx = max(mx, k.x);
            if (i0 + 3 < cnt) {
                mn = min(min(mn, k.y), min(k.z, k.w));
                mx = max(max(mx, k.y), max(k.z, k.w));
            } else {
                if (i0 + 1 < cnt) { mn = min(mn, k.y); mx = max(mx, k.y); }
                if (i0 + 2 < cnt) { mn = min(mn, k.z); mx = max(mx, k.z); }
            }
        }
        mn = __reduce_min_sync(0xffffffffu, mn);
        mx = __reduce_max_sync(0xffffffffu, mx);
        __syncthreads();  // the range is initialised
        if (lane == 0) {
            atomicMin(&ts.kmin, mn);
            atomicMax(&ts.kmax, mx);
        }
        __syncthreads();
        need = K;
        if (ts.kmin != ts.kmax) hi = 32 - __clz(ts.kmin ^ ts.kmax);
    }
    if (cnt > K) {
        uint32_t prefix = given ? 0u : (hi >= 32 ? 0u : (hi == 0 ? ts.kmin : (ts.kmin & (~0u << hi))));
        uint32_t inbin = (uint32_t)cnt;  // keys sharing the fixed bits
        while (hi > 0 && inbin > (uint32_t)kSelCands) {
            const int width = hi >= kRadixBits ? kRadixBits : hi;
            const int shift = hi - width;
            const uint32_t dmask = (1u << width) - 1u;
            if (!given) {
                for (int i = tid; i < kRadixBins; i += NT) ts.hist[i] = 0;
                __syncthreads();
                const uint32_t mask = hi >= 32 ? 0u : (~0u << hi);
                for (int j = tid; j < n4; j += NT) {
                    const uint4 k = src.get4(j, cnt);
                    const uint32_t u[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (4 * j + q < cnt && (u[q] & mask) == prefix)
                            atomicAdd(&ts.hist[(u[q] >> shift) & dmask], 1u);
                }
                __syncthreads();
            }
            given = false;
            block_find_bin<NT, kRadixBins>(ts.hist, (uint32_t)need, ts);
            prefix |= ts.v << shift;
            need -= (int)ts.before;
            inbin = ts.inbin;
            hi = shift;
            if ((int)inbin == need) break;
        }
        lo = prefix;
        hi_excl = lo + (1ull << hi);
        if ((int)inbin == need) {
            lo = hi_excl;  // the whole bin is taken
            need = 0;
        } else {
            mode = inbin <= (uint32_t)kSelCands ? 1 : 2;  // mode 2: hi == 0, one key value
        }
    }
    uint64_t* cand = reinterpret_cast<uint64_t*>(ts.hist);
    const uint32_t aux_cap = (uint32_t)sel_aux_slots(P2);
    if (tid == 0) {
        ts.count = 0;
        ts.ncand = 0;
        ts.nmem = 0;
    }
    for (int i = tid; i < P2; i += NT) s_sel[i] = ~0ull;
    __syncthreads();
    {
        // a thread counts its keys below the bin (taken) and in it (candidates), reserves
        // its slots with one atomic per list, then writes them in a second sweep
        const uint64_t b_hi = mode == 1 ? hi_excl : lo;
        uint32_t na = 0, nb = 0;
        for (int j = tid; j < n4; j += NT) {
            const uint4 k = src.get4(j, cnt);
            const uint32_t u[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool ok = 4 * j + q < cnt;
                na += ok && (uint64_t)u[q] < lo;
                nb += ok && (uint64_t)u[q] >= lo && (uint64_t)u[q] < b_hi;
            }
        }
        uint32_t sa = na ? atomicAdd(&ts.count, na) : 0u;
        uint32_t sb = nb ? atomicAdd(&ts.ncand, nb) : 0u;
        for (int j = tid; j < n4 && (na | nb) != 0u; j += NT) {
            const uint4 k = src.get4(j, cnt);
            const uint32_t u[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = 4 * j + q;
                if (i >= cnt) continue;
                const uint64_t key = ((uint64_t)u[q] << 32) | (uint32_t)i;
                if ((uint64_t)u[q] < lo) {
                    if (sa < (uint32_t)P2) s_sel[sa] = key;
                    ++sa;
                    --na;
                } else if ((uint64_t)u[q] < b_hi) {
                    if (sb < (uint32_t)kSelCands) cand[sb] = key;
                    ++sb;
                    --nb;
                }
            }
        }
    }
    __syncthreads();
    if (mode == 1) {
        // the candidates' own descent, on 8-bit digits
        const int nc = min((int)ts.ncand, kSelCands);
        uint32_t* chist = ts.hist + 2 * kSelCands;
        uint32_t cprefix = (uint32_t)lo;
        int chi = hi;
        int cin = nc;
        while (chi > 0 && cin > kSelRankMax) {
            const int width = chi >= kCandBits ? kCandBits : chi;
            const int shift = chi - width;
            const uint32_t dmask = (1u << width) - 1u;
            for (int i = tid; i < kCandBins; i += NT) chist[i] = 0;
            __syncthreads();
            const uint32_t mask = chi >= 32 ? 0u : (~0u << chi);
            for (int j = tid; j < nc; j += NT) {
                const uint32_t u = (uint32_t)(cand[j] >> 32);
                if ((u & mask) == cprefix) atomicAdd(&chist[(u >> shift) & dmask], 1u);
            }
            __syncthreads();
            block_find_bin<NT, kCandBins>(chist, (uint32_t)need, ts);
            cprefix |= ts.v << shift;
            need -= (int)ts.before;
            cin = (int)ts.inbin;
            chi = shift;
            if (cin == need) break;
        }
        const uint64_t c_lo = cprefix, c_hi = c_lo + (1ull << chi);
        const bool whole = cin == need;
        // candidates below the bin are taken (and the bin, when all of it is needed); the
        // bin's keys otherwise go to a member list ranked pairwise
        for (int base = 0; base < nc; base += NT) {
            const int j = base + tid;
            uint64_t key = 0;
            bool tk = false, mem = false;
            if (j < nc) {
                key = cand[j];
                const uint64_t u = key >> 32;
                tk = u < c_lo || (whole && u < c_hi);
                mem = !tk && u < c_hi;
            }
            warp_append(tk, key, s_sel, &ts.count, (uint32_t)P2);
            warp_append(mem, key, s_aux, &ts.nmem, aux_cap);
        }
        __syncthreads();
        const uint32_t taken = ts.count;
        const int m = min((int)ts.nmem, (int)aux_cap);
        for (int j = tid; j < m; j += NT) {
            const uint64_t key = s_aux[j];
            int r = 0;
            for (int i = 0; i < m; ++i) r += s_aux[i] < key;
            if (r < need && taken + r < (uint32_t)P2) s_sel[taken + r] = key;
        }
    } else if (mode == 2 && warp == 0) {
        // keys equal to the K-th key: the smallest ids, scanned in id order
        const uint32_t tie_key = (uint32_t)lo;
        uint32_t taken = ts.count;
        int left = need;
        for (int base = 0; base < cnt && left > 0; base += 32) {
            const int i = base + lane;
            const bool eq = i < cnt && src(i) == tie_key;
            const uint32_t m = __ballot_sync(0xffffffffu, eq);
            const int r = __popc(m & ((1u << lane) - 1u));
            if (eq && r < left && taken + r < (uint32_t)P2)
                s_sel[taken + r] = ((uint64_t)tie_key << 32) | (uint32_t)i;
            const int c = min(__popc(m), left);
            taken += c;
            left -= c;
        }
    }
    __syncthreads();
    return cnt < K ? cnt : K;
}

// Ascending sort of the take unique keys in s_sel[0..take) (s_sel padded with ~0 up to
// P2).  A counting sort on the 11 bits below those the selected score keys share: the
// digit counts, their exclusive scan, a scatter into s_aux, then each key's place in its
// segment by counting the segment's smaller keys.  When a segment is longer than
// kSelRankMax (or every score key is equal) the bitonic sort runs instead.  Must be
// called by all NT threads.
template <int NT>
__device__ void block_sort_selected(uint64_t* s_sel, int take, int P2, uint64_t* s_aux, TopkSmem& ts) {
    const int tid = threadIdx.x, lane = tid & 31;
    if (take <= 1) return;
    if (tid == 0) {
        ts.kmin = ~0u;
        ts.kmax = 0u;
        ts.segmax = 0u;
    }
    uint32_t mn = ~0u, mx = 0u;
    for (int j = tid; j < take; j += NT) {
        const uint32_t u = (uint32_t)(s_sel[j] >> 32);
        mn = min(mn, u);
        mx = max(mx, u);
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    __syncthreads();
    if (lane == 0) {
        atomicMin(&ts.kmin, mn);
        atomicMax(&ts.kmax, mx);
    }
    for (int i = tid; i < kRadixBins; i += NT) ts.hist[i] = 0;
    __syncthreads();
    const uint32_t kmin = ts.kmin, kmax = ts.kmax;
    bool counting = kmin != kmax;
    if (counting) {
        const int hi = 32 - __clz(kmin ^ kmax);
        const int shift = hi > kRadixBits ? hi - kRadixBits : 0;
        const uint32_t dmask = (1u << (hi - shift)) - 1u;
        for (int j = tid; j < take; j += NT)
            atomicAdd(&ts.hist[(uint32_t)(s_sel[j] >> (32 + shift)) & dmask], 1u);
        __syncthreads();
        block_excl_scan_bins<NT, kRadixBins>(ts.hist, ts);
        counting = ts.segmax <= (uint32_t)kSelRankMax;
        if (counting) {
            for (int j = tid; j < take; j += NT) {
                const uint64_t key = s_sel[j];
                const uint32_t d = (uint32_t)(key >> (32 + shift)) & dmask;
                s_aux[atomicAdd(&ts.hist[d], 1u)] = key;
            }
            __syncthreads();
            // hist[d] is now the end of segment d, and hist[d - 1] its start
            for (int j = tid; j < take; j += NT) {
                const uint64_t key = s_aux[j];
                const uint32_t d = (uint32_t)(key >> (32 + shift)) & dmask;
                const int s0 = d ? (int)ts.hist[d - 1] : 0;
                const int s1 = (int)ts.hist[d];
                int r = s0;
                for (int i = s0; i < s1; ++i) r += s_aux[i] < key;
                s_sel[r] = key;
            }
            __syncthreads();
        }
    }
    if (!counting) block_bitonic_sort<NT>(s_sel, P2);
}

// block_select_set followed by an ascending sort of the gathered keys.
template <int NT, class Src>
__device__ int block_topk(const Src& src, int cnt, int K, int P2, uint64_t* s_sel, uint64_t* s_aux, TopkSmem& ts,
                          bool first_given = false) {
    const int take = block_select_set<NT>(src, cnt, K, P2, s_sel, s_aux, ts, first_given);
    block_sort_selected<NT>(s_sel, take, P2, s_aux, ts);
    return take;
}

// Key sources for block_topk: the 32-bit score key desc(score) of id i, and of ids
// 4j..4j+3 at once (entries at or past cnt undefined).
struct SmemKeys {  // keys in shared memory, indexed by region id, 16-byte aligned and
                   // readable up to the next multiple of 4
    const uint32_t* key;
    __device__ __forceinline__ uint32_t operator()(int i) const { return key[i]; }
    __device__ __forceinline__ uint4 get4(int j, int) const { return reinterpret_cast<const uint4*>(key)[j]; }
};
struct ScoreKeys {  // every score of the row, from global memory
    const float* scores;
    __device__ __forceinline__ uint32_t operator()(int i) const { return desc_key(scores[i]); }
    __device__ __forceinline__ uint4 get4(int j, int cnt) const {
        const int i = 4 * j;
        return make_uint4(desc_key(scores[i]), i + 1 < cnt ? desc_key(scores[i + 1]) : 0u,
                          i + 2 < cnt ? desc_key(scores[i + 2]) : 0u, i + 3 < cnt ? desc_key(scores[i + 3]) : 0u);
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
            ids[i] = (int32_t)(uint32_t)(key & 0xffffffffu) + p.region_lo;
            if (ss) ss[i] = score_of_desc_key((uint32_t)(key >> 32));
        } else {
            ids[i] = -1;
            if (ss) ss[i] = -INFINITY;
        }
    }
    if (threadIdx.x == 0) p.sel_count[ng] = take;
}

// ----------------------------------------------------------------- fused path

constexpr int kFusedThreads = 256;

// FROM_SCORES: the scores are already in p.scores (written by the tensor-core scoring
// kernel); the block only selects.
template <int HPG, bool FROM_SCORES>
__global__ void __launch_bounds__(kFusedThreads) score_fused_kernel(ScoreParams p, int P2, int key_cap) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint64_t* s_sel = reinterpret_cast<uint64_t*>(smem);                 // P2
    uint64_t* s_aux = s_sel + P2;                                        // sel_aux_slots(P2)
    uint32_t* s_key = reinterpret_cast<uint32_t*>(s_aux + sel_aux_slots(P2));  // key_cap
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
    // the counts of the keys' top kRadixBits bits are taken as the keys are written (the
    // selection's first digit)
    for (int i = threadIdx.x; i < kRadixBins; i += kFusedThreads) ts.hist[i] = 0;
    __syncthreads();
    if constexpr (FROM_SCORES) {
        // the row's scores: 16 bytes a thread and four loads in flight, where aligned
        int r_done = 0;
        if ((reinterpret_cast<uintptr_t>(exp_scores) & 15u) == 0) {
            const float4* s4 = reinterpret_cast<const float4*>(exp_scores);
            uint4* k4 = reinterpret_cast<uint4*>(s_key);
            const int R4 = R >> 2;
            constexpr int U = 4;
            for (int j0 = 0; j0 < R4; j0 += U * kFusedThreads) {
                float4 v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = j0 + u * kFusedThreads + threadIdx.x;
                    v[u] = j < R4 ? __ldcg(s4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = j0 + u * kFusedThreads + threadIdx.x;
                    if (j < R4) {
                        const uint4 kk = make_uint4(desc_key(v[u].x), desc_key(v[u].y), desc_key(v[u].z),
                                                    desc_key(v[u].w));
                        k4[j] = kk;
                        atomicAdd(&ts.hist[kk.x >> (32 - kRadixBits)], 1u);
                        atomicAdd(&ts.hist[kk.y >> (32 - kRadixBits)], 1u);
                        atomicAdd(&ts.hist[kk.z >> (32 - kRadixBits)], 1u);
                        atomicAdd(&ts.hist[kk.w >> (32 - kRadixBits)], 1u);
                    }
                }
            }
            r_done = R4 << 2;
        }
        for (int r = r_done + threadIdx.x; r < R; r += kFusedThreads) {
            const uint32_t kk = desc_key(__ldcg(exp_scores + r));
            s_key[r] = kk;
            atomicAdd(&ts.hist[kk >> (32 - kRadixBits)], 1u);
        }
    } else if constexpr (HPG == 4) {
        __shared__ uint4 s_qh[32];
        float w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) w[h] = p.w[(int64_t)n * p.idx_heads + (int64_t)g * 4 + h];
        stage_query<4>(p, n, g, pos, s_q);
        build_qh(s_q, reinterpret_cast<uint32_t*>(s_qh));
        for (int r0 = 0; r0 < R; r0 += 2 * kFusedThreads) {
            const int ra = r0 + threadIdx.x, rb = ra + kFusedThreads;
            uint4 va[4], vb[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                va[k] = ra < R ? __ldg(base + (int64_t)ra * 4 + k) : make_uint4(0, 0, 0, 0);
                vb[k] = rb < R ? __ldg(base + (int64_t)rb * 4 + k) : make_uint4(0, 0, 0, 0);
            }
            float sa, sb;
            score_rows2(va, vb, s_qh, w, sa, sb);
            if (ra < R) {
                const uint32_t ka = desc_key(sa);
                s_key[ra] = ka;
                atomicAdd(&ts.hist[ka >> (32 - kRadixBits)], 1u);
                if (exp_scores) exp_scores[ra] = sa;
            }
            if (rb < R) {
                const uint32_t kb = desc_key(sb);
                s_key[rb] = kb;
                atomicAdd(&ts.hist[kb >> (32 - kRadixBits)], 1u);
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
                const uint32_t k = desc_key(mysc);
                s_key[r] = k;
                atomicAdd(&ts.hist[k >> (32 - kRadixBits)], 1u);
                if (exp_scores) exp_scores[r] = mysc;
            }
        }
    }
    __syncthreads();
    const int take = block_topk<kFusedThreads>(SmemKeys{s_key}, R, p.top_k, P2, s_sel, s_aux, ts, true);
    write_selection<kFusedThreads>(p, n, g, take, s_sel);
}

// ----------------------------------------------------------------- split path

constexpr int kSplitThreads = 512;                     // one block per SM
// Registers per thread.  An SM's registers are split over its 4 schedulers (16,384
// each) and a warp takes its registers from one of them: 4 warps x 32 x 112 leave 2,048
// per scheduler, room for a warp of a 64-thread summary block of the launch before (at
// most 48 registers a thread; step (1) of the same decode step), so the scoring block of
// that SM starts at once instead of after it.
constexpr int kSplitMaxRegs = 112;
constexpr int kSplitWarps = kSplitThreads / 32;
constexpr int kBinsPerThread = kHistBins / kSplitThreads;  // histogram bins a thread owns

// ----------------------------------------------------------------- split path scoring
//
// Persistent blocks (one per SM) each walk an even share of the flattened (row, group,
// region) space in tiles of kTileRegions consecutive regions of one (row, group),
// contiguous in the summary store and fetched by TMA into a 2-stage shared-memory ring
// while the previous tile is scored.  Each run of tiles of one (row, group) adds its
// shared-memory histogram to the global one.

constexpr int kTileRegions = 2 * kSplitThreads;   // 64 KB of summaries
static_assert(kTileRegions == kSplitTileRegions, "host and device tile sizes differ");
constexpr int kTileBytes = kTileRegions * 64;
constexpr int kBoxRows = 256;                     // rows of one summary tensor-map box
constexpr int kSlots = kSplitThreads / 4;         // region slots of the 4-lane layout
constexpr int kTileU = kTileRegions / kSlots;     // regions per slot per tile (8)
constexpr int kScoreStages = 2;
constexpr uint32_t kQeBytes = 16 * 64;              // a group's e4m3 query tile (B operand)
constexpr size_t kScoreSmem = kScoreStages * kTileBytes + 2 * kQeBytes + 1024;
constexpr uint32_t kScoreTmemCols = 256;            // two accumulators of 8 subtiles x 16 columns
constexpr uint32_t kScoreIdesc = tc::instr_desc(tc::kFmtE4M3, false, false, 128, 16);

struct Tile {
    int valid, ng, n, g, b, pos, R, c0, c1;
};

// A block's walk over its range of the flattened (row, group, region) space (r_cap
// regions per (row, group)): the position, the regions of the range still ahead, and the
// position data of the current row (loaded once per row).
struct Walk {
    int64_t left;
    int ng, r;
    int cn, cb, cpos, cR;
};

__device__ __forceinline__ Walk walk_start(const ScoreParams& p, int64_t x, int64_t hi) {
    Walk k;
    k.left = hi - x;
    k.ng = (int)(x / p.r_cap);
    k.r = (int)(x - (int64_t)k.ng * p.r_cap);
    k.cn = -1;
    k.cb = k.cpos = k.cR = 0;
    return k;
}

// The next tile of the walk: at most kTileRegions consecutive candidate regions of one
// (row, group).  Regions past a row's R, and rows out of range, are skipped.
__device__ __forceinline__ Tile next_tile(const ScoreParams& p, Walk& k, int limit = kTileRegions) {
    Tile t;
    t.valid = 0;
    while (k.left > 0) {
        const int n = k.ng / p.G;
        if (n != k.cn) {
            k.cn = n;
            k.cR = row_regions(p, n, k.cb, k.cpos);
            if (k.cR < 0 && threadIdx.x == 0) raise_status(p.status, kDevRange);
        }
        if (k.r >= k.cR) {  // the rest of this (row, group) holds no candidate
            k.left -= p.r_cap - k.r;
            ++k.ng;
            k.r = 0;
            continue;
        }
        int c1 = min(k.cR, k.r + limit);
        if ((int64_t)(c1 - k.r) > k.left) c1 = k.r + (int)k.left;
        t.valid = 1;
        t.ng = k.ng;
        t.n = n;
        t.g = k.ng - n * p.G;
        t.b = k.cb;
        t.pos = k.cpos;
        t.R = k.cR;
        t.c0 = k.r;
        t.c1 = c1;
        k.left -= c1 - k.r;
        k.r = c1;
        return t;
    }
    return t;
}

// Scores one staged tile: thread (slot, qd) covers regions u * kSlots + slot, u < kTileU;
// lane qd of each region quad keeps the score and histogram update of every fourth
// region.  FULL: the tile holds kTileRegions regions (no bounds checks).
template <int HPG, bool FULL>
__device__ __forceinline__ void score_tile(const QFrag<HPG>& f, const uint4* tile, int nreg, float* scores,
                                           float* keep, uint32_t* s_hist, int qd, int slot) {
#pragma unroll
    for (int u4 = 0; u4 < kTileU; u4 += 4) {
        float sc[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int lr = (u4 + u) * kSlots + slot;
            const uint4 v = (FULL || lr < nreg) ? tile[lr * 4 + qd] : make_uint4(0, 0, 0, 0);
            sc[u] = score_from_vec<HPG>(f, v);
        }
        const float mysc = qd == 0 ? sc[0] : qd == 1 ? sc[1] : qd == 2 ? sc[2] : sc[3];
        const int lr = (u4 + qd) * kSlots + slot;
        if (FULL || lr < nreg) {
            scores[lr] = mysc;
            if (keep) keep[lr] = mysc;
            atomicAdd(&s_hist[desc_key(mysc) >> (32 - kHistBits)], 1u);
        }
    }
}

// The split path stages a (row, group)'s query in two parts so that its loads overlap
// the first tile's copy: load_query_raw reads the bf16 q (and NEOX partner dims) and the
// weights, which need only (n, g); load_rope reads cos/sin at the row's position;
// finish_query rotates, rounds to e4m3 and stores the query and weights into one of two
// shared-memory buffers.
template <int HPG>
struct QRaw {
    static constexpr int kPer = (HPG * 64 + kSplitThreads - 1) / kSplitThreads;
    uint16_t q[kPer], qp[kPer];  // element i = threadIdx.x + kSplitThreads * j
    float w;                     // weight of head threadIdx.x (threads below HPG)
};

template <int HPG>
__device__ __forceinline__ void load_query_raw(const ScoreParams& p, int n, int g, QRaw<HPG>& r) {
    const int half = p.rope_dims >> 1;
#pragma unroll
    for (int j = 0; j < QRaw<HPG>::kPer; ++j) {
        const int i = threadIdx.x + kSplitThreads * j;
        r.q[j] = r.qp[j] = 0;
        if (i < HPG * 64) {
            const int h = i >> 6, d = i & 63;
            const uint16_t* qrow = p.idx_q + ((int64_t)n * p.idx_heads + (int64_t)g * HPG + h) * 64;
            r.q[j] = qrow[d];
            if (p.cos != nullptr && d < p.rope_dims) r.qp[j] = qrow[d < half ? d + half : d - half];
        }
    }
    r.w = threadIdx.x < HPG ? p.w[(int64_t)n * p.idx_heads + (int64_t)g * HPG + threadIdx.x] : 0.0f;
}

// The bf16 cos/sin of each staged element's NEOX pair at position pos (zero when the
// element is not rotated).
template <int HPG>
struct QRope {
    uint16_t c[QRaw<HPG>::kPer], s[QRaw<HPG>::kPer];
};

template <int HPG>
__device__ __forceinline__ void load_rope(const ScoreParams& p, int pos, QRope<HPG>& r) {
    const int half = p.rope_dims >> 1;
#pragma unroll
    for (int j = 0; j < QRaw<HPG>::kPer; ++j) {
        const int i = threadIdx.x + kSplitThreads * j;
        const int d = i & 63;
        r.c[j] = r.s[j] = 0;
        if (i < HPG * 64 && p.cos != nullptr && d < p.rope_dims) {
            const int pi = d < half ? d : d - half;
            r.c[j] = p.cos[(int64_t)pos * half + pi];
            r.s[j] = p.sin[(int64_t)pos * half + pi];
        }
    }
}

// Shared-memory query buffers of the split scoring kernel.  HPG == 4 keeps the query as
// the f16 pairs of score_rows2 (qh); the others as q[h * 64 + d].
template <int HPG>
struct QBuf {
    static constexpr int kQ = HPG == 4 ? 4 : HPG * 64;
    static constexpr int kQh = HPG == 4 ? HPG * 64 : 8;
    float q[kQ];
    __align__(16) uint16_t qh[kQh];
    float w[HPG];
};

// e4m3(bf16(NEOX(q))) of each staged element, and the weights, into buffer qb.  The
// caller synchronises before reading it.
template <int HPG>
__device__ __forceinline__ void finish_query(const ScoreParams& p, const QRaw<HPG>& r, const QRope<HPG>& ro,
                                             QBuf<HPG>& qb, uint8_t* qe = nullptr) {
    const int half = p.rope_dims >> 1;
#pragma unroll
    for (int j = 0; j < QRaw<HPG>::kPer; ++j) {
        const int i = threadIdx.x + kSplitThreads * j;
        if (i < HPG * 64) {
            const int h = i >> 6, d = i & 63;
            uint16_t rb = r.q[j];
            if (p.cos != nullptr && d < p.rope_dims)
                rb = neox_rotate(bf16_to_f32(rb), bf16_to_f32(r.qp[j]), bf16_to_f32(ro.c[j]), bf16_to_f32(ro.s[j]),
                                 d < half);
            const uint8_t code = f32_to_e4m3(bf16_to_f32(rb));
            const float v = e4m3x2_to_f32x2(code).x;
            if constexpr (HPG == 4) {
                qb.qh[(d >> 1) * 8 + h * 2 + (d & 1)] = __half_as_ushort(__float2half_rn(v));
                // the tensor cores' B operand: head h = row h, K-major, 64-byte swizzle
                if (qe) qe[h * 64 + ((((d >> 4) ^ ((h >> 1) & 3))) << 4) + (d & 15)] = code;
            } else {
                qb.q[i] = v;
            }
        }
    }
    if (threadIdx.x < HPG) qb.w[threadIdx.x] = r.w;
    if (qe) fence_proxy_async();  // the MMAs read the tile through the async proxy
}

// The 4-lanes-per-region query registers from a staged buffer (after a __syncthreads).
template <int HPG>
__device__ __forceinline__ void qfrag_from_smem(const QBuf<HPG>& qb, QFrag<HPG>& f) {
    const int qd = threadIdx.x & 3;
#pragma unroll
    for (int h = 0; h < HPG; ++h) f.w[h] = qb.w[h];
#pragma unroll
    for (int h = 0; h < HPG; ++h) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            f.q[h][i] = pack_f16x2(qb.q[h * 64 + 16 * qd + 2 * i], qb.q[h * 64 + 16 * qd + 2 * i + 1]);
    }
}

// Position of row n for its rope lookup, 0 when the row is out of range (its tiles are
// skipped).
__device__ __forceinline__ int row_pos_or0(const ScoreParams& p, int n) {
    int b, pos;
    return row_regions(p, n, b, pos) < 0 ? 0 : pos;
}

// One staged tile on the tensor cores (4 indexer heads per group), in two halves so that
// the products of the next tile overlap the epilogue of this one:
//  * tc_tile_issue (thread 0): for each 128-region subtile that holds regions, two e4m3
//    MMAs (K = 32 each) of the subtile against the group's query tile (heads as rows 0-3
//    of N = 16) into TMEM columns d + 16 m .. d + 16 m + 3, then a commit to dbar;
//  * tc_tile_epilogue (all threads, after dbar): the 16 warps read their regions' head
//    sums (warp w: subtiles w / 4 and w / 4 + 4, lanes 32 (w % 4) ..) and finish each score as the
//    CUDA-core path does: sum_h relu(dot_h) * w_h in fp32, heads in order.
// The e4m3 products are exact, so the scores differ from the CUDA-core path's only by the
// summation order of each 64-term dot product.
__device__ __forceinline__ void tc_tile_issue(const uint8_t* tile, const uint8_t* qe, int nreg, uint32_t d,
                                              uint64_t* dbar) {
    tc::fence_after_sync();
    const int nsub = (nreg + 127) >> 7;
    const uint64_t db = tc::smem_desc(smem_u32(qe), 16, 512, tc::kSwizzle64);
    const uint64_t da0 = tc::smem_desc(smem_u32(tile), 16, 512, tc::kSwizzle64);
    for (int m = 0; m < nsub; ++m) {
        const uint64_t da = da0 + (uint64_t)(512 * m);  // + m * 8 KB, in 16-byte units
        tc::mma_f8(d + 16u * m, da, db, kScoreIdesc, false);
        tc::mma_f8(d + 16u * m, da + 2, db + 2, kScoreIdesc, true);  // dims 32-63 (+32 bytes)
    }
    tc::commit(dbar);
}

__device__ __forceinline__ void tc_tile_epilogue(int nreg, uint32_t d, const float* wsm, float* scores, float* keep,
                                                 uint32_t* s_hist) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsub = (nreg + 127) >> 7;
    const int q = warp & 3;
    float w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) w[h] = wsm[h];
    for (int m = warp >> 2; m < nsub; m += kSplitWarps / 4) {  // (uniform per warp)
        float dv[4];
        tc::ld4(tc::taddr(d, 32 * q, 16u * m), dv);
        const int lr = m * 128 + 32 * q + lane;
        if (lr < nreg) {
            float sc = 0.0f;
#pragma unroll
            for (int h = 0; h < 4; ++h) sc = fmaf(fmaxf(dv[h], 0.0f), w[h], sc);
            sc = __fadd_rn(sc, 0.0f);  // -0 -> +0
            scores[lr] = sc;
            if (keep) keep[lr] = sc;
            atomicAdd(&s_hist[desc_key(sc) >> (32 - kHistBits)], 1u);
        }
    }
    tc::fence_before_sync();
}

// ----------------------------------------------------------------- grid-wide steps

// Block-wide exclusive scan of one count per thread; returns the thread's offset and
// leaves the block total in *total.  s_w: kSplitThreads / 32 words of scratch.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* s_w, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kSplitThreads / 32; ++w) {
        const uint32_t c = s_w[w];
        before += w < warp ? c : 0u;
        tot += c;
    }
    __syncthreads();
    *total = tot;
    return before + incl - v;
}

// Fine bin holding the K-th smallest key of a (row, group) with R regions, from its
// whole histogram (one 16 KB read shared by the block: each thread owns kBinsPerThread
// consecutive bins, h); kHistBins - 1 when R <= K or the histogram counts fewer than K
// keys.  Called by the whole block; the result lands in *s_out.
__device__ void block_threshold(const uint4 (&h)[kBinsPerThread / 4], int R, int K, uint32_t* s_w, int* s_out) {
    if (threadIdx.x == 0) *s_out = kHistBins - 1;
    uint32_t loc[kBinsPerThread];
#pragma unroll
    for (int q = 0; q < kBinsPerThread / 4; ++q) {
        loc[4 * q] = h[q].x;
        loc[4 * q + 1] = h[q].y;
        loc[4 * q + 2] = h[q].z;
        loc[4 * q + 3] = h[q].w;
    }
    uint32_t sum = 0;
#pragma unroll
    for (int q = 0; q < kBinsPerThread; ++q) sum += loc[q];
    uint32_t tot = 0;
    const uint32_t before = block_excl_scan(sum, s_w, &tot);  // synchronises (after the default)
    if (R > K && before < (uint32_t)K && (uint32_t)K <= before + sum) {
        uint32_t c = before;
        int bin = kBinsPerThread - 1;
#pragma unroll
        for (int q = 0; q < kBinsPerThread; ++q) {
            if (bin == kBinsPerThread - 1 && c + loc[q] >= (uint32_t)K) bin = q;
            c += loc[q];
        }
        *s_out = threadIdx.x * kBinsPerThread + bin;
    }
    __syncthreads();
}

// Block holding flattened position x of a launch whose block b covers
// [total * b / grid, total * (b + 1) / grid).
__device__ __forceinline__ int block_of(int64_t x, int64_t total, int grid) {
    return (int)(((x + 1) * grid - 1) / total);
}

// Last of the blocks that contribute candidates to one (row, group) to arrive:
// releases this block's candidate writes and, for the last, acquires everyone's.
__device__ __forceinline__ bool arrive_last(uint32_t* ctr, uint32_t nblocks) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(ctr) : "memory");
    return old == nblocks - 1u;
}

// Per-(row, group) synchronisation words of the split path.  Each is a generation
// number (high bits) with a payload, so none needs clearing between calls:
//  * thr[ng] = gen << 12 | bin: the threshold bin, published by the last block to add
//    its histogram share (counted in arrive1[ng], which that block clears);
//  * bar2[ng] = gen << 16 | arrivals: a barrier over the (row, group)'s blocks once
//    their candidates are written; the last arrival clears the count and advances the
//    generation with one release add.

// Threshold of one (row, group), by the whole block that added its histogram share
// last: the fine bin holding the K-th key (block_threshold over the complete
// histogram).  Clears the arrival counter and the candidate counter for the candidates
// that follow, publishes thr[ng] = (gen + 1) << 12 | bin with release semantics, then
// clears the histogram.
__device__ void publish_threshold(const ScoreParams& p, int ng, uint32_t gen, uint32_t* s_w, int* s_tmp) {
    const int tid = threadIdx.x;
    uint4* gh = reinterpret_cast<uint4*>(p.hist + (int64_t)ng * kHistBins) + tid * (kBinsPerThread / 4);
    uint4 h[kBinsPerThread / 4];
#pragma unroll
    for (int q = 0; q < kBinsPerThread / 4; ++q) h[q] = __ldcg(gh + q);
    int b, pos;
    int R = row_regions(p, ng / p.G, b, pos);
    if (R < 0) R = 0;
    block_threshold(h, R, p.top_k, s_w, s_tmp);  // ends with a __syncthreads
    if (tid == 0) {
        p.arrive1[ng] = 0;
        p.cand_count[ng] = 0;
        st_release_u32(p.thr + ng, ((gen + 1u) << 12) | (uint32_t)*s_tmp);
    }
    // every share has been added, and nothing reads the histogram again in this launch:
    // it is cleared for the next one after the threshold is out
#pragma unroll
    for (int q = 0; q < kBinsPerThread / 4; ++q) gh[q] = make_uint4(0, 0, 0, 0);
}

// Waits (thread 0) for the threshold of (row, group) ng published after generation
// gen; -1 when the wait gives up (after p.wait_polls polls).
__device__ int wait_threshold(const ScoreParams& p, int ng, uint32_t gen) {
    for (uint32_t it = 0; it < p.wait_polls; ++it) {
        const uint32_t v = ld_relaxed_u32(p.thr + ng);
        if ((v >> 12) != gen) {
            fence_acquire_gpu();
            return (int)(v & (kHistBins - 1));
        }
    }
    return -1;
}

// The selection of (row, group) ng from every score of its row, by one block (the
// candidate list overflowed): the block top-k.  Out of line: rarely run.
__device__ __noinline__ void select_all_scores(const ScoreParams& p, int ng, uint8_t* ring) {
    const int n = ng / p.G;
    int b, pos;
    int R = row_regions(p, n, b, pos);
    if (R < 0) R = 0;
    int P2 = 32;
    while (P2 < p.top_k) P2 <<= 1;
    uint64_t* s_sel = reinterpret_cast<uint64_t*>(ring);
    TopkSmem& ts = *reinterpret_cast<TopkSmem*>(ring + kMaxTopK * 8);
    uint64_t* s_aux = reinterpret_cast<uint64_t*>(ring + kMaxTopK * 8 + ((sizeof(TopkSmem) + 15) & ~(size_t)15));
    const int take = block_topk<kSplitThreads>(ScoreKeys{p.scores + (int64_t)ng * p.r_cap}, R, p.top_k, P2, s_sel,
                                               s_aux, ts);
    write_selection<kSplitThreads>(p, n, ng - n * p.G, take, s_sel);
}

// Ranks of the candidates of (row, group) ng, after every candidate is written: block
// `sub` of the nb blocks covering it takes chunks of 32 candidates (one per lane), and
// each warp counts the smaller keys in its share of the list; a candidate ranked below
// K is written at its rank.  Block 0 writes the padding and the count, or, when the
// list overflowed, selects from every score of the row.
__device__ void rank_segment(const ScoreParams& p, int ng, int sub, int nb, uint8_t* ring, uint32_t* s_w) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = p.top_k;
    // the count and the first slots of the list are requested at once
    const uint64_t* cl = p.cand + (int64_t)ng * kCandCap;
    constexpr int kSpec = kCandCap / kSplitThreads;  // slots per thread read before the count is known
    uint64_t cv[kSpec];
    const bool works = sub * 32 < kCandCap;
#pragma unroll
    for (int u = 0; u < kSpec; ++u) cv[u] = works ? __ldcg(cl + u * kSplitThreads + tid) : 0ull;
    const int C = (int)__ldcg(p.cand_count + ng);
    int32_t* ids = p.sel_ids + (int64_t)ng * K;
    float* ss = p.sel_scores ? p.sel_scores + (int64_t)ng * K : nullptr;
    if (C > kCandCap) {
        if (sub == 0) select_all_scores(p, ng, ring);
        return;
    }
    if (sub * 32 < C) {
        uint64_t* s_keys = reinterpret_cast<uint64_t*>(ring);
#pragma unroll
        for (int u = 0; u < kSpec; ++u)
            if (u * kSplitThreads + tid < C) s_keys[u * kSplitThreads + tid] = cv[u];
        for (int i = kSpec * kSplitThreads + tid; i < C; i += kSplitThreads) s_keys[i] = __ldcg(cl + i);
        __syncthreads();
        const int j0 = (int)((int64_t)C * warp / kSplitWarps), j1 = (int)((int64_t)C * (warp + 1) / kSplitWarps);
        for (int c0 = sub * 32; c0 < C; c0 += nb * 32) {
            const int idx = c0 + lane;
            const uint64_t key = idx < C ? s_keys[idx] : ~0ull;
            uint32_t less = 0;
            for (int j = j0; j < j1; ++j) less += s_keys[j] < key ? 1u : 0u;
            s_w[warp * 32 + lane] = less;
            __syncthreads();
            if (warp == 0 && idx < C) {
                uint32_t rank = 0;
#pragma unroll
                for (int w = 0; w < kSplitWarps; ++w) rank += s_w[w * 32 + lane];
                if (rank < (uint32_t)K) {
                    ids[rank] = (int32_t)(uint32_t)(key & 0xffffffffu) + p.region_lo;
                    if (ss) ss[rank] = score_of_desc_key((uint32_t)(key >> 32));
                }
            }
            __syncthreads();
        }
    }
    if (sub == 0) {
        const int take = C < K ? C : K;
        for (int i = take + tid; i < K; i += kSplitThreads) {
            ids[i] = -1;
            if (ss) ss[i] = -INFINITY;
        }
        if (tid == 0) p.sel_count[ng] = take;
    }
}

constexpr int kKeep = 4096;                      // scores of a block's range kept on chip
constexpr int kMaxShareSegs = 32;                // (row, group)s one block's share may cover
constexpr int kKeepPer = kKeep / kSplitThreads;
constexpr int kRankWarps = kSplitThreads / 32;

// Split path, one persistent launch (every block resident):
//  1. score an even share of the (row, group, region) space and add shared-memory
//     histograms of the keys to the global histograms; the last block of each
//     (row, group) to add its share publishes the bin holding the (row, group)'s K-th key;
//  2. copy every key of the share in or below that bin into the (row, group)'s
//     candidate list;
//  3. once all blocks of the (row, group) have done so, they split its candidates and
//     write each one ranked below K at its rank (rank_segment).
// Histograms and counters are left zero and the synchronisation words carry
// generations, so nothing needs clearing between calls.  A share covers at most
// kMaxShareSegs (row, group)s (the host launches row batches).
template <int HPG>
__global__ void __maxnreg__(kSplitMaxRegs) score_select_kernel(const __grid_constant__ CUtensorMap smap,
                                                                        ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = align_smem(smem_raw, 1024);
    __shared__ uint32_t s_hist[kHistBins];
    __shared__ __align__(16) QBuf<HPG> s_qb[2];
    __shared__ float s_keep[kKeep];
    __shared__ __align__(8) uint64_t s_bar[kScoreStages];
    __shared__ uint32_t s_w[kRankWarps * 32];
    __shared__ int s_thr[2], s_R[2];
    __shared__ uint32_t s_base[2];
    const int tid = threadIdx.x;
    const int qd = tid & 3, slot = tid >> 2;

    // set-up that touches no input: barriers, the histogram, the tensor map
    if (tid == 0) {
        for (int st = 0; st < kScoreStages; ++st) mbar_init(&s_bar[st], 1);
        fence_mbar_init();
        if constexpr (HPG == 4) prefetch_tmap(&smap);
    }
    for (int i = tid; i < kHistBins; i += kSplitThreads) s_hist[i] = 0;
    // the tensor cores' query tiles (rows 4-15 stay zero) and accumulators (HPG == 4)
    uint8_t* qe_tiles = ring + kScoreStages * kTileBytes;
    __shared__ __align__(8) uint64_t s_dbar2[2];
    __shared__ uint32_t s_tmem;
    if constexpr (HPG == 4) {
        for (int i = tid; i < (int)(2 * kQeBytes / 16); i += kSplitThreads)
            reinterpret_cast<uint4*>(qe_tiles)[i] = make_uint4(0, 0, 0, 0);
        if (tid == 0) {
            mbar_init(&s_dbar2[0], 1);
            mbar_init(&s_dbar2[1], 1);
        }
        if (tid < 32) tc::alloc(&s_tmem, kScoreTmemCols);
        tc::fence_before_sync();
    }
    STEP5_STAMP(1, 0);
    __syncthreads();
    // With overlap_prologue the launch before this one writes none of the query,
    // weight, row and rope inputs, so they are read before waiting for it (only the
    // summaries are, and thread 0 waits before the first copy that may read them);
    // otherwise every read waits.
    if (!p.overlap_prologue) pdl_wait();
    STEP5_STAMP(1, 1);
    // this block's even share of the flattened (row, group, region) space
    const int NG = p.N * p.G;
    const int64_t total = (int64_t)NG * p.r_cap;
    const int64_t xbeg = total * blockIdx.x / gridDim.x;
    const int64_t xend = total * (blockIdx.x + 1) / gridDim.x;
    const int ngA = (int)(xbeg / p.r_cap);
    const int ngB = (int)((xend - 1) / p.r_cap);
    // the share's scores stay on chip when it is short and spans at most two (row, group)s
    const bool keep_all = xend - xbeg <= kKeep && ngB <= ngA + 1;
    Walk wk = walk_start(p, xbeg, xend);
    // The queries of the first two (row, group)s of the range are requested together
    // with their rows' positions, their cos/sin before the first tiles, so these small
    // reads do not queue behind every block's tile copies; later (row, group)s (ranges
    // over short rows) are staged when reached.
    int staged0 = ngA;  // (row, group) held by query buffer 0 / 1 (-1: none)
    int staged1 = ngB > ngA ? ngA + 1 : -1;
    QRaw<HPG> r0, r1;
    QRope<HPG> o0, o1;
    // Thread 0 walks the share; the descriptors of the tiles in the two stages live in
    // shared memory (the other threads only read them).
    __shared__ Tile s_tile[kScoreStages];
    // the deferred summary ranges of up to kSplitThreads sequences, staged with the
    // first reads so that the first copies wait on one round trip only
    __shared__ int2 s_def[kSplitThreads];
    const bool def_staged = p.defer_begin != nullptr && p.B <= kSplitThreads;
    {
        const int n0 = staged0 / p.G;
        const int n1 = staged1 < 0 ? n0 : staged1 / p.G;
        load_query_raw<HPG>(p, n0, staged0 - n0 * p.G, r0);
        if (staged1 >= 0) load_query_raw<HPG>(p, n1, staged1 - n1 * p.G, r1);
        if (def_staged && tid < p.B) s_def[tid] = make_int2(__ldg(p.defer_begin + tid), __ldg(p.defer_end + tid));
        if (tid == 0) {
            // a short first tile, so that every SM starts scoring before the first
            // requests of all SMs have drained
            s_tile[0] = next_tile(p, wk, kBoxRows);
            for (int k = 1; k < kScoreStages; ++k) s_tile[k] = next_tile(p, wk);
        }
        const int pos0 = row_pos_or0(p, n0);
        const int pos1 = n1 == n0 ? pos0 : row_pos_or0(p, n1);
        load_rope<HPG>(p, pos0, o0);
        if (staged1 >= 0) load_rope<HPG>(p, pos1, o1);
    }
    __syncthreads();  // s_tile, s_def (and the TMEM base)
    if constexpr (HPG == 4) tc::fence_after_sync();
    const uint32_t tmem = HPG == 4 ? s_tmem : 0u;
    uint8_t* const qe0 = HPG == 4 ? qe_tiles : nullptr;
    uint8_t* const qe1 = HPG == 4 ? qe_tiles + kQeBytes : nullptr;
    // thread 0 (the only one that reads summaries, through the copies it issues) waits
    // for the launch before once a tile may hold summaries that launch writes
    bool waited = !p.overlap_prologue;
    auto issue = [&](const Tile& x, int st) {
        if (tid == 0) {
            if (!waited) {
                bool clear = p.defer_begin != nullptr;
                if (clear) {
                    const int2 d = def_staged ? s_def[x.b]
                                              : make_int2(__ldg(p.defer_begin + x.b), __ldg(p.defer_end + x.b));
                    clear = x.c1 <= d.x || d.y <= x.c0;
                }
                if (!clear) {
                    pdl_wait();
                    waited = true;
                }
            }
            if constexpr (HPG == 4) {
                // the boxes that hold the tile's regions (rows past the tensor end arrive
                // as zeros)
                const int y = (int)(((int64_t)x.b * p.G + x.g) * p.r_cap + x.c0);
                const int nbox = (x.c1 - x.c0 + kBoxRows - 1) / kBoxRows;
                mbar_arrive_expect_tx(&s_bar[st], (uint32_t)(nbox * kBoxRows * 64));
                for (int k = 0; k < nbox; ++k)
                    tma_load_2d(ring + st * kTileBytes + k * kBoxRows * 64, &smap, &s_bar[st], 0, y + k * kBoxRows);
            } else {
                const uint32_t bytes = (uint32_t)(x.c1 - x.c0) * 64u;
                mbar_arrive_expect_tx(&s_bar[st], bytes);
                bulk_load(ring + st * kTileBytes, p.summ + (((int64_t)x.b * p.G + x.g) * p.r_cap + x.c0) * 64,
                          bytes, &s_bar[st]);
            }
        }
    };
    if (tid == 0) {
        for (int k = 0; k < kScoreStages; ++k)
            if (s_tile[k].valid) issue(s_tile[k], k);
    }
    finish_query<HPG>(p, r0, o0, s_qb[0], qe0);
    if (staged1 >= 0) finish_query<HPG>(p, r1, o1, s_qb[1], qe1);
    __syncthreads();  // staged queries visible
    STEP5_STAMP(1, 2);

    int seg_ng = -1, qbuf = 0;
    QFrag<HPG> f;
    float w4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    // makes (row, group) x.ng the current segment, staging its query if needed
    auto enter = [&](const Tile& x) {
        int bsel = staged0 == x.ng ? 0 : staged1 == x.ng ? 1 : -1;
        if (bsel < 0) {
            bsel = qbuf ^ 1;  // the buffer of the segment just finished is free
            QRaw<HPG> r;
            QRope<HPG> o;
            load_query_raw<HPG>(p, x.n, x.g, r);
            load_rope<HPG>(p, x.pos, o);
            finish_query<HPG>(p, r, o, s_qb[bsel], bsel ? qe1 : qe0);
            if (bsel) staged1 = x.ng; else staged0 = x.ng;
            __syncthreads();
        }
        qbuf = bsel;
        seg_ng = x.ng;
        if constexpr (HPG == 4) {
#pragma unroll
            for (int h = 0; h < 4; ++h) w4[h] = s_qb[bsel].w[h];
        } else {
            qfrag_from_smem<HPG>(s_qb[bsel], f);
        }
    };
    auto flush_hist = [&](int ng) {
        __syncthreads();
        uint32_t* gh = p.hist + (int64_t)ng * kHistBins;
        // each thread flushes its kBinsPerThread consecutive bins
#pragma unroll
        for (int i = 0; i < kHistBins / kSplitThreads; ++i) {
            const int bin = tid * (kHistBins / kSplitThreads) + i;
            const uint32_t c = s_hist[bin];
            if (c) atomicAdd(gh + bin, c);
        }
    };

    // ---------------- phase 1: scores and histograms
    uint32_t phases = 0;  // bit k: the phase stage k waits for
    int st = 0, ntile = 0;
    bool ok = true;
    uint32_t dphases = 0;  // bit b: the phase accumulator b waits for
    bool mma_fail = false;
    if constexpr (HPG == 4) {
        // Software pipeline over the tiles: tile t's products were issued in the previous
        // iteration; once they are done its stage is refilled at once (the epilogue reads
        // TMEM, not the stage), tile t + 1's products are issued into the other
        // accumulator, and only then tile t's epilogue runs.
        auto buffer_for = [&](const Tile& x, int busy) -> int {  // stages x's query if needed
            int bsel = staged0 == x.ng ? 0 : staged1 == x.ng ? 1 : -1;
            if (bsel < 0) {
                bsel = busy == 0 ? 1 : 0;  // not the buffer the tile in flight reads
                QRaw<HPG> r;
                QRope<HPG> o;
                load_query_raw<HPG>(p, x.n, x.g, r);
                load_rope<HPG>(p, x.pos, o);
                finish_query<HPG>(p, r, o, s_qb[bsel], bsel ? qe1 : qe0);
                if (bsel) staged1 = x.ng; else staged0 = x.ng;
                __syncthreads();
            }
            return bsel;
        };
        // waits (thread 0) for the copy of the tile in stage k, issues its products
        auto start_tile = [&](int k, const Tile& x, int buf, int acc) -> bool {
            bool got = true;
            if (tid == 0) {
                got = mbar_wait(&s_bar[k], (phases >> k) & 1u);
                if (got) tc_tile_issue(ring + k * kTileBytes, buf ? qe1 : qe0, x.c1 - x.c0, tmem + 128u * acc,
                                       &s_dbar2[acc]);
            }
            phases ^= 1u << k;
            return !__syncthreads_or(!got);
        };
        Tile cur = s_tile[0];
        int buf = -1, hist_ng = -1;
        if (cur.valid) {
            buf = buffer_for(cur, -1);
            if (!start_tile(0, cur, buf, 0)) ok = false;
        }
        for (int t = 0; ok && cur.valid; ++t) {
            if (ntile < 3) STEP5_STAMP(1, 3 + 2 * ntile);
            // tile t's products done: its stage takes the walk's next tile
            const int acc = t & 1;
            const bool got = mbar_wait(&s_dbar2[acc], (dphases >> acc) & 1u);
            dphases ^= 1u << acc;
            tc::fence_after_sync();
            if (tid == 0) {
                const Tile nx = next_tile(p, wk);
                s_tile[st] = nx;
                if (nx.valid) {
                    fence_proxy_async();
                    issue(nx, st);
                }
            }
            if (ntile < 3) STEP5_STAMP(1, 4 + 2 * ntile);
            ++ntile;
            // tile t + 1's products into the other accumulator (its last reader, tile t - 1's
            // epilogue, finished before the end of the previous iteration)
            const int nst = st + 1 == kScoreStages ? 0 : st + 1;
            const Tile nxt = s_tile[nst];
            int nbuf = -1;
            bool ok2 = true;
            if (nxt.valid) {
                nbuf = buffer_for(nxt, buf);
                ok2 = start_tile(nst, nxt, nbuf, acc ^ 1);
            }
            // tile t's epilogue (the shared histogram counts one (row, group) at a time)
            if (cur.ng != hist_ng) {
                if (hist_ng >= 0) {
                    flush_hist(hist_ng);
                    __syncthreads();  // every bin is flushed before it is cleared
                    for (int i = tid; i < kHistBins; i += kSplitThreads) s_hist[i] = 0;
                    __syncthreads();
                }
                hist_ng = cur.ng;
            }
            const int64_t x0 = (int64_t)cur.ng * p.r_cap + cur.c0;
            float* keep = keep_all ? s_keep + (int)(x0 - xbeg) : nullptr;
            tc_tile_epilogue(cur.c1 - cur.c0, tmem + 128u * acc, s_qb[buf].w, p.scores + x0, keep, s_hist);
            if (__syncthreads_or(!got || !ok2)) {
                mma_fail = true;
                ok = false;
                break;
            }
            cur = nxt;
            buf = nbuf;
            st = nst;
        }
        seg_ng = hist_ng;
    } else for (;;) {
        const Tile cur = s_tile[st];
        if (!cur.valid) break;
        if (cur.ng != seg_ng) {
            if (seg_ng >= 0) {
                flush_hist(seg_ng);
                __syncthreads();  // every bin is flushed before it is cleared
                for (int i = tid; i < kHistBins; i += kSplitThreads) s_hist[i] = 0;
            }
            enter(cur);
        }
        if (ntile < 3) STEP5_STAMP(1, 3 + 2 * ntile);
        // one thread waits for the tile; the barrier releases the others (they do not
        // spin on the issue slots the other block of the SM is computing with)
        bool got = true;
        if (tid == 0) got = mbar_wait(&s_bar[st], (phases >> st) & 1u);
        if (__syncthreads_or(!got)) {
            ok = false;
            break;
        }
        if (ntile < 3) STEP5_STAMP(1, 4 + 2 * ntile);
        ++ntile;
        phases ^= 1u << st;
        const int64_t x0 = (int64_t)cur.ng * p.r_cap + cur.c0;
        float* scores = p.scores + x0;
        float* keep = keep_all ? s_keep + (int)(x0 - xbeg) : nullptr;
        const int nreg = cur.c1 - cur.c0;
        {
            const uint4* tile = reinterpret_cast<const uint4*>(ring + st * kTileBytes);
            if (nreg == kTileRegions)
                score_tile<HPG, true>(f, tile, nreg, scores, keep, s_hist, qd, slot);
            else
                score_tile<HPG, false>(f, tile, nreg, scores, keep, s_hist, qd, slot);
        }
        // every thread is done with this stage (and the accumulators) before it is refilled
        if (__syncthreads_or(mma_fail)) {
            ok = false;
            break;
        }
        if (tid == 0) {
            const Tile nx = next_tile(p, wk);
            s_tile[st] = nx;
            if (nx.valid) {
                fence_proxy_async();
                issue(nx, st);
            }
        }
        st = st + 1 == kScoreStages ? 0 : st + 1;
    }
    if (!ok) {
        if (tid == 0) {
            raise_status(p.status, kDevTimeout);
            // give copies still in flight a bounded chance to land before the block exits
            for (int k = 0; k < kScoreStages; ++k)
                if (s_tile[k].valid) mbar_wait(&s_bar[k], (phases >> k) & 1u);
            if (HPG == 4 && mma_fail) {  // the products in flight
                mbar_wait(&s_dbar2[0], dphases & 1u);
                mbar_wait(&s_dbar2[1], (dphases >> 1) & 1u);
            }
        }
        if constexpr (HPG == 4) {
            tc::fence_before_sync();
            __syncthreads();
            if (tid < 32) tc::dealloc(tmem, kScoreTmemCols);
        }
        return;
    }
    if constexpr (HPG == 4) {  // the accumulators are not needed past the scoring
        tc::fence_before_sync();
        __syncthreads();
        if (tid < 32) tc::dealloc(tmem, kScoreTmemCols);
    }
    STEP5_STAMP(1, 9);
    if (seg_ng >= 0) flush_hist(seg_ng);
    STEP5_STAMP(1, 10);
    // Every block that covers part of a (row, group) arrives once its histogram share is
    // in; the last one computes and publishes the (row, group)'s threshold bin.  The
    // threshold word's generation is read before arriving.
    __shared__ int s_last;
    __shared__ int s_tmp;
    __shared__ uint32_t s_gen1[kMaxShareSegs], s_gen2[kMaxShareSegs];
    auto seg_first = [&](int ng) { return block_of((int64_t)ng * p.r_cap, total, gridDim.x); };
    auto seg_blocks = [&](int ng) { return block_of((int64_t)(ng + 1) * p.r_cap - 1, total, gridDim.x) - seg_first(ng) + 1; };
    for (int ng = ngA; ng <= ngB; ++ng) {
        __syncthreads();  // the block's histogram additions come before its arrival
        if (tid == 0) {
            const uint32_t gen = ld_acquire_u32(p.thr + ng) >> 12;
            s_gen1[ng - ngA] = gen;
            s_last = arrive_last(p.arrive1 + ng, (uint32_t)seg_blocks(ng));
        }
        __syncthreads();
        if (s_last) publish_threshold(p, ng, s_gen1[ng - ngA], s_w, &s_tmp);
    }
    STEP5_STAMP(1, 11);
    pdl_launch_dependents();

    // ---------------- phase 2: candidates of this block's share
    if (keep_all) {
        // the thresholds (and R) of the share's one or two (row, group)s
        if (tid == 0) {
            int b, pos;
            const int RA = row_regions(p, ngA / p.G, b, pos);
            const int RB = row_regions(p, ngB / p.G, b, pos);
            s_R[0] = RA < 0 ? 0 : RA;
            s_R[1] = RB < 0 ? 0 : RB;
            s_thr[0] = wait_threshold(p, ngA, s_gen1[0]);
            s_thr[1] = ngB != ngA ? wait_threshold(p, ngB, s_gen1[1]) : s_thr[0];
        }
        if (__syncthreads_or(tid == 0 && (s_thr[0] < 0 || s_thr[1] < 0))) {
            if (tid == 0) raise_status(p.status, kDevTimeout);
            return;
        }
        const int64_t bstart = (int64_t)(ngA + 1) * p.r_cap;  // first position of the second
        const int len = (int)(xend - xbeg);
        uint64_t keys[kKeepPer];
        uint32_t sel = 0, inb = 0, cnt = 0;  // bit u: key u selected / in the second; counts
#pragma unroll
        for (int u = 0; u < kKeepPer; ++u) {
            const int i = tid + u * kSplitThreads;
            keys[u] = 0;
            if (i < len) {
                const int64_t x = xbeg + i;
                const int second = x >= bstart;
                const int r = (int)(x - (second ? bstart : (int64_t)ngA * p.r_cap));
                if (r < s_R[second]) {
                    const uint32_t k = desc_key(s_keep[i]);
                    if ((int)(k >> (32 - kHistBits)) <= s_thr[second]) {
                        keys[u] = ((uint64_t)k << 32) | (uint32_t)r;
                        sel |= 1u << u;
                        inb |= (uint32_t)second << u;
                        cnt += second ? 0x10000u : 1u;
                    }
                }
            }
        }
        uint32_t tot = 0;
        uint32_t off = block_excl_scan(cnt, s_w, &tot);
        if (tid == 0) {
            const uint32_t ta = tot & 0xffffu, tb = tot >> 16;
            s_base[0] = ta ? atomicAdd(p.cand_count + ngA, ta) : 0u;
            s_base[1] = tb ? atomicAdd(p.cand_count + ngB, tb) : 0u;
        }
        __syncthreads();
        uint32_t sa = s_base[0] + (off & 0xffffu), sb = s_base[1] + (off >> 16);
        uint64_t* ca = p.cand + (int64_t)ngA * kCandCap;
        uint64_t* cb = p.cand + (int64_t)ngB * kCandCap;
#pragma unroll
        for (int u = 0; u < kKeepPer; ++u) {
            if (sel >> u & 1u) {
                if (inb >> u & 1u) {
                    if (sb < (uint32_t)kCandCap) cb[sb] = keys[u];
                    ++sb;
                } else {
                    if (sa < (uint32_t)kCandCap) ca[sa] = keys[u];
                    ++sa;
                }
            }
        }
    } else {
        // long shares: batches of up to kKeep regions of one (row, group), scores re-read
        Walk fw = walk_start(p, xbeg, xend);
        int thr_ng = -1;
        for (;;) {
            // the batch: consecutive tiles of one (row, group), at most kKeep regions
            Tile t = next_tile(p, fw);
            if (!t.valid) break;
            int c1 = t.c1;
            while (c1 - t.c0 + kTileRegions <= kKeep && fw.left > 0 && fw.ng == t.ng && fw.r < fw.cR) {
                const Tile u = next_tile(p, fw);
                c1 = u.c1;
            }
            if (t.ng != thr_ng) {
                if (tid == 0) s_thr[0] = wait_threshold(p, t.ng, s_gen1[t.ng - ngA]);
                if (__syncthreads_or(tid == 0 && s_thr[0] < 0)) {
                    if (tid == 0) raise_status(p.status, kDevTimeout);
                    return;
                }
                thr_ng = t.ng;
            }
            const float* sc = p.scores + (int64_t)t.ng * p.r_cap;
            uint64_t keys[kKeepPer];
            uint32_t sel = 0, cnt = 0;
            const int T = s_thr[0];
#pragma unroll
            for (int u = 0; u < kKeepPer; ++u) {
                const int r = t.c0 + tid + u * kSplitThreads;
                keys[u] = 0;
                if (r < c1) {
                    const uint32_t k = desc_key(__ldcg(sc + r));
                    if ((int)(k >> (32 - kHistBits)) <= T) {
                        keys[u] = ((uint64_t)k << 32) | (uint32_t)r;
                        sel |= 1u << u;
                        ++cnt;
                    }
                }
            }
            uint32_t tot = 0;
            uint32_t off = block_excl_scan(cnt, s_w, &tot);
            if (tid == 0) s_base[0] = tot ? atomicAdd(p.cand_count + t.ng, tot) : 0u;
            __syncthreads();
            uint32_t slot2 = s_base[0] + off;
            uint64_t* cl = p.cand + (int64_t)t.ng * kCandCap;
#pragma unroll
            for (int u = 0; u < kKeepPer; ++u) {
                if (sel >> u & 1u) {
                    if (slot2 < (uint32_t)kCandCap) cl[slot2] = keys[u];
                    ++slot2;
                }
            }
            __syncthreads();  // s_thr / s_base reused by the next batch
        }
    }
    STEP5_STAMP(1, 12);
    // ---------------- phase 3: ranks, once every block of the (row, group) has written
    // its candidates (arrive at every (row, group) of the share first, then wait)
    for (int ng = ngA; ng <= ngB; ++ng) {
        __syncthreads();  // the block's candidate writes come before its arrival
        if (tid == 0) s_gen2[ng - ngA] = arrive_gen(p.bar2 + ng, (uint32_t)seg_blocks(ng));
    }
    for (int ng = ngA; ng <= ngB; ++ng) {
        __syncthreads();
        if (__syncthreads_or(tid == 0 && !wait_gen(p.bar2 + ng, s_gen2[ng - ngA], p.wait_polls))) {
            if (tid == 0) raise_status(p.status, kDevTimeout);
            return;
        }
        STEP5_STAMP(1, 13);
        rank_segment(p, ng, blockIdx.x - seg_first(ng), seg_blocks(ng), ring, s_w);
    }
    STEP5_STAMP(1, 14);
}

int pow2_at_least(int x) {
    int p2 = 32;
    while (p2 < x) p2 <<= 1;
    return p2;
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

template <int HPG, bool FROM_SCORES = false>
cudaError_t fused_for(const ScoreParams& p, cudaStream_t stream, bool pdl) {
    const int P2 = pow2_at_least(p.top_k);
    const int key_cap = (p.r_cap < kFusedMaxRegions ? p.r_cap : kFusedMaxRegions);
    const size_t smem = (size_t)(P2 + sel_aux_slots(P2)) * 8 + (size_t)((key_cap + 3) & ~3) * 4 + HPG * 64 * 4;
    auto kern = score_fused_kernel<HPG, FROM_SCORES>;
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
    // one persistent launch with every block resident: one block per SM, at most one per
    // tile
    static std::atomic<uint64_t> ready{0};
    cudaError_t e0 = once_per_device(ready, [] {
        cudaError_t e = cudaFuncSetAttribute(score_select_kernel<HPG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kScoreSmem);
        if (e != cudaSuccess) return e;
        int b = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, score_select_kernel<HPG>, kSplitThreads, kScoreSmem);
        if (e != cudaSuccess) return e;
        return b < 1 ? cudaErrorInvalidConfiguration : cudaSuccess;
    });
    if (e0 != cudaSuccess) return e0;
    const int per_sm = 1;
    // rows in batches small enough that a block's share covers at most kMaxShareSegs
    // (row, group)s
    const int64_t full_grid = (int64_t)per_sm * p_in.num_sms;
    int64_t rows_per = (full_grid * (kMaxShareSegs - 2)) / p_in.G;
    if (rows_per < 1) rows_per = 1;
    for (int n0 = 0; n0 < p_in.N; n0 += (int)rows_per) {
        ScoreParams p = p_in;
        p.N = (int)((p_in.N - n0) < rows_per ? (p_in.N - n0) : rows_per);
        const int64_t g0 = (int64_t)n0 * p.G;  // first (row, group) of the batch
        p.idx_q = p_in.idx_q + (int64_t)n0 * p.idx_heads * 64;
        p.w = p_in.w + (int64_t)n0 * p.idx_heads;
        p.row_seq = p_in.row_seq + n0;
        p.row_pos = p_in.row_pos + n0;
        p.sel_ids = p_in.sel_ids + g0 * p.top_k;
        p.sel_count = p_in.sel_count + g0;
        p.sel_scores = p_in.sel_scores ? p_in.sel_scores + g0 * p.top_k : nullptr;
        p.scores = p_in.scores + g0 * p.r_cap;
        p.hist = p_in.hist + g0 * kHistBins;
        p.cand_count = p_in.cand_count + g0;
        p.cand = p_in.cand + g0 * kCandCap;
        p.arrive1 = p_in.arrive1 + g0;
        p.thr = p_in.thr + g0;
        p.bar2 = p_in.bar2 + g0;
        // at most one block per tile, but enough blocks that no share covers more than
        // kMaxShareSegs - 2 (row, group)s (short rows)
        const int64_t tiles = ((int64_t)p.N * p.G * p.r_cap + kTileRegions - 1) / kTileRegions;
        const int64_t need = ((int64_t)p.N * p.G + kMaxShareSegs - 3) / (kMaxShareSegs - 2);
        int64_t grid = tiles > need ? tiles : need;
        if (grid > full_grid) grid = full_grid;
        cudaError_t e = launch_map(score_select_kernel<HPG>, dim3((unsigned)grid), dim3(kSplitThreads), kScoreSmem,
                                   stream, pdl && n0 == 0, smap, p);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
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

cudaError_t launch_select_scores(const ScoreParams& p, cudaStream_t stream, bool pdl) {
    return fused_for<1, true>(p, stream, pdl);  // (HPG is not used when selecting from scores)
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
