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
    float w[HPG];
};

// e4m3(bf16(NEOX(q))) for the group's HPG heads into shared memory, then each thread
// keeps the 16 dims it multiplies (qd = lane & 3).
template <int HPG>
__device__ void load_qfrag(const ScoreParams& p, int n, int g, int pos, float* s_q, QFrag<HPG>& f) {
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
    const int qd = threadIdx.x & 3;
#pragma unroll
    for (int h = 0; h < HPG; ++h) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            f.q[h][i] = make_float2(s_q[h * 64 + 16 * qd + 2 * i], s_q[h * 64 + 16 * qd + 2 * i + 1]);
        f.w[h] = p.w[(int64_t)n * p.idx_heads + (int64_t)g * HPG + h];
    }
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

// ----------------------------------------------------------------- block top-k

struct TopkSmem {
    uint32_t hist[256];
    uint32_t count;
    uint32_t v, before, inbin;
};

// Selects the K smallest of cnt unique 64-bit keys (all of them if cnt <= K), writes
// them sorted ascending to s_sel[0..P2) (padded with ~0), returns min(cnt, K).
// get(i) returns key i.  Must be called by all NT threads of the block.
template <int NT, class Get>
__device__ int block_topk(Get get, int cnt, int K, int P2, uint64_t* s_sel, TopkSmem& ts) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint64_t bound = ~0ull;
    if (cnt > K) {
        uint64_t prefix = 0;
        int need = K;
        for (int shift = 56; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += NT) ts.hist[i] = 0;
            __syncthreads();
            const uint64_t mask = (shift == 56) ? 0ull : (~0ull << (shift + 8));
            for (int base = 0; base < cnt; base += NT) {
                const int i = base + tid;
                bool act = false;
                uint32_t bin = 0;
                if (i < cnt) {
                    const uint64_t k = get(i);
                    if ((k & mask) == prefix) {
                        act = true;
                        bin = (uint32_t)(k >> shift) & 255u;
                    }
                }
                const uint32_t am = __ballot_sync(0xffffffffu, act);
                if (act) {
                    const uint32_t peers = __match_any_sync(am, bin);
                    if (lane == __ffs(peers) - 1) atomicAdd(&ts.hist[bin], (uint32_t)__popc(peers));
                }
            }
            __syncthreads();
            if (warp == 0) {
                uint32_t loc[8];
                uint32_t sum = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    loc[k] = ts.hist[8 * lane + k];
                    sum += loc[k];
                }
                uint32_t incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                const uint32_t excl = incl - sum;
                if (excl < (uint32_t)need && (uint32_t)need <= incl) {
                    uint32_t c = excl;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        if (c + loc[k] >= (uint32_t)need) {
                            ts.v = 8 * lane + k;
                            ts.before = c;
                            ts.inbin = loc[k];
                            break;
                        }
                        c += loc[k];
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
    for (int k = 2; k <= P2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < P2; i += NT) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const uint64_t a = s_sel[i], b = s_sel[ixj];
                    const bool asc = (i & k) == 0;
                    if ((a > b) == asc) {
                        s_sel[i] = b;
                        s_sel[ixj] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    return cnt < K ? cnt : K;
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
    int b, pos;
    int R = row_regions(p, n, b, pos);
    if (R < 0 || R > key_cap) {
        if (threadIdx.x == 0) raise_status(p.status, kDevRange);
        R = 0;
        b = 0;
        pos = 0;
    }
    QFrag<HPG> f;
    load_qfrag<HPG>(p, n, g, pos, s_q, f);

    const int qd = threadIdx.x & 3;
    const int slot = threadIdx.x >> 2;  // 64 regions per pass
    const uint4* base = reinterpret_cast<const uint4*>(p.summ + ((int64_t)b * p.G + g) * p.r_cap * 64);
    float* exp_scores = p.scores ? p.scores + ((int64_t)n * p.G + g) * p.r_cap : nullptr;
    constexpr int U = 4;
    for (int r0 = 0; r0 < R; r0 += 64 * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = r0 + u * 64 + slot;
            v[u] = (r < R) ? __ldg(base + (int64_t)r * 4 + qd) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = r0 + u * 64 + slot;
            const float sc = score_from_vec<HPG>(f, v[u]);
            if (qd == 0 && r < R) {
                s_key[r] = desc_key(sc);
                if (exp_scores) exp_scores[r] = sc;
            }
        }
    }
    pdl_launch_dependents();
    __syncthreads();
    const int take = block_topk<kFusedThreads>(SmemKeys{s_key}, R, p.top_k, P2, s_sel, ts);
    write_selection<kFusedThreads>(p, n, g, take, s_sel);
}

// ----------------------------------------------------------------- split path

constexpr int kSplitThreads = 256;
constexpr int kSplitRegions = 512;  // regions scored by one block of the split path

template <int HPG>
__global__ void __launch_bounds__(kSplitThreads, 2) score_hist_kernel(ScoreParams p) {
    __shared__ uint32_t s_hist[kHistBins];
    __shared__ float s_q[HPG * 64];
    const int g = blockIdx.y, n = blockIdx.z;
    pdl_wait();
    int b, pos;
    const int R = row_regions(p, n, b, pos);
    if (R < 0) {
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_status(p.status, kDevRange);
        return;
    }
    const int c0 = blockIdx.x * kSplitRegions;
    const int c1 = min(R, c0 + kSplitRegions);
    if (c0 >= c1) return;
    // the block's summaries are requested before anything else (they do not depend on
    // the query): 8 regions of 16 bytes per thread in flight
    const int qd = threadIdx.x & 3;
    const int slot = threadIdx.x >> 2;
    const uint4* base = reinterpret_cast<const uint4*>(p.summ + ((int64_t)b * p.G + g) * p.r_cap * 64);
    constexpr int U = kSplitRegions / 64;
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int r = c0 + u * 64 + slot;
        v[u] = (r < c1) ? __ldg(base + (int64_t)r * 4 + qd) : make_uint4(0, 0, 0, 0);
    }
    for (int i = threadIdx.x; i < kHistBins; i += kSplitThreads) s_hist[i] = 0;
    QFrag<HPG> f;
    load_qfrag<HPG>(p, n, g, pos, s_q, f);  // has a __syncthreads

    float* scores = p.scores + ((int64_t)n * p.G + g) * p.r_cap;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int r = c0 + u * 64 + slot;
        const float sc = score_from_vec<HPG>(f, v[u]);
        if (qd == 0 && r < c1) {
            scores[r] = sc;
            atomicAdd(&s_hist[desc_key(sc) >> (32 - kHistBits)], 1u);
        }
    }
    __syncthreads();
    uint32_t* gh = p.hist + ((int64_t)n * p.G + g) * kHistBins;
    for (int i = threadIdx.x; i < kHistBins; i += kSplitThreads) {
        const uint32_t c = s_hist[i];
        if (c) atomicAdd(gh + i, c);
    }
    pdl_launch_dependents();
}

// Bin holding the K-th smallest key of (row, group), from the global histogram; all
// bins when the row has at most K regions.
__device__ int threshold_bin(const uint32_t* gh, int R, int K, int* s_part, int* s_out) {
    constexpr int per = kHistBins / kSplitThreads;  // 16
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (R <= K) return kHistBins - 1;
    int loc[per];
    int sum = 0;
#pragma unroll
    for (int k = 0; k < per; ++k) {
        loc[k] = (int)gh[tid * per + k];
        sum += loc[k];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_part[warp] = incl;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += s_part[w];
    incl += wbase;
    const int excl = incl - sum;
    if (excl < K && K <= incl) {
        int c = excl;
        for (int k = 0; k < per; ++k) {
            c += loc[k];
            if (c >= K) {
                *s_out = tid * per + k;
                break;
            }
        }
    }
    __syncthreads();
    return *s_out;
}

__global__ void __launch_bounds__(kSplitThreads) filter_kernel(ScoreParams p) {
    __shared__ int s_part[kSplitThreads / 32];
    __shared__ int s_bin;
    const int g = blockIdx.y, n = blockIdx.z;
    pdl_wait();
    int b, pos;
    const int R = row_regions(p, n, b, pos);
    if (R < 0) return;
    const int c0 = blockIdx.x * p.regions_per_cta;
    const int c1 = min(R, c0 + p.regions_per_cta);
    if (c0 >= c1) return;
    const int64_t ng = (int64_t)n * p.G + g;
    const int b1 = threshold_bin(p.hist + ng * kHistBins, R, p.top_k, s_part, &s_bin);
    const float* scores = p.scores + ng * p.r_cap;
    uint64_t* cand = p.cand + ng * kCandCap;
    const int lane = threadIdx.x & 31;
    for (int r0 = c0; r0 < c1; r0 += kSplitThreads) {
        const int r = r0 + threadIdx.x;
        bool act = false;
        uint32_t key = 0;
        if (r < c1) {
            key = desc_key(scores[r]);
            act = (int)(key >> (32 - kHistBits)) <= b1;
        }
        const uint32_t am = __ballot_sync(0xffffffffu, act);
        uint32_t slot = 0;
        if (lane == 0 && am) slot = atomicAdd(p.cand_count + ng, (uint32_t)__popc(am));
        slot = __shfl_sync(0xffffffffu, slot, 0);
        if (act) {
            const uint32_t idx = slot + __popc(am & ((1u << lane) - 1u));
            if (idx < (uint32_t)kCandCap) cand[idx] = ((uint64_t)key << 32) | (uint32_t)r;
        }
    }
    pdl_launch_dependents();
}

constexpr int kFinalThreads = 512;

__global__ void __launch_bounds__(kFinalThreads) final_select_kernel(ScoreParams p, int P2, int /*unused*/) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint64_t* s_sel = reinterpret_cast<uint64_t*>(smem);
    uint64_t* s_cand = s_sel + P2;  // kCandCap
    __shared__ TopkSmem ts;
    const int g = blockIdx.x, n = blockIdx.y;
    pdl_wait();
    int b, pos;
    int R = row_regions(p, n, b, pos);
    if (R < 0) R = 0;
    const int64_t ng = (int64_t)n * p.G + g;
    const int c = (int)p.cand_count[ng];
    int take;
    if (c <= kCandCap) {
        const uint64_t* cand = p.cand + ng * kCandCap;
        for (int i = threadIdx.x; i < c; i += kFinalThreads) s_cand[i] = __ldcg(cand + i);
        __syncthreads();
        take = block_topk<kFinalThreads>(CandKeys{s_cand}, c, p.top_k, P2, s_sel, ts);
    } else {
        take = block_topk<kFinalThreads>(ScoreKeys{p.scores + ng * p.r_cap}, R, p.top_k, P2, s_sel, ts);
    }
    pdl_launch_dependents();
    write_selection<kFinalThreads>(p, n, g, take, s_sel);
    // leave the histogram and the candidate counter zero for the next call
    __syncthreads();
    uint32_t* gh = p.hist + ng * kHistBins;
    for (int i = threadIdx.x; i < kHistBins; i += kFinalThreads) gh[i] = 0;
    if (threadIdx.x == 0) p.cand_count[ng] = 0;
}

int pow2_at_least(int x) {
    int p2 = 1;
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

template <int HPG>
cudaError_t split_for(const ScoreParams& p, cudaStream_t stream, bool pdl) {
    const int chunks = (p.r_cap + kSplitRegions - 1) / kSplitRegions;
    cudaError_t e = launch_ex(score_hist_kernel<HPG>, dim3(chunks, p.G, p.N), dim3(kSplitThreads), 0,
                              stream, pdl, p);
    if (e != cudaSuccess) return e;
    const int fchunks = (p.r_cap + p.regions_per_cta - 1) / p.regions_per_cta;
    e = launch_ex(filter_kernel, dim3(fchunks, p.G, p.N), dim3(kSplitThreads), 0, stream, true, p);
    if (e != cudaSuccess) return e;
    const int P2 = pow2_at_least(p.top_k);
    const size_t smem = (size_t)P2 * 8 + (size_t)kCandCap * 8;
    e = cudaFuncSetAttribute(final_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_ex2(final_select_kernel, dim3(p.G, p.N), dim3(kFinalThreads), smem, stream, true, p,
                      P2, 0);
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

cudaError_t launch_score_split(const ScoreParams& p, cudaStream_t stream, bool pdl) {
    switch (p.hpg) {
        case 1: return split_for<1>(p, stream, pdl);
        case 2: return split_for<2>(p, stream, pdl);
        case 4: return split_for<4>(p, stream, pdl);
        case 8: return split_for<8>(p, stream, pdl);
    }
    return cudaErrorInvalidValue;
}

}  // namespace step5
