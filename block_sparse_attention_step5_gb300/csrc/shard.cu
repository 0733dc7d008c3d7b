// shard.cu -- sequence-sharded decode: the merge of the shards' picks and the combine of
// their partial attention states.
//
// A row's regions (and tokens) split over S shards, each holding its part of the
// summaries and caches (on one GPU each, or one after another on one GPU): every shard
// picks its own top K with step5_index_score_topk_shard (its picks carry the row's
// region ids and their scores); the row's top K by (-score, id) is the K smallest keys
// of the union of the shards' picks (exactly the pick over all regions: a region in the
// row's top K is in its own shard's top K).  Attention then runs per shard over the
// picks and the own region inside it (step5_sparse_attn_shard), each leaving a softmax
// state (m, l, o per query head), and the states combine into the output.
//
// Merge: up to 16 blocks per (row, KV group); each stages the S lists (each in key order)
// in shared memory, and every key's rank in the union is its place in its own list plus
// a binary search in each other list; a key ranked below K is written at its rank.
// Combine: one warp per (row, query head), lanes over 4 output dims each.
#include "kernels.cuh"

namespace step5 {

namespace {

constexpr int kMergeThreads = 512;

// Number of keys below key in a list of n keys in ascending order (n >= 1, top = the
// largest power of two <= n): a branch-free binary search.
__device__ __forceinline__ int count_below(const uint64_t* lst, int n, int top, uint64_t key) {
    int at = 0;
    for (int step = top; step > 0; step >>= 1)
        if (at + step <= n && lst[at + step - 1] < key) at += step;
    return at;
}

// Grid (splits, NG): every block of a (row, group) stages all S lists and ranks the keys
// of its slice of them (keys j with j % splits == its index), so that a (row, group)'s
// ranking is spread over several SMs; block 0 writes the padding and the count.
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(MergeParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint64_t* keys = reinterpret_cast<uint64_t*>(smem_raw);  // [S][K], unused slots ~0
    __shared__ int s_cnt[kMaxShards];
    const int ng = blockIdx.y, tid = threadIdx.x;
    const int part = blockIdx.x, parts = gridDim.x;
    pdl_wait();
    pdl_launch_dependents();  // the attention after the merge may take its SMs now
    const int K = p.top_k, S = p.S;
    const int64_t NGK = (int64_t)p.NG * K;
    if (tid < S) {
        int c = p.counts[(int64_t)tid * p.NG + ng];
        if (c < 0 || c > K) {
            raise_status(p.status, kDevRange);
            c = c < 0 ? 0 : K;
        }
        s_cnt[tid] = c;
    }
    __syncthreads();
    for (int j = tid; j < S * K; j += kMergeThreads) {
        const int s = j / K, i = j - s * K;
        uint64_t key = ~0ull;  // above every real key (ids < 2^31)
        if (i < s_cnt[s]) {
            const int64_t at = s * NGK + (int64_t)ng * K + i;
            key = ((uint64_t)desc_key(__ldg(p.scores + at)) << 32) | (uint32_t)__ldg(p.ids + at);
        }
        keys[j] = key;
    }
    __syncthreads();
    int32_t* ids = p.sel_ids + (int64_t)ng * K;
    float* ss = p.sel_scores ? p.sel_scores + (int64_t)ng * K : nullptr;
    int total = 0;
    for (int s = 0; s < S; ++s) total += s_cnt[s];
    int top = 1;
    while (2 * top <= K) top *= 2;
    // a key's rank in the union: its place in its own list plus the keys below it in
    // each other list (keys are distinct: ids are)
    for (int j = part + parts * tid; j < S * K; j += parts * kMergeThreads) {
        const int s = j / K, i = j - s * K;
        if (i >= s_cnt[s]) continue;
        const uint64_t key = keys[j];
        int rank = i;
        for (int t = 0; t < S; ++t)
            if (t != s) rank += count_below(keys + (int64_t)t * K, K, top, key);
        if (rank < K) {
            ids[rank] = (int32_t)(uint32_t)(key & 0xffffffffu);
            if (ss) ss[rank] = score_of_desc_key((uint32_t)(key >> 32));
        }
    }
    if (part != 0) return;
    const int take = total < K ? total : K;
    for (int i = take + tid; i < K; i += kMergeThreads) {
        ids[i] = -1;
        if (ss) ss[i] = -INFINITY;
    }
    if (tid == 0) p.sel_count[ng] = take;
}

constexpr int kCombineThreads = 256;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t hrow = (int64_t)blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5);  // n * Hq + h
    if (hrow >= (int64_t)p.N * p.Hq) return;
    const int64_t stride = (int64_t)p.N * p.Hq * kAttnSlotFloats;  // one shard's states
    const float m = lane < p.S ? p.states[lane * stride + hrow * kAttnSlotFloats] : -INFINITY;
    const float l = lane < p.S ? p.states[lane * stride + hrow * kAttnSlotFloats + 1] : 0.0f;
    float M = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float base = M == -INFINITY ? 0.0f : M;
    const float w = exp2f(m - base);  // 0 for an empty shard and for lanes past S
    float L = l * w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    float O[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int s = 0; s < p.S; ++s) {  // shard order
        const float ws = __shfl_sync(0xffffffffu, w, s);
        const float* o = p.states + s * stride + hrow * kAttnSlotFloats + 2 + lane * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) O[i] += (ws != 0.0f ? o[i] * ws : 0.0f);
    }
    float gate = 1.0f;
    if (p.gate != nullptr) gate = 1.0f / (1.0f + expf(-bf16_to_f32(p.gate[hrow])));
    uint16_t y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = L > 0.0f ? f32_to_bf16_bits(O[i] / L * gate) : (uint16_t)0;
    *reinterpret_cast<uint2*>(p.out + hrow * 128 + lane * 4) =
        make_uint2((uint32_t)y[0] | ((uint32_t)y[1] << 16), (uint32_t)y[2] | ((uint32_t)y[3] << 16));
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, int num_sms, cudaStream_t stream, bool pdl) {
    static std::atomic<uint64_t> attr{0};
    cudaError_t e = once_per_device(attr, [] {
        return cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)((size_t)kMaxShardKeys * 8));
    });
    if (e != cudaSuccess) return e;
    // blocks per (row, group): as many as fill the SMs once, up to 16
    int parts = p.NG > 0 ? num_sms / p.NG : 1;
    parts = parts < 1 ? 1 : (parts > 16 ? 16 : parts);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)parts, (unsigned)p.NG, 1);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = (size_t)p.S * p.top_k * 8;
    cfg.stream = stream;
    cudaLaunchAttribute attr1[1];
    attr1[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr1[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr1;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, merge_kernel, p);
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    const int64_t rows = (int64_t)p.N * p.Hq;
    const int64_t blocks = (rows + kCombineThreads / 32 - 1) / (kCombineThreads / 32);
    combine_kernel<<<(unsigned)blocks, kCombineThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace step5
