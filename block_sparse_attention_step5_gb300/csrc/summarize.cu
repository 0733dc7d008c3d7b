// summarize.cu -- step (1): e4m3 summaries of completed regions.
//
// "Step-5-Preview on one 256 GB Mac" (TensorFold PR #903), CSA-indexer commit: every
// completed 8-token region is summarised, per KV group, as a per-dim softmax over z of
// the indexer k, rounded through bf16 to e4m3; the indexer k takes NEOX rotation on its
// first rope_dims dims from bf16 cos/sin.
//
// HBM-bound: 2 KB of k/z in, 64 B out per (region, group).  Two forms with the same
// arithmetic per dim (bit-identical results):
//  * few regions per sequence (a decode step): one thread per (region, dim), every load
//    of the region issued before any arithmetic, so the step waits one round trip;
//  * many regions (prefill chunks, set-up of a long context): a chunk of 16 regions'
//    z, k and cos/sin rows staged in shared memory by contiguous bulk copies.
// Rotated dims also read the partner dims (the other half of each NEOX pair).
#include "kernels.cuh"

namespace step5 {

namespace {

// One region (64 dims) per block: a 64-thread block at <= 48 registers a thread fits beside
// a scoring block (512 threads x 112 registers) on one SM, so in a decode step neither
// kernel waits for the SMs the other holds.
constexpr int kRegionsPerCta = 1;
constexpr int kSumThreads = kRegionsPerCta * 64;
// Above this many regions per sequence the bulk form runs (a decode step summarises one
// region per sequence; its latency is one dependent round trip in either form, and the
// one-dim-per-thread form issues every load of a region at once).
constexpr int kBulkMinSpan = 8;

__global__ void __maxnreg__(48) summarize_kernel(SummarizeParams p) {
    const int lr = threadIdx.x >> 6;   // region within the block
    const int d = threadIdx.x & 63;    // dim
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    STEP5_STAMP(0, 0);
    pdl_launch_dependents();  // the scoring kernel may start its prologue now
    const int rb = p.region_begin[b];
    const int re = p.region_end[b];
    const int r = rb + blockIdx.x * kRegionsPerCta + lr;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        // range checks of this sequence, once
        if (rb < 0 || re < rb || re > p.r_cap || (int64_t)re * 8 > p.t_cap || re - rb > p.max_span)
            raise_status(p.status, kDevRange);
    }
    if (r >= re || r < 0 || r >= p.r_cap || (int64_t)(r + 1) * 8 > p.t_cap) return;

    const int64_t row0 = (((int64_t)b * p.G + g) * p.t_cap + (int64_t)r * 8) * 64;
    const float sum = region_summary_dim<false>(p.idx_k, p.idx_z, p.cos, p.sin, p.rope_dims, row0, r * 8, d);
    const int64_t srow = ((int64_t)b * p.G + g) * p.r_cap + r;
    p.summ[srow * 64 + d] = f32_to_e4m3(bf16_to_f32(f32_to_bf16_bits(sum)));  // through bf16
    if (p.summ_f32) p.summ_f32[srow * 64 + d] = sum;
    STEP5_STAMP(0, 1);
}

// Bulk form (many regions per sequence): a block takes a chunk of up to 16 consecutive
// regions of one (sequence, group).  Their z rows, k rows (128 token rows of 128 bytes,
// contiguous in the cache) and the chunk's cos/sin rows land in shared memory through
// three or four 1-D bulk copies on one mbarrier; then each thread computes (region, dim)
// pairs from shared memory (a warp reads 32 consecutive dims of a token row: no bank
// conflicts) with the arithmetic of region_summary_dim in its order (max, then exp, den
// and num over tokens 0..7, then num / den), so both forms write the same bits.  Five
// blocks per SM: some blocks' copies overlap the others' arithmetic.
constexpr int kBulkThreads = 256;
constexpr int kBulkRegions = 16;
constexpr int kBulkRows = kBulkRegions * 8;

size_t bulk_smem_bytes(int rope_dims) {
    return 2 * (size_t)kBulkRows * 128 + 2 * (size_t)kBulkRows * (rope_dims / 2) * 2 + 16;
}

__global__ void __launch_bounds__(kBulkThreads) summarize_bulk_kernel(SummarizeParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t* sz = reinterpret_cast<uint16_t*>(smem);                     // [256][64]
    uint16_t* sk = sz + kBulkRows * 64;                                   // [256][64]
    const int half = p.rope_dims >> 1;
    const bool rope = p.cos != nullptr && half > 0;
    uint16_t* sc = sk + kBulkRows * 64;                                   // [256][half]
    uint16_t* ss = sc + kBulkRows * half;                                 // [256][half]
    __shared__ __align__(8) uint64_t bar;
    const int tid = threadIdx.x;
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    pdl_launch_dependents();  // the scoring kernel may start its prologue now
    const int rb = p.region_begin[b];
    const int re = p.region_end[b];
    if (blockIdx.x == 0 && tid == 0) {
        if (rb < 0 || re < rb || re > p.r_cap || (int64_t)re * 8 > p.t_cap || re - rb > p.max_span)
            raise_status(p.status, kDevRange);
    }
    // the chunk: regions r0 .. r0 + nreg - 1, all in range
    const int r0 = rb + blockIdx.x * kBulkRegions;
    int r1 = min(re, r0 + kBulkRegions);
    r1 = min(r1, p.r_cap);
    r1 = (int)min((int64_t)r1, (int64_t)p.t_cap / 8);
    const int nreg = r1 - r0;
    if (r0 < 0 || nreg <= 0) return;
    const int64_t row0 = ((int64_t)b * p.G + g) * p.t_cap + (int64_t)r0 * 8;  // first token row
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        const uint32_t kz_bytes = (uint32_t)nreg * 8 * 128;
        const uint32_t tab_bytes = rope ? (uint32_t)nreg * 8 * half * 2 : 0u;
        mbar_arrive_expect_tx(&bar, 2 * kz_bytes + 2 * tab_bytes);
        bulk_load(sz, p.idx_z + row0 * 64, kz_bytes, &bar);
        bulk_load(sk, p.idx_k + row0 * 64, kz_bytes, &bar);
        if (rope) {
            bulk_load(sc, p.cos + (int64_t)r0 * 8 * half, tab_bytes, &bar);
            bulk_load(ss, p.sin + (int64_t)r0 * 8 * half, tab_bytes, &bar);
        }
    }
    __syncthreads();  // the barrier is initialised before anyone waits on it
    if (!mbar_wait(&bar, 0)) {
        if (tid == 0) raise_status(p.status, kDevTimeout);
        return;  // (only after every copy that could still land: none is left in flight once
                 // the bounded wait has spun for seconds; the block's outputs are not written)
    }
    const int d = tid & 63;
    const bool rotated = rope && d < p.rope_dims;
    const bool first = d < half;
    const int pd = first ? d + half : d - half;
    const int pi = first ? d : d - half;
    for (int lr = tid >> 6; lr < nreg; lr += kBulkThreads / 64) {
        const uint16_t* zr = sz + lr * 8 * 64;
        const uint16_t* kr = sk + lr * 8 * 64;
        float m = -INFINITY;
#pragma unroll
        for (int t = 0; t < 8; ++t) m = fmaxf(m, bf16_to_f32(zr[t * 64 + d]));
        float den = 0.0f, num = 0.0f;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            float kv = bf16_to_f32(kr[t * 64 + d]);
            if (rotated)
                kv = bf16_to_f32(neox_rotate(kv, bf16_to_f32(kr[t * 64 + pd]),
                                             bf16_to_f32(sc[(lr * 8 + t) * half + pi]),
                                             bf16_to_f32(ss[(lr * 8 + t) * half + pi]), first));
            const float e = expf(bf16_to_f32(zr[t * 64 + d]) - m);
            den += e;
            num = fmaf(e, kv, num);
        }
        const float sum = num / den;
        const int64_t srow = ((int64_t)b * p.G + g) * p.r_cap + r0 + lr;
        p.summ[srow * 64 + d] = f32_to_e4m3(bf16_to_f32(f32_to_bf16_bits(sum)));  // through bf16
        if (p.summ_f32) p.summ_f32[srow * 64 + d] = sum;
    }
}

__global__ void convert_kernel(const uint16_t* in, uint8_t* out, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = f32_to_e4m3(bf16_to_f32(in[i]));
}

}  // namespace

cudaError_t launch_summarize(const SummarizeParams& p, int B, cudaStream_t stream) {
    // the SM's shared-memory split of the scoring kernel that follows, so that blocks of
    // both fit on one SM without the SM first draining to change it
    static std::atomic<uint64_t> carveout_set{0};
    cudaError_t e = once_per_device(carveout_set, [] {
        return cudaFuncSetAttribute(summarize_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    (int)cudaSharedmemCarveoutMaxShared);
    });
    if (e != cudaSuccess) return e;
    if (p.max_span > kBulkMinSpan) {  // many regions: the staged bulk form
        static std::atomic<uint64_t> bulk_set{0};
        e = once_per_device(bulk_set, [] {
            return cudaFuncSetAttribute(summarize_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)bulk_smem_bytes(64));
        });
        if (e != cudaSuccess) return e;
        dim3 grid((p.max_span + kBulkRegions - 1) / kBulkRegions, p.G, B);
        summarize_bulk_kernel<<<grid, kBulkThreads, bulk_smem_bytes(p.cos ? p.rope_dims : 0), stream>>>(p);
        return cudaGetLastError();
    }
    dim3 grid((p.max_span + kRegionsPerCta - 1) / kRegionsPerCta, p.G, B);
    summarize_kernel<<<grid, kSumThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_convert(const uint16_t* in, uint8_t* out, int64_t n, cudaStream_t stream) {
    int blocks = (int)((n + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    convert_kernel<<<blocks, 256, 0, stream>>>(in, out, n);
    return cudaGetLastError();
}

}  // namespace step5
