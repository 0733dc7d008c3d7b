// summarize.cu -- step (1): e4m3 summaries of completed regions.
//
// "Step-5-Preview on one 256 GB Mac" (TensorFold PR #903), CSA-indexer commit: every
// completed 8-token region is summarised, per KV group, as a per-dim softmax over z of
// the indexer k, rounded through bf16 to e4m3; the indexer k takes NEOX rotation on its
// first rope_dims dims from bf16 cos/sin.
//
// HBM-bound: 2 KB of k/z in, 64 B out per (region, group).  One thread per (region,
// dim): a warp covers 32 consecutive dims, so each load instruction reads 64
// contiguous bytes of a token row, and each thread's dependency chain is 8 tokens long.
// Rotated dims also read the partner dim (the other half of the NEOX pair).
#include "kernels.cuh"

namespace step5 {

namespace {

// One region (64 dims) per block: a 64-thread block at <= 48 registers a thread fits beside
// a scoring block (512 threads x 112 registers) on one SM, so in a decode step neither
// kernel waits for the SMs the other holds.
constexpr int kRegionsPerCta = 1;
constexpr int kSumThreads = kRegionsPerCta * 64;

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
