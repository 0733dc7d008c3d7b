// front.cu -- the indexer's decode front end, ahead of step (1).
//
// "Step-5-Preview on one 256 GB Mac" (TensorFold PR #903), CSA-indexer commit: the
// indexer's q (16 heads) goes through RMSNorm with weight 1 + w and its k through a
// LayerNorm with bias (z is used as it is); k and z of every position are kept for the
// region summaries.  Per decode row this kernel normalises q (the scoring call rotates
// it), writes the row's normalised k and its z at the row's position of the caches, and
// when that token completes its 8-token region, writes the region's summary exactly as
// step5_region_summarize does.
//
// One 256-thread block per row: q in 16 groups of 16 threads (4 dims each, a butterfly
// over the group for the sum of squares), k as one thread per (group, dim) with its
// mean and variance summed over the group's two warps, then (region complete) one
// thread per (group, dim) of the summary, reading the region's tokens back through L2.
#include "kernels.cuh"

namespace step5 {

namespace {

constexpr int kFrontThreads = 256;

__global__ void __launch_bounds__(kFrontThreads) front_kernel(FrontParams p) {
    const int n = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __shared__ float s_red[2][8];  // per warp: sum, then sum of squared deviations
    // ---- q: RMSNorm (1 + w) of each head, 16 threads a head, 4 dims a thread
    for (int h0 = 0; h0 < p.idx_heads; h0 += kFrontThreads / 16) {
        const int h = h0 + tid / 16, d0 = (tid % 16) * 4;
        float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const bool on = h < p.idx_heads;
        if (on) {
            const uint2 v = *reinterpret_cast<const uint2*>(p.q_pre + ((int64_t)n * p.idx_heads + h) * 64 + d0);
            x[0] = bf16_to_f32((uint16_t)(v.x & 0xffffu));
            x[1] = bf16_to_f32((uint16_t)(v.x >> 16));
            x[2] = bf16_to_f32((uint16_t)(v.y & 0xffffu));
            x[3] = bf16_to_f32((uint16_t)(v.y >> 16));
        }
        float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (on) {
            const float rms = sqrtf(ss / 64.0f + p.eps);
            uint16_t y[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                y[i] = f32_to_bf16_bits(x[i] / rms * (1.0f + bf16_to_f32(p.q_w[d0 + i])));
            *reinterpret_cast<uint2*>(p.q_out + ((int64_t)n * p.idx_heads + h) * 64 + d0) =
                make_uint2((uint32_t)y[0] | ((uint32_t)y[1] << 16), (uint32_t)y[2] | ((uint32_t)y[3] << 16));
        }
    }
    const int b = p.row_seq[n], pos = p.row_pos[n];
    if (b < 0 || b >= p.B || pos < 0 || pos >= p.t_cap) {
        if (tid == 0) raise_status(p.status, kDevRange);
        return;  // the same for the whole block
    }
    // ---- k: LayerNorm with bias, z as it is, at token pos (one thread per (group, dim))
    const int g = tid >> 6, d = tid & 63;  // G <= 4
    const bool gon = g < p.G;
    const float kx = gon ? bf16_to_f32(p.k_pre[((int64_t)n * p.G + g) * 64 + d]) : 0.0f;
    float sum = kx;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) s_red[0][warp] = sum;
    __syncthreads();
    const float mean = (s_red[0][2 * g] + s_red[0][2 * g + 1]) / 64.0f;
    const float c = kx - mean;
    float sq = c * c;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0) s_red[1][warp] = sq;
    __syncthreads();
    const float var = (s_red[1][2 * g] + s_red[1][2 * g + 1]) / 64.0f;
    const int64_t row = (((int64_t)b * p.G + g) * p.t_cap + pos) * 64;
    if (gon) {
        p.idx_k[row + d] = f32_to_bf16_bits(c / sqrtf(var + p.eps) * bf16_to_f32(p.k_w[d]) + bf16_to_f32(p.k_b[d]));
        p.idx_z[row + d] = p.z_pre[((int64_t)n * p.G + g) * 64 + d];
    }
    // ---- the region this token completes
    const int r = pos >> 3;
    if ((pos & 7) != 7 || r >= p.r_cap) return;
    __syncthreads();  // the token's k and z are written before the region is read back
    if (gon) {
        const int64_t row0 = (((int64_t)b * p.G + g) * p.t_cap + (int64_t)r * 8) * 64;
        const float s = region_summary_dim<true>(p.idx_k, p.idx_z, p.cos, p.sin, p.rope_dims, row0, r * 8, d);
        p.summ[(((int64_t)b * p.G + g) * p.r_cap + r) * 64 + d] = f32_to_e4m3(bf16_to_f32(f32_to_bf16_bits(s)));
    }
}

}  // namespace

cudaError_t launch_front(const FrontParams& p, cudaStream_t stream) {
    front_kernel<<<p.N, kFrontThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace step5
