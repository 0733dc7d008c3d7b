// summarize.cu -- step (1): e4m3 summaries of completed regions.
//
// "Step-5-Preview on one 256 GB Mac" (TensorFold PR #903), CSA-indexer commit: every
// completed 8-token region is summarised, per KV group, as a per-dim softmax over z of
// the indexer k, rounded through bf16 to e4m3; the indexer k takes NEOX rotation on its
// first rope_dims dims from bf16 cos/sin.
//
// HBM-bound: 2 KB of k/z in, 64 B out per (region, group).  One region is handled by
// 8 threads, each owning 8 dims (one 16-byte vector per token row), so a warp reads
// four full 128-byte token rows per load instruction.  Rotated dims also read the
// partner slice (the other half of each NEOX pair) from the same rows.
#include "kernels.cuh"

namespace step5 {

namespace {

constexpr int kRegionsPerCta = 32;  // 8 threads each -> 256 threads

__global__ void __launch_bounds__(256) summarize_kernel(SummarizeParams p) {
    const int lr = threadIdx.x >> 3;   // region within the CTA
    const int j = threadIdx.x & 7;     // 8-dim slice
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    const int rb = p.region_begin[b];
    const int re = p.region_end[b];
    const int r = rb + blockIdx.x * kRegionsPerCta + lr;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        // range checks of this sequence, once
        if (rb < 0 || re < rb || re > p.r_cap || (int64_t)re * 8 > p.t_cap ||
            re - rb > p.max_span)
            raise_status(p.status, kDevRange);
    }
    if (r >= re || r < 0 || r >= p.r_cap || (int64_t)(r + 1) * 8 > p.t_cap) return;

    const int half = p.rope_dims >> 1;
    const int d0 = j * 8;
    const bool rotated = p.cos != nullptr && d0 < p.rope_dims;
    const bool first = d0 < half;
    const int partner = first ? d0 + half : d0 - half;
    const int pair0 = first ? d0 : d0 - half;   // NEOX pair index of element 0

    const int64_t row0 = ((int64_t)b * p.G + g) * p.t_cap + (int64_t)r * 8;
    const uint4* kz_k = reinterpret_cast<const uint4*>(p.idx_k);
    const uint4* kz_z = reinterpret_cast<const uint4*>(p.idx_z);

    // pass 1: per-dim max of z over the region's 8 tokens
    uint4 zv[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) zv[t] = __ldg(kz_z + ((row0 + t) * 64 + d0) / 8);
    float m[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) m[u] = -INFINITY;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t w4[4] = {zv[t].x, zv[t].y, zv[t].z, zv[t].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            m[2 * q] = fmaxf(m[2 * q], bf16_lo(w4[q]));
            m[2 * q + 1] = fmaxf(m[2 * q + 1], bf16_hi(w4[q]));
        }
    }

    // every load of the region is issued before any arithmetic
    uint4 kv[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) kv[t] = __ldg(kz_k + ((row0 + t) * 64 + d0) / 8);
    uint4 pv[8], cv[8], sv[8];
    if (rotated) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int64_t tabrow = (int64_t)(r * 8 + t) * half + pair0;
            pv[t] = __ldg(kz_k + ((row0 + t) * 64 + partner) / 8);
            cv[t] = __ldg(reinterpret_cast<const uint4*>(p.cos + tabrow));
            sv[t] = __ldg(reinterpret_cast<const uint4*>(p.sin + tabrow));
        }
    }

    // pass 2: weights and weighted sum (fp32, tokens in order)
    float den[8], num[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) den[u] = num[u] = 0.0f;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        float kr[8];
        const uint32_t kw[4] = {kv[t].x, kv[t].y, kv[t].z, kv[t].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            kr[2 * q] = bf16_lo(kw[q]);
            kr[2 * q + 1] = bf16_hi(kw[q]);
        }
        if (rotated) {
            const uint32_t pw[4] = {pv[t].x, pv[t].y, pv[t].z, pv[t].w};
            const uint32_t cw[4] = {cv[t].x, cv[t].y, cv[t].z, cv[t].w};
            const uint32_t sw[4] = {sv[t].x, sv[t].y, sv[t].z, sv[t].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                kr[2 * q] = bf16_to_f32(neox_rotate(kr[2 * q], bf16_lo(pw[q]), bf16_lo(cw[q]),
                                                    bf16_lo(sw[q]), first));
                kr[2 * q + 1] = bf16_to_f32(neox_rotate(kr[2 * q + 1], bf16_hi(pw[q]),
                                                        bf16_hi(cw[q]), bf16_hi(sw[q]), first));
            }
        }
        const uint32_t zw[4] = {zv[t].x, zv[t].y, zv[t].z, zv[t].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float e0 = expf(bf16_lo(zw[q]) - m[2 * q]);
            const float e1 = expf(bf16_hi(zw[q]) - m[2 * q + 1]);
            den[2 * q] += e0;
            den[2 * q + 1] += e1;
            num[2 * q] = fmaf(e0, kr[2 * q], num[2 * q]);
            num[2 * q + 1] = fmaf(e1, kr[2 * q + 1], num[2 * q + 1]);
        }
    }

    float s[8];
    uint32_t code_lo = 0, code_hi = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        s[u] = num[u] / den[u];
        const float sb = bf16_to_f32(f32_to_bf16_bits(s[u]));   // through bf16
        const uint32_t c = f32_to_e4m3(sb);
        if (u < 4)
            code_lo |= c << (8 * u);
        else
            code_hi |= c << (8 * (u - 4));
    }
    const int64_t srow = ((int64_t)b * p.G + g) * p.r_cap + r;
    reinterpret_cast<uint2*>(p.summ)[(srow * 64 + d0) / 8] = make_uint2(code_lo, code_hi);
    if (p.summ_f32) {
        float4* o = reinterpret_cast<float4*>(p.summ_f32 + srow * 64 + d0);
        o[0] = make_float4(s[0], s[1], s[2], s[3]);
        o[1] = make_float4(s[4], s[5], s[6], s[7]);
    }
}

__global__ void convert_kernel(const uint16_t* in, uint8_t* out, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = f32_to_e4m3(bf16_to_f32(in[i]));
}

}  // namespace

cudaError_t launch_summarize(const SummarizeParams& p, int B, cudaStream_t stream) {
    dim3 grid((p.max_span + kRegionsPerCta - 1) / kRegionsPerCta, p.G, B);
    summarize_kernel<<<grid, 256, 0, stream>>>(p);
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
