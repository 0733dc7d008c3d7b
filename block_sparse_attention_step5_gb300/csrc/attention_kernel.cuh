// attention_kernel.cuh -- step (4): attention over the picked regions plus the row's own region
// (and, optionally, the per-head sigmoid output gate that follows it).
//
// "Step-5-Preview on one 256 GB Mac" (TensorFold PR #903), CSA-indexer commit: each row
// attends to its picked regions plus its own region; with at most 512 regions that is
// every region, i.e. the dense attention the indexer replaces.  The same page's decode
// kernel spreads a row's keys over many workers (a single worker per row was
// load-latency bound) and merges their online-softmax states in a fixed order.
//
// Design (sm_103a):
//  * S blocks per (row, KV group) (S = 1..64, as many as the SMs allow: one SM gathers
//    scattered 2 KB regions at only ~35-65 GB/s, so the gather needs many SMs) split
//    the row's key list (picked regions in selection order, then the own region) into
//    runs of whole 16-token pairs; 8 warps per block, each warp with its own pipeline of
//    2 pair buffers (warp 0: 3).
//  * a region is a contiguous 2 KB tile of the [B][G][t_cap][128] cache; it is fetched
//    with one TMA box of a 3-D view (64 dims x 8 rows x 2 row halves) into two
//    128-byte-swizzled half tiles, so the ldmatrix reads below hit 8 distinct bank
//    groups.
//  * S = Q K^T and O += P V run on bf16 mma.sync (m16n8k16, fp32 accumulate) with the
//    group's query heads as the 16-row left operand (4, 8 or 16 heads; unused rows are
//    zero); P is rounded to bf16 for the PV product, the softmax state is fp32.
//  * the warps merge through shared memory (weights once per (warp, head)); with S > 1
//    every block writes its state (m, l, o per head) to the workspace and raises its flag
//    (an epoch per (row, group) tells launches apart); once all S flags are up each block
//    merges a slice of the outputs over all S states in split order, so the result does
//    not depend on timing.
//
// The kernel template; attention.cu instantiates the whole-row kernel and
// attention_shard.cu the shard kernel, each in its own translation unit.
#pragma once

#include "kernels.cuh"

namespace step5 {

namespace {

constexpr int kThreads = kAttnWarps * 32;
constexpr int kRegionBytes = 2048;                    // 8 tokens x 128 dims x bf16
constexpr int kPairBytes = 4 * kRegionBytes;          // K (2 regions) + V (2 regions)
constexpr int kPairBufs = kAttnWarps * kAttnStages + 1;  // warp 0 has one more
constexpr int kStageBytes = kPairBufs * kPairBytes;
constexpr int kMergeRow = 136;                        // a row of O: 128 floats + 8 of padding
constexpr int kMergeFloatsPerWarp = 16 * kMergeRow + 32;  // O[16][kMergeRow], m[16], l[16]
constexpr int kBarBytes = kPairBufs * 8;
constexpr int kSlotFloats = kAttnSlotFloats;         // m, l, o[128] of one head row
static_assert(kAttnWarps * kMergeFloatsPerWarp * 4 <= kStageBytes, "warp merge area must fit");
static_assert((16 * 128 + kAttnMaxSplits) * 4 <= kStageBytes, "split merge area must fit");
static_assert((kMaxTopK + 2) * 4 + (kAttnWarps * 16 + 32 + 16 * kAttnMaxSplits + 16) * 4 <= kAttnStaticSmem,
              "static shared memory");

// Dynamic shared memory: [stage area | barriers | (cluster form) this block's state]
constexpr int kClusterStateBytes = 16 * kAttnSlotFloats * 4;
size_t attn_smem_bytes(bool cluster = false) {
    return 1024 + kStageBytes + kBarBytes + (cluster ? kClusterStateBytes : 0);
}

// Shared-memory byte offset of (token row t, 16-byte chunk c16 of the 256-byte row) in a
// region tile written by two 64-dim TMA boxes with 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_off(int t, int c16) {
    const int half = c16 >> 3, c = c16 & 7;
    return (uint32_t)(half * 1024 + t * 128 + ((c ^ t) << 4));
}

// The per-head sigmoid output gate of query head h of row n (1 without a gate): every
// output dim of the head is scaled by sigmoid(logit) before the one bf16 rounding.
__device__ __forceinline__ float gate_factor(const AttnParams& p, int n, int h) {
    if (p.gate == nullptr) return 1.0f;
    const float g = bf16_to_f32(p.gate[(int64_t)n * p.Hq + h]);
    return 1.0f / (1.0f + expf(-g));
}

// kShard: a shard of the rows' tokens (tokens tok_lo .. tok_lo + t_cap - 1 of each
// sequence in the caches; keys outside are skipped; softmax states out instead of the
// output).  A separate instantiation, so that the whole-row kernel carries none of it.
// kCluster: the S blocks of a (row, group) form one thread-block cluster and exchange
// their states through distributed shared memory instead of the workspace (S <= 16).
template <bool kShard, bool kCluster = false>
__global__ void __launch_bounds__(kThreads) sparse_attn_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                const __grid_constant__ CUtensorMap vmap,
                                                                AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem(smem_raw, 1024);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStageBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, n = blockIdx.y, g = blockIdx.z;  // group-major (see the launch)
    const int64_t ng = (int64_t)n * p.G + g;
    const int hq_g = p.hq_g;
    const int S = p.splits;

    if (tid == 0) {
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
    }
    STEP5_STAMP(4, 0);
    pdl_wait();
    pdl_launch_dependents();
    STEP5_STAMP(4, 1);

    // the row's position, pick count and every picked id of this block's run, in one
    // round trip
    __shared__ int32_t s_ids[kMaxTopK + 2];  // eps <= top_k + 2 (whole pairs)
    const int32_t* ids = p.sel_ids + ng * p.top_k;
    const int e0 = split * p.entries_per_split;
    for (int i = tid; i < p.entries_per_split; i += kThreads)
        s_ids[i] = e0 + i < p.top_k ? __ldg(ids + e0 + i) : -1;
    const int b = p.row_seq[n];
    const int pos = p.row_pos[n];
    int cnt = p.sel_count[ng];
    const uint32_t epoch = (S > 1 && !kCluster) ? __ldcg(p.bar + ng) : 0u;
    __syncthreads();
    STEP5_STAMP(4, 8);
    // (a shard's position may lie past its tokens)
    if (b < 0 || b >= p.B || pos < 0 || (!kShard && pos >= p.t_cap)) {
        // the same for every block of the (row, group): all leave before its barrier
        if (split == 0) {
            if (tid == 0) raise_status(p.status, kDevRange);
            const int64_t h0 = (int64_t)n * p.Hq + (int64_t)g * hq_g;
            if constexpr (kShard) {  // an empty state
                for (int i = tid; i < hq_g * kSlotFloats; i += kThreads)
                    p.states[h0 * kSlotFloats + i] = i % kSlotFloats == 0 ? -INFINITY : 0.0f;
            } else {
                for (int i = tid; i < hq_g * 128; i += kThreads) p.out[h0 * 128 + i] = 0;
            }
        }
        return;
    }
    if (cnt < 0 || cnt > p.top_k) {
        if (split == 0 && tid == 0) raise_status(p.status, kDevRange);
        cnt = cnt < 0 ? 0 : p.top_k;
    }
    const int own = pos >> 3;
    const int own_tokens = pos - own * 8 + 1;
    const int E = cnt + 1;
    const int e1 = min(E, e0 + p.entries_per_split);
    const int64_t row_base = ((int64_t)b * p.G + g) * p.t_cap;
    const int npairs = e1 > e0 ? (e1 - e0 + 1) >> 1 : 0;
    const int nmy = npairs > warp ? (npairs - warp + kAttnWarps - 1) / kAttnWarps : 0;

    const int nst = warp == 0 ? kAttnStages + 1 : kAttnStages;  // this warp's pair buffers
    const int wfirst = warp == 0 ? 0 : warp * kAttnStages + 1;
    uint8_t* wstage = smem + wfirst * kPairBytes;
    uint64_t* wbar = bars + wfirst;
    if (lane == 0) {
        for (int st = 0; st < nst; ++st) mbar_init(&wbar[st], 1);
        fence_mbar_init();
    }
    __syncwarp();
    STEP5_STAMP(4, 9);

    // entry e -> (region id, valid tokens); invalid ids are masked out entirely, and so
    // are regions outside a shard's tokens (a shard's rid is then relative to tok_lo)
    const int rlo = kShard ? p.tok_lo >> 3 : 0, rhi = kShard ? (p.tok_lo + p.t_cap) >> 3 : 0;
    auto in_shard = [&](int& rid) -> bool {  // (always true for the whole row)
        if constexpr (kShard) {
            if (rid < rlo || rid >= rhi) {
                rid = -1;
                return false;
            }
            rid -= rlo;
        }
        return true;
    };
    auto entry = [&](int e, int& rid) -> int {
        if (e >= e1) {
            rid = -1;
            return 0;
        }
        if (e == cnt) {
            rid = own;
            return in_shard(rid) ? own_tokens : 0;
        }
        rid = s_ids[e - e0];
        if (rid < 0 || rid >= own) {
            raise_status(p.status, kDevRange);
            rid = -1;
            return 0;
        }
        return in_shard(rid) ? 8 : 0;
    };

    auto issue = [&](int li) {
        if (lane != 0) return;
        const int pi = warp + li * kAttnWarps;
        const int st = li % nst;
        uint8_t* kt = wstage + st * kPairBytes;
        uint8_t* vt = kt + 2 * kRegionBytes;
        int ra, rb;
        const int na = entry(e0 + 2 * pi, ra);
        const int nb = entry(e0 + 2 * pi + 1, rb);
        const uint32_t bytes = (uint32_t)(((na > 0) + (nb > 0)) * 2 * kRegionBytes);
        mbar_arrive_expect_tx(&wbar[st], bytes);
        if (na > 0) {
            const int y = (int)(row_base + (int64_t)ra * 8);
            tma_load_3d(kt, &kmap, &wbar[st], 0, y, 0);
            tma_load_3d(vt, &vmap, &wbar[st], 0, y, 0);
        }
        if (nb > 0) {
            const int y = (int)(row_base + (int64_t)rb * 8);
            tma_load_3d(kt + kRegionBytes, &kmap, &wbar[st], 0, y, 0);
            tma_load_3d(vt + kRegionBytes, &vmap, &wbar[st], 0, y, 0);
        }
    };

    for (int li = 0; li < nst && li < nmy; ++li) issue(li);
    STEP5_STAMP(4, 2);

    // query heads of the group as the A operand (rows >= hq_g are zero)
    const int qr = lane >> 2, qc = (lane & 3) * 2;
    uint32_t qa[8][4];
    {
        const uint16_t* qb = p.q + ((int64_t)n * p.Hq + (int64_t)g * hq_g) * 128;
        const bool v0 = qr < hq_g, v1 = qr + 8 < hq_g;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int c = kk * 16 + qc;
            qa[kk][0] = v0 ? *reinterpret_cast<const uint32_t*>(qb + qr * 128 + c) : 0u;
            qa[kk][1] = v1 ? *reinterpret_cast<const uint32_t*>(qb + (qr + 8) * 128 + c) : 0u;
            qa[kk][2] = v0 ? *reinterpret_cast<const uint32_t*>(qb + qr * 128 + c + 8) : 0u;
            qa[kk][3] = v1 ? *reinterpret_cast<const uint32_t*>(qb + (qr + 8) * 128 + c + 8) : 0u;
        }
    }

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    float o[16][4];
#pragma unroll
    for (int nn = 0; nn < 16; ++nn) o[nn][0] = o[nn][1] = o[nn][2] = o[nn][3] = 0.0f;

    int li_fail = -1;
    for (int li = 0; li < nmy; ++li) {
        const int pi = warp + li * kAttnWarps;
        const int st = li % nst;
        uint8_t* kt = wstage + st * kPairBytes;
        uint8_t* vt = kt + 2 * kRegionBytes;
        int ra, rb;
        const int na = entry(e0 + 2 * pi, ra);
        const int nb = entry(e0 + 2 * pi + 1, rb);
        if (!mbar_wait(&wbar[st], (uint32_t)((li / nst) & 1))) {
            li_fail = li;
            break;
        }
        // zero the V rows of masked tokens so that 0-weight rows stay finite
        if (na < 8 || nb < 8) {
            for (int i = lane; i < 2 * 8 * 16; i += 32) {
                const int slot = i >> 7, t = (i >> 4) & 7, c16 = i & 15;
                const int valid = slot ? nb : na;
                if (t >= valid)
                    *reinterpret_cast<uint4*>(vt + slot * kRegionBytes + tile_off(t, c16)) =
                        make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
        }
        if (li == 0) STEP5_STAMP(4, 3);
        const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);

        // S = Q K^T over the 16 tokens (slot 0: tokens 0-7, slot 1: tokens 8-15)
        float s[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.0f;
            const int mat = lane >> 3, t = lane & 7;
#pragma unroll
            for (int kk = 0; kk < 8; kk += 2) {
                const int c16 = 2 * (kk + (mat >> 1)) + (mat & 1);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(b0, b1, b2, b3, kbase + j * kRegionBytes + tile_off(t, c16));
                mma_bf16_16816(s[j], qa[kk], b0, b1);
                mma_bf16_16816(s[j], qa[kk + 1], b2, b3);
            }
        }
        // scale, mask, online softmax (rows qr and qr + 8)
        const int tq = (lane & 3) * 2;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int valid = j ? nb : na;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = tq + (e & 1);
                s[j][e] = (t < valid) ? s[j][e] * p.scale_log2 : -INFINITY;
            }
            mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
            mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float base0 = (mn0 == -INFINITY) ? 0.0f : mn0;
        const float base1 = (mn1 == -INFINITY) ? 0.0f : mn1;
        const float a0 = exp2f(m0 - base0), a1 = exp2f(m1 - base1);
        m0 = mn0;
        m1 = mn1;
        float pr[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            pr[j][0] = exp2f(s[j][0] - base0);
            pr[j][1] = exp2f(s[j][1] - base0);
            pr[j][2] = exp2f(s[j][2] - base1);
            pr[j][3] = exp2f(s[j][3] - base1);
        }
        l0 = l0 * a0 + (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
        l1 = l1 * a1 + (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
#pragma unroll
        for (int nn = 0; nn < 16; ++nn) {
            o[nn][0] *= a0;
            o[nn][1] *= a0;
            o[nn][2] *= a1;
            o[nn][3] *= a1;
        }
        uint32_t pa[4];
        pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
        pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
        pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
        pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
        // O += P V
        {
            const int mat = lane >> 3, t = lane & 7;
            const int slot = mat & 1;
#pragma unroll
            for (int nn = 0; nn < 16; nn += 2) {
                const int c16 = nn + (mat >> 1);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(b0, b1, b2, b3, vbase + slot * kRegionBytes + tile_off(t, c16));
                mma_bf16_16816(o[nn], pa, b0, b1);
                mma_bf16_16816(o[nn + 1], pa, b2, b3);
            }
        }
        __syncwarp();
        fence_proxy_async();
        if (li + nst < nmy) issue(li + nst);
    }
    if (li_fail >= 0) {
        if (lane == 0) raise_status(p.status, kDevTimeout);
        // give the copies this warp issued and did not consume a bounded chance to land
        // before the block's shared memory goes away
        for (int li = li_fail; li < nmy && li < li_fail + nst; ++li)
            mbar_wait(&wbar[li % nst], (uint32_t)((li / nst) & 1));
    }

    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    // ---- merge the warps through shared memory (reuses the stage buffers)
    STEP5_STAMP(4, 4);
    __syncthreads();
    // rows at or past hq_g hold zero queries and are skipped; the padded rows put the 8
    // rows of one store on 8 different bank groups (float2 stores)
    float* mw = reinterpret_cast<float*>(smem) + warp * kMergeFloatsPerWarp;
    if (qr < hq_g) {
#pragma unroll
        for (int nn = 0; nn < 16; ++nn)
            *reinterpret_cast<float2*>(mw + qr * kMergeRow + nn * 8 + qc) = make_float2(o[nn][0], o[nn][1]);
    }
    if (qr + 8 < hq_g) {
#pragma unroll
        for (int nn = 0; nn < 16; ++nn)
            *reinterpret_cast<float2*>(mw + (qr + 8) * kMergeRow + nn * 8 + qc) = make_float2(o[nn][2], o[nn][3]);
    }
    if ((lane & 3) == 0) {
        mw[16 * kMergeRow + qr] = m0;
        mw[16 * kMergeRow + qr + 8] = m1;
        mw[16 * kMergeRow + 16 + qr] = l0;
        mw[16 * kMergeRow + 16 + qr + 8] = l1;
    }
    __syncthreads();
    STEP5_STAMP(4, 5);

    // per-row max, warp weights and sum, once per (row, warp) by warp 0 (its lanes take
    // 4 rows x 8 warps per pass); then thread (rpar, d) combines dim d of rows rpar,
    // rpar + 2, ... with those weights
    __shared__ float s_wsc[kAttnWarps][16], s_M[16], s_L[16];
    const int d = tid & 127, rpar = tid >> 7;
    const float* mall = reinterpret_cast<const float*>(smem);
    if (warp == 0) {
        for (int r0 = 0; r0 < hq_g; r0 += 32 / kAttnWarps) {
            const int r = r0 + lane / kAttnWarps, w = lane % kAttnWarps;
            const bool ok = r < hq_g;
            const float m = ok ? mall[w * kMergeFloatsPerWarp + 16 * kMergeRow + r] : -INFINITY;
            float M = m;
#pragma unroll
            for (int o = 1; o < kAttnWarps; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float sc = exp2f(m - ((M == -INFINITY) ? 0.0f : M));
            float L = ok ? mall[w * kMergeFloatsPerWarp + 16 * kMergeRow + 16 + r] * sc : 0.0f;
#pragma unroll
            for (int o = 1; o < kAttnWarps; o <<= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
            if (ok) {
                s_wsc[w][r] = sc;
                if (w == 0) {
                    s_M[r] = M;
                    s_L[r] = L;
                }
            }
        }
    }
    __syncthreads();
    if (S == 1) {
        for (int r = rpar; r < hq_g; r += 2) {
            float O = 0.0f;
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) O += mall[w * kMergeFloatsPerWarp + r * kMergeRow + d] * s_wsc[w][r];
            const int64_t hrow = (int64_t)n * p.Hq + (int64_t)g * hq_g + r;
            if constexpr (kShard) {  // the state, not the output
                float* st = p.states + hrow * kSlotFloats;
                st[2 + d] = O;
                if (d == 0) {
                    st[0] = s_M[r];
                    st[1] = s_L[r];
                }
            } else {
                p.out[hrow * 128 + d] = f32_to_bf16_bits(O / s_L[r] * gate_factor(p, n, g * hq_g + r));
            }
        }
        return;
    }

    if constexpr (kCluster) {
        // ---- S blocks per (row, group) in one cluster: this block's state into its own
        // shared memory, a cluster barrier, then a slice of the outputs merged over the S
        // states read through distributed shared memory, and a second barrier so that no
        // block leaves while another still reads its state.  Every block of the cluster
        // reaches both barriers (the early exits above are the same for all of them).
        float* st = reinterpret_cast<float*>(smem + kStageBytes + kBarBytes);  // [hq_g][130]
        for (int r = rpar; r < hq_g; r += 2) {
            float O = 0.0f;
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) O += mall[w * kMergeFloatsPerWarp + r * kMergeRow + d] * s_wsc[w][r];
            st[r * kSlotFloats + 2 + d] = O;
            if (d == 0) {
                st[r * kSlotFloats] = s_M[r];
                st[r * kSlotFloats + 1] = s_L[r];
            }
        }
        STEP5_STAMP(4, 11);
        cluster_sync();
        STEP5_STAMP(4, 6);
        const uint32_t st_addr = smem_u32(st);
        const int EO = hq_g * 128;
        const int e_lo = EO * split / S, e_hi = EO * (split + 1) / S, nout = e_hi - e_lo;
        __shared__ float s_cw[16][16], s_cL[16];  // weight of split sp for a slice row; row sums
        const int r_lo = e_lo >> 7, r_hi = (e_hi - 1) >> 7;
        for (int r = r_lo + warp; r <= r_hi; r += kAttnWarps) {  // lanes take splits
            const bool on = lane < S;
            const uint32_t at = st_addr + (uint32_t)(r * kSlotFloats) * 4u;
            const float m = on ? ld_cluster_f32(map_cluster(at, lane)) : -INFINITY;
            const float l = on ? ld_cluster_f32(map_cluster(at + 4u, lane)) : 0.0f;
            float M = m;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float sc = exp2f(m - ((M == -INFINITY) ? 0.0f : M));
            float L = l * sc;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
            if (on) s_cw[r - r_lo][lane] = sc;
            if (lane == 0) {
                s_cL[r - r_lo] = L;
                if constexpr (kShard) {
                    float* gs = p.states + ((int64_t)n * p.Hq + (int64_t)g * hq_g + r) * kSlotFloats;
                    gs[0] = M;
                    gs[1] = L;
                }
            }
        }
        __syncthreads();
        for (int t = tid; t < nout; t += kThreads) {
            const int e = e_lo + t, r = e >> 7;
            const uint32_t at = st_addr + (uint32_t)(r * kSlotFloats + 2 + (e & 127)) * 4u;
            float O = 0.0f;
            for (int sp = 0; sp < S; ++sp) O += ld_cluster_f32(map_cluster(at, sp)) * s_cw[r - r_lo][sp];
            const int64_t hrow = (int64_t)n * p.Hq + (int64_t)g * hq_g + r;
            if constexpr (kShard)
                p.states[hrow * kSlotFloats + 2 + (e & 127)] = O;
            else
                p.out[hrow * 128 + (e & 127)] = f32_to_bf16_bits(O / s_cL[r - r_lo] * gate_factor(p, n, g * hq_g + r));
        }
        STEP5_STAMP(4, 7);
        cluster_sync();
        return;
    }

    // ---- S blocks per (row, group): this block's state into the workspace
    const float* pall = p.part + ng * S * hq_g * kSlotFloats;  // [S][hq_g][130]
    {
        float* mine = p.part + (ng * S + split) * hq_g * kSlotFloats;
        for (int r = rpar; r < hq_g; r += 2) {
            float O = 0.0f;
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) O += mall[w * kMergeFloatsPerWarp + r * kMergeRow + d] * s_wsc[w][r];
            mine[r * kSlotFloats + 2 + d] = O;
            if (d == 0) {
                mine[r * kSlotFloats] = s_M[r];
                mine[r * kSlotFloats + 1] = s_L[r];
            }
        }
    }
    STEP5_STAMP(4, 11);
    // The exchange: each block raises its flag to the (row, group)'s epoch + 1 (release)
    // once its state is out, and reads the states after seeing every flag raised
    // (acquire); block 0 then advances the epoch for the next launch (every block has
    // read it by then, since each reads it before raising its flag).
    __syncthreads();
    uint32_t* fl = p.flags + ng * kAttnMaxSplits;
    if (tid == 0) st_release_u32(fl + split, epoch + 1u);
    bool ok = true;
    if (warp == 0) {
        ok = false;
        for (uint32_t it = 0; it < kBarrierPolls; ++it) {
            bool all = true;
            for (int sp = lane; sp < S; sp += 32) all &= ld_relaxed_u32(fl + sp) == epoch + 1u;
            if (__all_sync(0xffffffffu, all)) {
                ok = true;
                break;
            }
        }
        fence_acquire_gpu();  // the flags' release stores happen before the reads below
    }
    if (__syncthreads_or(!ok)) {
        if (tid == 0) raise_status(p.status, kDevTimeout);
        return;
    }
    if (split == 0 && tid == 0) p.bar[ng] = epoch + 1u;
    STEP5_STAMP(4, 6);

    // ---- this block's slice [e_lo, e_hi) of the hq_g * 128 outputs, merged over the S
    // states in split order.  Every (split, output) value of the slice (at most
    // EO + S) is requested at once: item j = tid + kThreads * u -> split j / nout, output j % nout.
    const int EO = hq_g * 128;
    const int e_lo = EO * split / S, e_hi = EO * (split + 1) / S, nout = e_hi - e_lo;
    float* s_val = reinterpret_cast<float*>(smem);  // [S][nout], reuses the stage area
    constexpr int kItems = (16 * 128 + kAttnMaxSplits + kThreads - 1) / kThreads;  // S * nout <= EO + S
    float v[kItems];
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
        const int j = tid + kThreads * u;
        v[u] = 0.0f;
        if (j < S * nout) {
            const int sp = j / nout, e = e_lo + j - sp * nout;
            v[u] = __ldcg(pall + ((int64_t)sp * hq_g + (e >> 7)) * kSlotFloats + 2 + (e & 127));
        }
    }
    // weights of every split for the rows the slice touches: warp w takes rows
    // r_lo + w, r_lo + w + 8, ...; lanes take splits
    __shared__ float s_sw[16][kAttnMaxSplits], s_sL[16];
    const int r_lo = e_lo >> 7, r_hi = (e_hi - 1) >> 7;
    for (int r = r_lo + warp; r <= r_hi; r += kAttnWarps) {
        float m[kAttnMaxSplits / 32], l[kAttnMaxSplits / 32];
#pragma unroll
        for (int k = 0; k < kAttnMaxSplits / 32; ++k) {
            const int sp = lane + 32 * k;
            m[k] = sp < S ? __ldcg(pall + ((int64_t)sp * hq_g + r) * kSlotFloats) : -INFINITY;
            l[k] = sp < S ? __ldcg(pall + ((int64_t)sp * hq_g + r) * kSlotFloats + 1) : 0.0f;
        }
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < kAttnMaxSplits / 32; ++k) M = fmaxf(M, m[k]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float base = (M == -INFINITY) ? 0.0f : M;
        float L = 0.0f;
#pragma unroll
        for (int k = 0; k < kAttnMaxSplits / 32; ++k) {
            const int sp = lane + 32 * k;
            const float sc = exp2f(m[k] - base);
            if (sp < S) s_sw[r - r_lo][sp] = sc;
            L += l[k] * sc;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (lane == 0) {
            s_sL[r - r_lo] = L;
            if constexpr (kShard) {  // (every block touching the row writes the same)
                float* st = p.states + ((int64_t)n * p.Hq + (int64_t)g * hq_g + r) * kSlotFloats;
                st[0] = M;
                st[1] = L;
            }
        }
    }
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
        const int j = tid + kThreads * u;
        if (j < S * nout) s_val[j] = v[u];
    }
    __syncthreads();
    for (int t = tid; t < nout; t += kThreads) {
        const int e = e_lo + t, r = e >> 7;
        float O = 0.0f;
        for (int sp = 0; sp < S; ++sp) O += s_val[sp * nout + t] * s_sw[r - r_lo][sp];
        const int64_t hrow = (int64_t)n * p.Hq + (int64_t)g * hq_g + r;
        if constexpr (kShard)
            p.states[hrow * kSlotFloats + 2 + (e & 127)] = O;
        else
            p.out[hrow * 128 + (e & 127)] = f32_to_bf16_bits(O / s_sL[r - r_lo] * gate_factor(p, n, g * hq_g + r));
    }
    STEP5_STAMP(4, 7);
}

// Sets the kernel's shared-memory limit once, then launches it (kCluster: the split
// blocks of a (row, group) as one cluster of p.splits blocks).
template <bool kShard, bool kCluster = false>
cudaError_t launch_sparse_attn(const AttnParams& p, int N, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               cudaStream_t stream, bool pdl) {
    static std::atomic<uint64_t> attr_set{0};
    cudaError_t e = once_per_device(attr_set, [] {
        cudaError_t e1 = cudaFuncSetAttribute(sparse_attn_kernel<kShard, kCluster>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)attn_smem_bytes(kCluster));
        if (e1 == cudaSuccess && kCluster)
            e1 = cudaFuncSetAttribute(sparse_attn_kernel<kShard, kCluster>,
                                      cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        return e1;
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    // rows before groups: blocks that run together share one KV group's cache (for a
    // prefill chunk, 1/G of the K/V it reads), which then stays in L2
    cfg.gridDim = dim3(p.splits, N, p.G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = attn_smem_bytes(kCluster);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (kCluster) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)p.splits;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, sparse_attn_kernel<kShard, kCluster>, kmap, vmap, p);
}

}  // namespace

}  // namespace step5
