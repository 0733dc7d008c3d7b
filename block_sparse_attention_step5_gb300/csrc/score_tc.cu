// score_tc.cu -- step (2) on the tcgen05 tensor cores for launches with many rows per
// sequence (prefill chunks): every row's score of every candidate region, into fp32.
//
// "Step-5-Preview on one 256 GB Mac" (TensorFold PR #903), CSA-indexer commit: a region's
// score in KV group g is sum_h relu(e4m3(q_h) . summary) * w_h over g's indexer heads; the
// same page scores a prompt chunk's rows in blocks of 64 rows.  The rows of a chunk share
// their sequence's summaries, so the scoring is a dense FP8 contraction per group:
//
//   D [128 regions x 128] = S_tile [128 regions x 64 dims] . Qe^T [64 x (128 / H rows x H heads)]
//
// (kind::f8f6f4, e4m3 x e4m3 products exact, fp32 accumulation in TMEM), followed by
// score[row][r] = sum_h relu(D[r][row, h]) * w[row][h] in fp32.  One CTA takes a block of
// 128 / H consecutive rows (H = indexer heads per group) and one group: the rows' rotated,
// e4m3-rounded queries are the B operand (built once in shared memory, K-major with
// 64-byte swizzle), the summaries stream through TMA boxes of 256 regions as they lie in
// HBM (64-byte swizzle, used in place as the K-major A operand of two M = 128 tiles).
// A control warp issues the copies and the MMAs (two per tile) into two TMEM
// accumulators; four epilogue warps (one region per thread, its TMEM lane) apply relu * w
// and store the scores of the regions below each row's own region.  Rows of other
// sequences in a block are handled by a pass per sequence.  Selection follows in a
// separate launch (one block per (row, group), as the fused path selects).
#include "tcgen05.cuh"
#include "kernels.cuh"

namespace step5 {

namespace {

constexpr int kScEpiWarps = 4;
constexpr int kScThreads = kScEpiWarps * 32 + 32;   // epilogue warps + the control warp
constexpr int kScCols = 128;                        // N of one MMA (rows x heads of the block)
constexpr int kScSlots = 5;                         // 256-region boxes (~91 KB: two CTAs and their TMEM per SM)
constexpr uint32_t kScBoxBytes = 256 * 64;
constexpr uint32_t kScQBytes = 128 * 64;
constexpr uint32_t kScTmemCols = 2 * kScCols;       // two accumulators
constexpr uint32_t kScIdesc = tc::instr_desc(tc::kFmtE4M3, false, false, 128, kScCols);

size_t sc_smem_bytes() { return 1024 + kScSlots * kScBoxBytes + kScQBytes; }

template <int HPG>
__global__ void __launch_bounds__(kScThreads) score_tc_kernel(const __grid_constant__ CUtensorMap smap, ScoreParams p) {
    constexpr int NR = kScCols / HPG;  // rows of the block
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem(smem_raw, 1024);
    uint8_t* slots = smem;
    uint8_t* qt = smem + kScSlots * kScBoxBytes;
    __shared__ __align__(8) uint64_t full[kScSlots], empty[kScSlots], dfull[2], dempty[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_b[NR], s_R[NR], s_pos[NR], s_seq[NR], s_nseq, s_fail;
    __shared__ float s_w[kScCols];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.y;
    const int n0 = blockIdx.x * NR;

    if (tid == 0) {
        prefetch_tmap(&smap);
        for (int s = 0; s < kScSlots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&dfull[s], 1);
            mbar_init(&dempty[s], kScEpiWarps * 32);
        }
        fence_mbar_init();
        s_fail = 0;
    }
    if (warp == 0) tc::alloc(&s_tmem, kScTmemCols);
    pdl_wait();
    pdl_launch_dependents();

    // the block's rows: sequence, candidate count (-1: out of range or past N)
    for (int j = tid; j < NR; j += kScThreads) {
        const int n = n0 + j;
        int b = -1, R = -1, pos = 0;
        if (n < p.N) {
            R = row_regions(p, n, b, pos);
            if (R < 0) raise_status(p.status, kDevRange);
        }
        s_b[j] = R < 0 ? -1 : b;
        s_R[j] = R;
        s_pos[j] = pos;
    }
    __syncthreads();
    // the rows' queries, rotated and rounded to e4m3, as B rows j * HPG + h (K-major,
    // 64-byte swizzle: 16-byte chunk c of row r at chunk c ^ ((r >> 1) & 3)); rows of
    // invalid rows are zero
    const int half = p.rope_dims >> 1;
    for (int e = tid; e < kScCols * 64; e += kScThreads) {
        const int nb = e >> 6, d = e & 63, j = nb / HPG, h = nb - j * HPG;
        const int n = n0 + j;
        uint8_t code = 0;
        if (n < p.N) {
            const int pos = s_pos[j];
            if (s_b[j] >= 0) {
                const uint16_t* qrow = p.idx_q + ((int64_t)n * p.idx_heads + (int64_t)g * HPG + h) * 64;
                uint16_t rb = qrow[d];
                if (p.cos != nullptr && d < p.rope_dims) {
                    const bool first = d < half;
                    const int pd = first ? d + half : d - half;
                    const int pi = first ? d : d - half;
                    rb = neox_rotate(bf16_to_f32(rb), bf16_to_f32(qrow[pd]), bf16_to_f32(p.cos[(int64_t)pos * half + pi]),
                                     bf16_to_f32(p.sin[(int64_t)pos * half + pi]), first);
                }
                code = f32_to_e4m3(bf16_to_f32(rb));
            }
        }
        qt[nb * 64 + ((((d >> 4) ^ ((nb >> 1) & 3))) << 4) + (d & 15)] = code;
    }
    for (int i = tid; i < kScCols; i += kScThreads) {
        const int j = i / HPG, h = i - j * HPG, n = n0 + j;
        s_w[i] = n < p.N ? p.w[(int64_t)n * p.idx_heads + (int64_t)g * HPG + h] : 0.0f;
    }
    fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {  // the distinct sequences of the block's rows, in first-seen order
        int ns = 0;
        for (int j = 0; j < NR; ++j) {
            const int b = s_b[j];
            if (b < 0) continue;
            bool seen = false;
            for (int k = 0; k < ns; ++k) seen |= s_seq[k] == b;
            if (!seen) s_seq[ns++] = b;
        }
        s_nseq = ns;
    }
    __syncthreads();
    const uint32_t tmem = s_tmem;
    const int nseq = s_nseq;
    // regions of a pass (one sequence): up to the largest R of its rows
    auto pass_regions = [&](int b) {
        int m = 0;
        for (int j = 0; j < NR; ++j)
            if (s_b[j] == b) m = max(m, s_R[j]);
        return m;
    };

    if (warp == kScEpiWarps) {
        // ---------------- control warp: boxes of 256 regions (TMA), two MMAs per tile of 128
        bool ok = true;
        int box = 0, tile = 0;  // running counts over all passes (barrier phases)
        const uint64_t dq = tc::smem_desc(smem_u32(qt), 16, 512, tc::kSwizzle64);
        uint64_t* last_commit = nullptr;
        uint32_t last_parity = 0;
        for (int sq = 0; sq < nseq && ok; ++sq) {
            const int b = s_seq[sq];
            const int nt = (pass_regions(b) + 127) >> 7;
            const int nbox = (nt + 1) >> 1;
            const int box0 = box;
            int issued = 0;
            auto issue_box = [&](int u) {  // box u of this pass
                const int gb = box0 + u, slot = gb % kScSlots, use = gb / kScSlots;
                if (use > 0 && !mbar_wait(&empty[slot], (uint32_t)((use - 1) & 1))) {
                    ok = false;
                    return;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[slot], kScBoxBytes);
                    tma_load_2d(slots + slot * kScBoxBytes, &smap, &full[slot], 0,
                                (int)(((int64_t)b * p.G + g) * p.r_cap + 256 * u));
                }
                __syncwarp();
            };
            for (; issued < nbox && issued < kScSlots - 1 && ok; ++issued) issue_box(issued);
            for (int t = 0; t < nt && ok; ++t, ++tile) {
                const int u = t >> 1, gb = box0 + u, slot = gb % kScSlots;
                if (!mbar_wait(&full[slot], (uint32_t)((gb / kScSlots) & 1))) {
                    ok = false;
                    break;
                }
                if (tile >= 2 && !mbar_wait(&dempty[tile & 1], (uint32_t)(((tile >> 1) - 1) & 1))) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const bool last_of_box = (t & 1) || t + 1 == nt;
                if (lane == 0) {
                    const uint64_t da =
                        tc::smem_desc(smem_u32(slots + slot * kScBoxBytes) + (uint32_t)(t & 1) * 8192u, 16, 512, tc::kSwizzle64);
                    const uint32_t d = tmem + (uint32_t)(tile & 1) * kScCols;
                    tc::mma_f8(d, da, dq, kScIdesc, false);
                    tc::mma_f8(d, da + 2, dq + 2, kScIdesc, true);  // the second 32 dims (+32 bytes)
                    tc::commit(&dfull[tile & 1]);
                    if (last_of_box) tc::commit(&empty[slot]);
                }
                __syncwarp();
                last_commit = &dfull[tile & 1];
                last_parity = (uint32_t)((tile >> 1) & 1);
                if (last_of_box && issued < nbox) issue_box(issued++);
            }
            box += nbox;
        }
        if (!ok) {
            if (lane == 0) {
                raise_status(p.status, kDevTimeout);
                atomicExch(&s_fail, 1);
                for (int gb = (box > kScSlots ? box - kScSlots : 0); gb < box; ++gb)
                    mbar_wait(&full[gb % kScSlots], (uint32_t)((gb / kScSlots) & 1));
                if (last_commit) mbar_wait(last_commit, last_parity);
            }
            __syncwarp();
        }
    } else {
        // ---------------- epilogue warps: region r = 128 t + tid of the tile, every row
        int tile = 0;
        const float* w = s_w;
        for (int sq = 0; sq < nseq; ++sq) {
            const int b = s_seq[sq];
            const int nt = (pass_regions(b) + 127) >> 7;
            for (int t = 0; t < nt; ++t, ++tile) {
                const bool got = mbar_wait(&dfull[tile & 1], (uint32_t)((tile >> 1) & 1));
                if (!__all_sync(0xffffffffu, got && *reinterpret_cast<volatile int*>(&s_fail) == 0)) {
                    atomicExch(&s_fail, 1);
                    raise_status(p.status, kDevTimeout);
                    sq = nseq;
                    break;
                }
                tc::fence_after_sync();
                const int r = t * 128 + tid;
                const uint32_t base = tc::taddr(tmem, warp * 32, (uint32_t)(tile & 1) * kScCols);
#pragma unroll
                for (int c = 0; c < kScCols / 16; ++c) {  // 16 columns = 16 / HPG rows at a time
                    float dv[16];
                    tc::ld16(base + 16u * c, dv);
#pragma unroll
                    for (int jj = 0; jj < 16 / HPG; ++jj) {
                        const int j = c * (16 / HPG) + jj;
                        if (s_b[j] == b && r < s_R[j]) {
                            float sc = 0.0f;
#pragma unroll
                            for (int h = 0; h < HPG; ++h) sc = fmaf(fmaxf(dv[jj * HPG + h], 0.0f), w[j * HPG + h], sc);
                            p.scores[((int64_t)(n0 + j) * p.G + g) * p.r_cap + r] = __fadd_rn(sc, 0.0f);  // -0 -> +0
                        }
                    }
                }
                tc::fence_before_sync();
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&dempty[tile & 1])) : "memory");
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::dealloc(tmem, kScTmemCols);
}

template <int HPG>
cudaError_t score_tc_for(const ScoreParams& p, const CUtensorMap& smap, cudaStream_t stream, bool pdl) {
    static std::atomic<uint64_t> attr_set{0};
    cudaError_t e = once_per_device(attr_set, [] {
        return cudaFuncSetAttribute(score_tc_kernel<HPG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sc_smem_bytes());
    });
    if (e != cudaSuccess) return e;
    constexpr int NR = kScCols / HPG;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.N + NR - 1) / NR), (unsigned)p.G, 1);
    cfg.blockDim = dim3(kScThreads);
    cfg.dynamicSmemBytes = sc_smem_bytes();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, score_tc_kernel<HPG>, smap, p);
}

}  // namespace

cudaError_t launch_score_tc(const ScoreParams& p, const CUtensorMap& smap, cudaStream_t stream, bool pdl) {
    switch (p.hpg) {
        case 1: return score_tc_for<1>(p, smap, stream, pdl);
        case 2: return score_tc_for<2>(p, smap, stream, pdl);
        case 4: return score_tc_for<4>(p, smap, stream, pdl);
        case 8: return score_tc_for<8>(p, smap, stream, pdl);
    }
    return cudaErrorInvalidValue;
}

}  // namespace step5
