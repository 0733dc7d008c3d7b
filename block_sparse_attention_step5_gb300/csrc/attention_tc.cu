// attention_tc.cu -- step (4) on the tcgen05 tensor cores: attention over the picked regions
// plus the row's own region, one CTA per (row, KV group), for launches with many
// (row, group) pairs (prefill chunks, large decode batches).
//
// "Step-5-Preview on one 256 GB Mac" (TensorFold PR #903), CSA-indexer commit: each row
// attends to its picked regions plus its own region; with at most 512 regions that is the
// dense attention the indexer replaces.  The same page's prompt-chunk kernel puts the
// group's query heads on the tensor units against a block of gathered keys; here the
// gathered keys are the M side instead, so that the M = 128 tile of the tensor core is
// filled by keys and the group's 4-16 query heads are the N = 16 side:
//
//   S^T [128 keys x 16 heads]  = K_tile [128 x 128 dims]  . Q^T          (TMEM cols  0-31, two buffers)
//   O^T [128 dims x 16 heads] += V_tile^T [128 dims x 128] . P^T [128 x 16]  (TMEM cols 32-47)
//
// A tile is 16 regions (128 keys).  Each region's K (and V) is one 2 KB TMA box of the
// cache's 3-D map, landing as two 128-byte-swizzled 1 KB halves [half][token][64 dims]:
// as the A operand of the first product that is a K-major tile (8-row groups 2 KB
// apart, the second 64 dims 1 KB in), and as the A operand of the second an MN-major
// tile (64-dim blocks 1 KB apart, 8-token groups 2 KB apart), so neither needs a copy.
// The softmax runs with one thread per key (the TMEM lane of its row): per-head maxima
// over the tile through warp shuffles, a running maximum that is only moved (and O
// rescaled in TMEM) when a tile's maximum exceeds it by more than 2^8, P rounded to bf16
// into shared memory as the second product's B operand (MN-major, no swizzle), and the
// row sums kept per thread until the end.  A fifth warp issues the MMAs (lane 0) and a
// sixth the copies (16 lanes, one region box each; a CTA's TMA issue stalls once its
// copies in flight reach its rate, which must not hold up the MMAs); three 32 KB slots
// hold the copies in flight, K running a tile ahead of V (K_0, K_1, V_0, K_2, V_1, ...),
// and mbarriers hand over between the stages (copy landed, slot free again, S ready,
// P ready, second product done).  ~112 KB of shared memory and 64 TMEM columns per CTA leave room
// for two CTAs per SM: one CTA's TMA gathers from L2 run at about half the rate that two
// CTAs reach on an SM.
#include "tcgen05.cuh"
#include "kernels.cuh"

namespace step5 {

namespace {

constexpr int kTcSoftmaxWarps = 4;                   // one thread per key of a tile
constexpr int kTcSoftmaxThreads = kTcSoftmaxWarps * 32;
constexpr int kTcMmaWarp = kTcSoftmaxWarps;           // issues the MMAs (lane 0)
constexpr int kTcLoadWarp = kTcSoftmaxWarps + 1;      // first of the warps issuing the copies
constexpr int kTcLoadWarps = 2;                       // each issues 8 of a tile's 16 boxes
constexpr int kTcThreads = kTcSoftmaxThreads + 32 + 32 * kTcLoadWarps;
constexpr int kTcTileRegions = 16;
constexpr int kTcSlots = 3;
constexpr uint32_t kTcSlotBytes = kTcTileRegions * 2048;
constexpr uint32_t kTcQBytes = 4096;   // B of the first product: 16 head rows x 256 B
constexpr uint32_t kTcPBytes = 4096;   // B of the second product: 128 keys x 16 heads bf16
constexpr uint32_t kTcCols = 64;       // S (2 x 16 columns), O (16 columns)
constexpr float kTcSlack = 8.0f;       // log2 units the running maximum may trail a tile's

constexpr uint32_t kIdesc1 = tc::instr_desc(tc::kFmtBF16, false, false, 128, 16);
constexpr uint32_t kIdesc2 = tc::instr_desc(tc::kFmtBF16, true, true, 128, 16);

size_t tc_smem_bytes(int top_k) {
    return 1024 + (size_t)kTcSlots * kTcSlotBytes + kTcQBytes + 2 * kTcPBytes + (((size_t)(top_k + 2) * 4 + 15) & ~(size_t)15);
}

// Reduction of NV values per lane (NV a power of two <= 32) over the warp with one
// shuffle per value halving: each stage splits the values between the two lanes of a
// pair (the lane with the stage's bit set keeps the upper half), so that after log2(NV)
// stages every lane holds one value, reduced over the lanes that differ in those bits,
// and the remaining stages reduce it over the other lanes.  *idx receives the index of
// the value the lane holds; the lanes (lane & (32 / NV - 1)) == 0 hold each index once.
template <int NV, int M, class Op>
__device__ __forceinline__ float xpose_reduce(float* w, int lane, int* idx, Op op) {
    if constexpr (M == 0) {
        return w[0];
    } else if constexpr (NV > 1) {
        const bool up = (lane & M) != 0;
#pragma unroll
        for (int j = 0; j < NV / 2; ++j) {
            const float send = up ? w[j] : w[j + NV / 2];
            const float keep = up ? w[j + NV / 2] : w[j];
            w[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, M));
        }
        if (up) *idx += NV / 2;
        return xpose_reduce<NV / 2, M / 2>(w, lane, idx, op);
    } else {
        w[0] = op(w[0], __shfl_xor_sync(0xffffffffu, w[0], M));
        return xpose_reduce<1, M / 2>(w, lane, idx, op);
    }
}
struct MaxOp {
    __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct AddOp {
    __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};

// Barrier 1 over the softmax warps only, returning whether any of them passed `v`.
__device__ __forceinline__ bool softmax_sync_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "n"(kTcSoftmaxThreads)
        : "memory");
    return r != 0;
}

template <int HQ>
__global__ void __launch_bounds__(kTcThreads) sparse_attn_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                     const __grid_constant__ CUtensorMap vmap,
                                                                     AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem(smem_raw, 1024);
    uint8_t* slots = smem;
    uint8_t* qt = smem + kTcSlots * kTcSlotBytes;
    uint8_t* pt = qt + kTcQBytes;  // two P buffers
    int32_t* s_ids = reinterpret_cast<int32_t*>(pt + 2 * kTcPBytes);
    __shared__ __align__(8) uint64_t full[kTcSlots], empty[kTcSlots], sbar[2], obar[2], pbar[2];
    __shared__ uint32_t s_tmem;
    __shared__ float red[2][4][16];
    __shared__ int s_fail;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = blockIdx.x, g = blockIdx.y;  // rows first: CTAs that run together share a group's cache
    const int64_t ng = (int64_t)n * p.G + g;
    constexpr int hq_g = HQ;

    if (tid == 0) {
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
        for (int s = 0; s < kTcSlots; ++s) {
            mbar_init(&full[s], kTcLoadWarps);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sbar[s], 1);
            mbar_init(&obar[s], 1);
            mbar_init(&pbar[s], kTcSoftmaxThreads);
        }
        fence_mbar_init();
        s_fail = 0;
    }
    if (warp == 0) tc::alloc(&s_tmem, kTcCols);
    // unloaded regions of a tile (invalid ids, entries past the list) keep what the slot
    // held before: zero it once so that it is finite (their P is zero)
    for (int i = tid; i < (int)(kTcSlots * kTcSlotBytes / 16); i += kTcThreads)
        reinterpret_cast<uint4*>(slots)[i] = make_uint4(0, 0, 0, 0);
    pdl_wait();
    pdl_launch_dependents();

    const int b = p.row_seq[n];
    const int pos = p.row_pos[n];
    int cnt = p.sel_count[ng];
    const int32_t* ids = p.sel_ids + ng * p.top_k;
    for (int i = tid; i < p.top_k; i += kTcThreads) s_ids[i] = __ldg(ids + i);
    // the group's query heads as the B operand of S^T (rows >= hq_g zero), K-major with
    // 128-byte swizzle: [half][16 rows][64 dims]
    {
        const uint16_t* qb = p.q + ((int64_t)n * p.Hq + (int64_t)g * hq_g) * 128;
        for (int i = tid; i < 256; i += kTcThreads) {
            const int r = i >> 4, c16 = i & 15, half = c16 >> 3, c = c16 & 7;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < hq_g) v = *reinterpret_cast<const uint4*>(qb + r * 128 + c16 * 8);
            *reinterpret_cast<uint4*>(qt + half * 2048 + r * 128 + ((c ^ (r & 7)) << 4)) = v;
        }
    }
    fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;

    const bool row_ok = !(b < 0 || b >= p.B || pos < 0 || pos >= p.t_cap);
    if (!row_ok) {
        if (tid == 0) raise_status(p.status, kDevRange);
        const int64_t h0 = (int64_t)n * p.Hq + (int64_t)g * hq_g;
        for (int i = tid; i < hq_g * 128; i += kTcThreads) p.out[h0 * 128 + i] = 0;
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 0) tc::dealloc(tmem, kTcCols);
        return;
    }
    if (cnt < 0 || cnt > p.top_k) {
        if (tid == 0) raise_status(p.status, kDevRange);
        cnt = cnt < 0 ? 0 : p.top_k;
    }
    const int own = pos >> 3;
    const int own_tokens = pos - own * 8 + 1;
    const int E = cnt + 1;
    const int ntiles = (E + kTcTileRegions - 1) / kTcTileRegions;
    const int64_t row_base = ((int64_t)b * p.G + g) * p.t_cap;

    // entry e -> (region, tokens): picked regions in selection order, then the own
    // region; invalid ids and entries past the list take no tokens
    auto entry = [&](int e, int& rid) -> int {
        rid = -1;
        if (e >= E) return 0;
        if (e == cnt) {
            rid = own;
            return own_tokens;
        }
        const int r = s_ids[e];
        if (r < 0 || r >= own) return 0;
        rid = r;
        return 8;
    };

    // Load items, in the order the slots are filled: K_0, K_1, V_0, K_2, V_1, K_3, ...
    // (K runs a tile ahead of V, so that each copy has a tile or more of the loop to
    // land): item 0 = K_0; odd j = K_(j+1)/2; even j >= 2 = V_(j-2)/2.  Item j reuses the
    // slot of item j - 3 once the product that read that item is done.  The one item
    // number without a tile (K_ntiles) is skipped.
    const int last_item = 2 * ntiles;
    auto item_of_k = [](int i) { return i == 0 ? 0 : 2 * i - 1; };
    auto item_of_v = [](int i) { return 2 * i + 2; };

    bool failed = false;
    auto item_tile = [&](int j, bool& isv) -> int {
        if (j == 0) {
            isv = false;
            return 0;
        }
        isv = !(j & 1);
        return (j & 1) ? (j + 1) >> 1 : (j - 2) >> 1;
    };
    if (warp >= kTcLoadWarp) {
        // ---------------- load warps: every item in order, each into its slot once the
        // product that read the slot's previous item is done; load warp lw issues boxes
        // 8 lw .. 8 lw + 7 of each tile (one per lane), so that a tile's copies are issued
        // by two warps at once
        constexpr int per = kTcTileRegions / kTcLoadWarps;
        const int lw = warp - kTcLoadWarp;
        bool ok = true;
        int j = 0;
        for (; j <= last_item && ok; ++j) {
            bool isv;
            const int tile = item_tile(j, isv);
            if (tile >= ntiles) continue;  // the skipped number
            const int slot = j % kTcSlots, use = j / kTcSlots;
            if (use > 0 && !mbar_wait(&empty[slot], (uint32_t)((use - 1) & 1))) {
                ok = false;
                break;
            }
            if (*reinterpret_cast<volatile int*>(&s_fail) != 0) {
                ok = false;
                break;
            }
            int rid = -1;
            const int q = lw * per + lane;  // the tile entry this lane copies
            const int ntok = lane < per ? entry(tile * kTcTileRegions + q, rid) : 0;
            const uint32_t have = __ballot_sync(0xffffffffu, ntok > 0);
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)__popc(have) * 2048u);
            __syncwarp();
            if (ntok > 0)
                tma_load_3d(slots + slot * kTcSlotBytes + q * 2048, isv ? &vmap : &kmap, &full[slot], 0,
                            (int)(row_base + (int64_t)rid * 8), 0);
        }
        if (!ok && lane == 0) {
            // a wait gave up: let the copies issued land (bounded) before the CTA's shared
            // memory goes away
            raise_status(p.status, kDevTimeout);
            atomicExch(&s_fail, 1);
            for (int k = (j > kTcSlots ? j - kTcSlots : 0); k < j; ++k) {
                bool isv;
                if (item_tile(k, isv) < ntiles) mbar_wait(&full[k % kTcSlots], (uint32_t)((k / kTcSlots) & 1));
            }
        }
        __syncwarp();
    } else if (warp == kTcMmaWarp) {
        // ---------------- MMA warp: lane 0 issues both products of every tile
        const uint32_t slot_addr = smem_u32(slots), p_addr = smem_u32(pt);
        // descriptors at offset 0; an MMA's start address is added in 16-byte units
        const uint64_t dq = tc::smem_desc(smem_u32(qt), 16, 1024, tc::kSwizzle128);
        bool ok = true;
        uint64_t* last_commit = nullptr;
        uint32_t last_parity = 0;
        auto mma1 = [&](int i) {
            const int j = item_of_k(i), slot = j % kTcSlots;
            if (!ok || !mbar_wait(&full[slot], (uint32_t)((j / kTcSlots) & 1))) {
                ok = false;
                return;
            }
            tc::fence_after_sync();
            if (lane == 0) {
                const uint64_t da = tc::smem_desc(slot_addr + slot * kTcSlotBytes, 16, 2048, tc::kSwizzle128);
                const uint32_t d = tmem + 16u * (i & 1);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t ka = k < 4 ? 32u * k : 1024u + 32u * (k - 4);
                    const uint32_t kb = k < 4 ? 32u * k : 2048u + 32u * (k - 4);
                    tc::mma_f16(d, da + (ka >> 4), dq + (kb >> 4), kIdesc1, k > 0);
                }
                tc::commit(&sbar[i & 1]);
                tc::commit(&empty[slot]);
            }
            __syncwarp();
            last_commit = &empty[slot];
            last_parity = (uint32_t)((j / kTcSlots) & 1);
        };
        auto mma2 = [&](int i) {
            const int j = item_of_v(i), slot = j % kTcSlots;
            if (!ok || !mbar_wait(&full[slot], (uint32_t)((j / kTcSlots) & 1))) {
                ok = false;
                return;
            }
            tc::fence_after_sync();
            if (lane == 0) {
                const uint64_t da = tc::smem_desc(slot_addr + slot * kTcSlotBytes, 1024, 2048, tc::kSwizzle128);
                const uint64_t db = tc::smem_desc(p_addr + (uint32_t)(i & 1) * kTcPBytes, 256, 128, tc::kSwizzleNone);
                // K steps of 16 keys (two regions); steps past the tile's entries add nothing
                const int nent = min(kTcTileRegions, E - i * kTcTileRegions);
                const int nsteps = (nent + 1) >> 1;
                for (int st = 0; st < nsteps; ++st)
                    tc::mma_f16(tmem + 32u, da + 256u * st, db + 32u * st, kIdesc2, i > 0 || st > 0);
                tc::commit(&obar[i & 1]);
                tc::commit(&empty[slot]);
            }
            __syncwarp();
            last_commit = &empty[slot];
            last_parity = (uint32_t)((j / kTcSlots) & 1);
        };
        mma1(0);
        for (int i = 0; i < ntiles && ok; ++i) {
            if (i + 1 < ntiles) mma1(i + 1);
            // the softmax of tile i is done: P_i written, O rescaled, S_i read
            if (ok && !mbar_wait(&pbar[i & 1], (uint32_t)((i >> 1) & 1))) ok = false;
            if (*reinterpret_cast<volatile int*>(&s_fail) != 0) ok = false;
            if (!ok) break;
            mma2(i);
        }
        if (!ok) {
            if (lane == 0) {
                raise_status(p.status, kDevTimeout);
                atomicExch(&s_fail, 1);
                if (last_commit) mbar_wait(last_commit, last_parity);
            }
            __syncwarp();
        }
    } else {
        // ---------------- softmax warps: one key per thread (its TMEM lane)
        float m_ref[HQ], l_part[HQ];
#pragma unroll
        for (int h = 0; h < HQ; ++h) {
            m_ref[h] = -INFINITY;
            l_part[h] = 0.0f;
        }
        const int my_q = tid >> 3, my_t = tid & 7;
        constexpr int kWriterMask = 32 / HQ - 1;  // lanes (lane & mask) == 0 hold each head once
        for (int i = 0; i < ntiles; ++i) {
            bool w_ok = mbar_wait(&sbar[i & 1], (uint32_t)((i >> 1) & 1));
            tc::fence_after_sync();
            float s[16];
            tc::ld16(tc::taddr(tmem, warp * 32, 16u * (i & 1)), s);
            int rid;
            const bool valid = my_t < entry(i * kTcTileRegions + my_q, rid);
            float w[HQ];
#pragma unroll
            for (int h = 0; h < HQ; ++h) {
                s[h] = valid ? s[h] * p.scale_log2 : -INFINITY;
                w[h] = s[h];
            }
            // tile maxima per head: over the warp, then over the four warps
            int hidx = 0;
            const float wmax = xpose_reduce<HQ, 16>(w, lane, &hidx, MaxOp{});
            float(&rd)[4][16] = red[i & 1];
            if ((lane & kWriterMask) == 0) rd[warp][hidx] = wmax;
            if (softmax_sync_or(!w_ok || *reinterpret_cast<volatile int*>(&s_fail) != 0)) {
                if (!w_ok) raise_status(p.status, kDevTimeout);
                failed = true;
                break;
            }
            // running maxima move only when a tile's maximum passes them by more than the
            // slack (then l and O are rescaled by alpha); every thread takes the same steps
            bool resc = false;
            float alpha[HQ];
#pragma unroll
            for (int h = 0; h < HQ; ++h) {
                const float tmax = fmaxf(fmaxf(rd[0][h], rd[1][h]), fmaxf(rd[2][h], rd[3][h]));
                const bool move = tmax > m_ref[h] + kTcSlack || (m_ref[h] == -INFINITY && tmax > -INFINITY);
                const float m_new = move ? tmax : m_ref[h];
                alpha[h] = (move && m_ref[h] != -INFINITY) ? exp2f(m_ref[h] - m_new) : (move ? 0.0f : 1.0f);
                m_ref[h] = m_new;
                resc |= move;
            }
            uint32_t pw[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) pw[k] = 0u;
#pragma unroll
            for (int h = 0; h < HQ; h += 2) {
                const float p0 = s[h] == -INFINITY ? 0.0f : exp2f(s[h] - m_ref[h]);
                const float p1 = s[h + 1] == -INFINITY ? 0.0f : exp2f(s[h + 1] - m_ref[h + 1]);
                l_part[h] = l_part[h] * alpha[h] + p0;
                l_part[h + 1] = l_part[h + 1] * alpha[h + 1] + p1;
                pw[h >> 1] = pack_bf16x2(p0, p1);
            }
            // the P buffer of this tile was last read by the second product two tiles back
            if (i >= 2) w_ok &= mbar_wait(&obar[i & 1], (uint32_t)(((i >> 1) - 1) & 1));
            uint8_t* pb = pt + (i & 1) * kTcPBytes + (tid >> 3) * 256 + (tid & 7) * 16;
            *reinterpret_cast<uint4*>(pb) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
            *reinterpret_cast<uint4*>(pb + 128) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
            // O rescale (after the previous second product), one TMEM lane per output dim
            if (resc && i > 0) {
                w_ok &= mbar_wait(&obar[(i - 1) & 1], (uint32_t)(((i - 1) >> 1) & 1));
                tc::fence_after_sync();
                float o[16];
                tc::ld16(tc::taddr(tmem, warp * 32, 32), o);
#pragma unroll
                for (int h = 0; h < HQ; ++h) o[h] *= alpha[h];
                tc::st16(tc::taddr(tmem, warp * 32, 32), o);
            }
            // the own region's tokens past the row's position: their V rows are zeroed (the
            // cache may hold anything there, and a zero weight must meet a finite value)
            const int own_q = cnt - i * kTcTileRegions;
            if (own_q >= 0 && own_q < kTcTileRegions && own_tokens < 8) {
                const int j = item_of_v(i), slot = j % kTcSlots;
                w_ok &= mbar_wait(&full[slot], (uint32_t)((j / kTcSlots) & 1));
                uint8_t* reg = slots + slot * kTcSlotBytes + own_q * 2048;
                const int half = tid >> 6, t = (tid >> 3) & 7, c = tid & 7;  // 128 (half, token, chunk)s
                if (t >= own_tokens) *reinterpret_cast<uint4*>(reg + half * 1024 + t * 128 + c * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async();
            tc::fence_before_sync();
            if (!w_ok) {
                raise_status(p.status, kDevTimeout);
                atomicExch(&s_fail, 1);
            }
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&pbar[i & 1])) : "memory");
        }
        if (!failed) {
            const int il = ntiles - 1;
            const bool w_ok = mbar_wait(&obar[il & 1], (uint32_t)((il >> 1) & 1));
            if (!w_ok) raise_status(p.status, kDevTimeout);
            tc::fence_after_sync();
            // row sums, then out = O / l (one thread per output dim)
            float(&rd)[4][16] = red[ntiles & 1];
            int hidx = 0;
            const float wsum = xpose_reduce<HQ, 16>(l_part, lane, &hidx, AddOp{});
            if ((lane & kWriterMask) == 0) rd[warp][hidx] = wsum;
            if (!softmax_sync_or(!w_ok || *reinterpret_cast<volatile int*>(&s_fail) != 0)) {
                float o[16];
                tc::ld16(tc::taddr(tmem, warp * 32, 32), o);
                const int64_t h0 = (int64_t)n * p.Hq + (int64_t)g * hq_g;
#pragma unroll
                for (int h = 0; h < HQ; ++h) {
                    const float L = (rd[0][h] + rd[1][h]) + (rd[2][h] + rd[3][h]);
                    float gf = 1.0f;
                    if (p.gate != nullptr) gf = 1.0f / (1.0f + expf(-bf16_to_f32(p.gate[h0 + h])));
                    p.out[(h0 + h) * 128 + tid] = f32_to_bf16_bits(o[h] / L * gf);
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::dealloc(tmem, kTcCols);
}

template <class K>
cudaError_t set_tc_attributes(K kernel) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem_bytes(kMaxTopK));
    if (e != cudaSuccess) return e;
    // all of the SM's unified memory as shared memory, so that two CTAs fit
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
}

}  // namespace

size_t attention_tc_smem_bytes(int top_k) { return tc_smem_bytes(top_k); }

cudaError_t launch_attention_tc(const AttnParams& p, int N, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                cudaStream_t stream, bool pdl) {
    static std::atomic<uint64_t> attr_set{0};
    cudaError_t e = once_per_device(attr_set, [] {
        cudaError_t e1 = set_tc_attributes(sparse_attn_tc_kernel<4>);
        if (e1 == cudaSuccess) e1 = set_tc_attributes(sparse_attn_tc_kernel<8>);
        if (e1 == cudaSuccess) e1 = set_tc_attributes(sparse_attn_tc_kernel<16>);
        return e1;
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)N, (unsigned)p.G, 1);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = tc_smem_bytes(p.top_k);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    switch (p.hq_g) {
        case 4: return cudaLaunchKernelEx(&cfg, sparse_attn_tc_kernel<4>, kmap, vmap, p);
        case 8: return cudaLaunchKernelEx(&cfg, sparse_attn_tc_kernel<8>, kmap, vmap, p);
        case 16: return cudaLaunchKernelEx(&cfg, sparse_attn_tc_kernel<16>, kmap, vmap, p);
    }
    return cudaErrorInvalidValue;
}

}  // namespace step5
