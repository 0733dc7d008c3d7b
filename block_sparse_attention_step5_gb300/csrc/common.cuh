// common.cuh -- device helpers shared by the sm_103a kernels of libstep5sa.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace step5 {

// ---------------------------------------------------------------------------------
// Phase trace (build with -DSTEP5_TRACE -rdc=true): thread 0 of each block records
// %globaltimer at numbered points into a buffer registered by step5_trace_buffer():
// trace[((kernel * 4096) + block) * 16 + point].  Compiles to nothing otherwise.
// ---------------------------------------------------------------------------------
#ifdef STEP5_TRACE
extern __device__ unsigned long long* g_trace;
#define STEP5_STAMP(kernel_id, point)                                                            \
    do {                                                                                         \
        if (threadIdx.x == 0 && g_trace) {                                                       \
            const unsigned long long bl_ =                                                       \
                blockIdx.x + (unsigned long long)gridDim.x * (blockIdx.y + (unsigned long long)gridDim.y * blockIdx.z); \
            unsigned long long t_;                                                               \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                               \
            if (bl_ < 4096) g_trace[((kernel_id) * 4096ull + bl_) * 16 + (point)] = t_;         \
        }                                                                                        \
    } while (0)
// Records the SM of the block (plus one) at `point` instead of a time.
#define STEP5_SMID(kernel_id, point)                                                             \
    do {                                                                                         \
        if (threadIdx.x == 0 && g_trace) {                                                       \
            uint32_t sm_;                                                                        \
            asm volatile("mov.u32 %0, %%smid;" : "=r"(sm_));                                     \
            if (blockIdx.x < 4096) g_trace[((kernel_id) * 4096ull + blockIdx.x) * 16 + (point)] = sm_ + 1; \
        }                                                                                        \
    } while (0)
// Records a value (plus one) at `point` instead of a time.
#define STEP5_VALUE(kernel_id, point, value)                                                     \
    do {                                                                                         \
        if (threadIdx.x == 0 && g_trace && blockIdx.x < 4096)                                    \
            g_trace[((kernel_id) * 4096ull + blockIdx.x) * 16 + (point)] = (unsigned long long)(value) + 1; \
    } while (0)
#else
#define STEP5_VALUE(kernel_id, point, value) \
    do {                                     \
    } while (0)
#define STEP5_STAMP(kernel_id, point) \
    do {                              \
    } while (0)
#define STEP5_SMID(kernel_id, point) \
    do {                             \
    } while (0)
#endif

constexpr uint32_t kDevRange = 1u;
constexpr uint32_t kDevTimeout = 2u;

// Bounded spin for mbarrier waits: ~2^26 polls (seconds), far beyond any copy latency.
constexpr uint32_t kSpinLimit = 1u << 26;

__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bit) {
    atomicOr(status, bit);
}

// ---------------------------------------------------------------------------------
// bf16 / e4m3 conversions
// ---------------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

// fp32 -> bf16 bits, round to nearest even.
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
    __nv_bfloat16 b = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&b);
}

// bf16(exact a + b) for fp32 a, b whose sum is not representable in fp32: rounds the
// exact sum once.  The fp32 sum s is off by the TwoSum residual e; the only case where
// rounding s to bf16 differs from rounding a + b is s sitting exactly on a bf16 halfway
// point, and there the residual's sign says which way the exact sum lies.
__device__ __forceinline__ uint16_t bf16_of_exact_sum(float a, float b) {
    float s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    uint32_t u = __float_as_uint(s);
    if ((u & 0xffffu) == 0x8000u && e != 0.0f) {
        // move s off the halfway point toward the exact value
        bool away = (e > 0.0f) == (s > 0.0f);
        u = away ? u + 1u : u - 1u;
        s = __uint_as_float(u);
    }
    return f32_to_bf16_bits(s);
}

// NEOX pair rotation of bf16 values with bf16 cos/sin: returns bf16 bits of
// x1*c - x2*s (first = true) or x2*c + x1*s (first = false), rounded once.
// Products of two bf16 values are exact in fp32.
__device__ __forceinline__ uint16_t neox_rotate(float x_self, float x_partner, float c, float s,
                                                bool first) {
    float p_self = __fmul_rn(x_self, c);
    float p_part = __fmul_rn(x_partner, s);
    return first ? bf16_of_exact_sum(p_self, -p_part) : bf16_of_exact_sum(p_self, p_part);
}

// e4m3 code of an fp32 value (round to nearest even, saturate to +-448).
__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
    return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// Two e4m3 codes (low byte first) -> two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t two) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
    __half2 hh = *reinterpret_cast<__half2*>(&h);
    return __half22float2(hh);
}

// Order-preserving map of a float score to a key that sorts DEScending by score:
// smaller key = larger score.  -0 is mapped like +0.
__device__ __forceinline__ uint32_t desc_key(float score) {
    uint32_t u = __float_as_uint(score);
    if (u == 0x80000000u) u = 0u;
    uint32_t ordered = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ~ordered;
}

__device__ __forceinline__ float score_of_desc_key(uint32_t key) {
    uint32_t ordered = ~key;
    uint32_t u = (ordered & 0x80000000u) ? (ordered & 0x7fffffffu) : ~ordered;
    return __uint_as_float(u);
}

// ---------------------------------------------------------------------------------
// mbarrier / TMA (inline PTX)
// ---------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// p advanced to the next multiple of `align` (a power of two) bytes of the shared
// window.  The offset is added to p itself so that the compiler keeps knowing p points to
// shared memory (a round trip through an integer would turn its accesses generic).
__device__ __forceinline__ uint8_t* align_smem(uint8_t* p, uint32_t align) {
    const uint32_t a = smem_u32(p);
    return p + (((a + align - 1u) & ~(align - 1u)) - a);
}

// Waits for phase `parity` of the barrier; gives up after kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    uint32_t addr = smem_u32(bar);
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// As mbar_wait, but each poll may suspend the thread for up to hint_ns (it resumes when
// the phase completes), so waiting warps leave the issue slots to the others; gives up
// after kSpinLimit / 64 polls.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t addr = smem_u32(bar);
    for (uint32_t i = 0; i < kSpinLimit / 64; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(addr), "r"(parity), "r"(hint_ns)
            : "memory");
        if (done) return true;
    }
    return false;
}

// ---------------------------------------------------------------------------------
// Global-memory synchronisation between the blocks of one launch (all resident)
// ---------------------------------------------------------------------------------

constexpr uint32_t kBarrierPolls = 1u << 22;  // polls of a global wait before giving up

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* a) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}

// Relaxed (no ordering) load for polling; pair with fence_acquire_gpu once it succeeds.
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* a) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}

// Acquire side of a release store seen by an earlier relaxed load of this thread.
__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void st_release_u32(uint32_t* a, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

// A barrier word holds a generation number (high 16 bits) and the arrivals of the
// current barrier (low 16 bits): the last of nb arrivals clears the count and advances
// the generation with one release add, so the word never needs clearing.
constexpr uint32_t kArrivedLast = 0x80000000u;

// Arrival (acquire + release): the generation seen, or kArrivedLast for the last
// arrival (which has released the others).
__device__ __forceinline__ uint32_t arrive_gen(uint32_t* word, uint32_t nb) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(word) : "memory");
    if ((old & 0xffffu) == nb - 1u) {
        asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(word), "r"(0x10000u - nb) : "memory");
        return kArrivedLast;
    }
    return old >> 16;
}

// Waits until the generation of a barrier word differs from gen (kArrivedLast: no
// wait); false when the wait gives up after `polls` polls.
__device__ __forceinline__ bool wait_gen(const uint32_t* word, uint32_t gen, uint32_t polls = kBarrierPolls) {
    if (gen == kArrivedLast) return true;
    for (uint32_t it = 0; it < polls; ++it)
        if ((ld_relaxed_u32(word) >> 16) != gen) {
            fence_acquire_gpu();
            return true;
        }
    return false;
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, uint64_t* bar, int32_t x,
                                            int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 3-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, uint64_t* bar, int32_t x, int32_t y,
                                            int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// 1-D bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) into shared
// memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------------------------
// Warp-level tensor-core helpers (bf16 m16n8k16, fp32 accumulate)
// ---------------------------------------------------------------------------------

__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                            uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------------------------
// Thread-block clusters
// ---------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Full cluster barrier with release/acquire semantics on shared memory.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_cluster(uint32_t local_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// ---------------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------------

// Waits until the grids this launch depends on have completed and flushed memory.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next grid on the stream begin launching (its pdl_wait still waits for us).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace step5
