// noalloc.cu -- a variant of steps (2)+(3) whose scratch memory is a fixed array inside
// the library, for callers that cannot allocate device memory themselves.
//
// Some callers have no way to obtain a workspace: for example code that runs inside a
// host framework which owns every device allocation, or a path that must not call
// cudaMalloc at all (no allocator is reachable, or allocating there would synchronise
// the device).  For them, step5_index_score_topk_noalloc takes the same inputs and
// outputs as step5_index_score_topk but keeps the scratch (score list, histograms,
// candidate lists) in kNoallocScratchBytes of static device memory that the library
// owns for as long as it is loaded.
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "step5_sparse_attn.h"

namespace step5 {
namespace {

// 4 MiB for steps (2)-(3), after the space a workspace keeps for step (4)
constexpr size_t kNoallocScratchBytes = ((size_t)4 << 20) + kAttnAreaMaxBytes;

// The scratch array: one copy on every device that loads the library, held until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of the array on the current device.  Looked up on every call (a
// cached address would go stale if the device's context were torn down and created
// again in this process); the lookup is cheap next to the memset that follows.
void* scratch_address(cudaError_t* err) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    return *err == cudaSuccess ? p : nullptr;
}

}  // namespace
}  // namespace step5

extern "C" step5_status step5_index_score_topk_noalloc(
    const step5_geometry* geom, int32_t N, int32_t B, int32_t t_cap, int32_t r_cap, const void* idx_q_bf16,
    const float* w, const int32_t* row_seq, const int32_t* row_pos, const void* rope_cos_bf16,
    const void* rope_sin_bf16, const uint8_t* summaries_e4m3, int32_t* sel_ids, int32_t* sel_count,
    float* scores_or_null, float* sel_scores_or_null, step5_stream_t stream) {
    using namespace step5;
    const size_t need = step5_workspace_bytes(geom, N, r_cap);
    if (need == 0) return geom == nullptr || N <= 0 || r_cap <= 0 ? STEP5_ERR_INVALID_ARGUMENT : STEP5_ERR_UNSUPPORTED;
    if (need > kNoallocScratchBytes) return STEP5_ERR_WORKSPACE;  // beyond the fixed scratch
    cudaError_t err = cudaSuccess;
    void* scratch = scratch_address(&err);
    if (scratch == nullptr) return STEP5_ERR_CUDA;
    // the array keeps whatever the previous call left (possibly another layout): the
    // part this call uses starts from zero
    if (cudaMemsetAsync(scratch, 0, need, (cudaStream_t)stream) != cudaSuccess) return STEP5_ERR_CUDA;
    return step5_index_score_topk(geom, N, B, t_cap, r_cap, idx_q_bf16, w, row_seq, row_pos, rope_cos_bf16,
                                  rope_sin_bf16, summaries_e4m3, sel_ids, sel_count, scores_or_null,
                                  sel_scores_or_null, scratch, kNoallocScratchBytes, stream);
}
