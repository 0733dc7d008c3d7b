// attention.cu -- step (4): attention over the picked regions plus the row's own region
// (and, optionally, the per-head sigmoid output gate that follows it).
//
// "Step-5-Preview on one 256 GB Mac" (TensorFold PR #903), CSA-indexer commit:
// "attention over those regions and the row's own"; below 512 regions every region is
// read, which is the dense attention it replaces.  The same page's decode kernel splits
// a row's keys over many workers and merges their online-softmax states in a fixed
// order ("one simdgroup walking every key alone left decode waiting on loads").
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
#include "attention_kernel.cuh"

namespace step5 {

size_t attention_smem_bytes() { return attn_smem_bytes(); }

cudaError_t launch_attention(const AttnParams& p, int N, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream, bool pdl) {
    return launch_sparse_attn<false>(p, N, kmap, vmap, stream, pdl);
}

}  // namespace step5
