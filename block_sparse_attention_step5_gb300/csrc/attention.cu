// attention.cu -- step (4): the whole-row instantiation of the attention kernel
// (attention_kernel.cuh holds the kernel and its design notes), compiled in a
// translation unit of its own; attention_shard.cu holds the shard instantiation.
#include "attention_kernel.cuh"

namespace step5 {

size_t attention_smem_bytes() { return attn_smem_bytes(); }

cudaError_t launch_attention(const AttnParams& p, int N, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream, bool pdl) {
    return launch_sparse_attn<false>(p, N, kmap, vmap, stream, pdl);
}

}  // namespace step5
