// attention_shard.cu -- step (4) on one sequence shard: the shard instantiation of the
// attention kernel (attention_kernel.cuh), in a translation unit of its own so that the
// whole-row kernel is compiled alone.  Keys outside the shard's tokens are skipped and
// each head's softmax state (m, l, o) is written instead of the output; the states of a
// row's shards combine into the output in shard.cu.
#include "attention_kernel.cuh"

namespace step5 {

cudaError_t launch_attention_shard(const AttnParams& p, int N, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                   cudaStream_t stream, bool pdl) {
    return launch_sparse_attn<true>(p, N, kmap, vmap, stream, pdl);
}

}  // namespace step5
