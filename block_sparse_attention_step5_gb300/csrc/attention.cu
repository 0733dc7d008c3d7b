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

cudaError_t launch_attention_cluster(const AttnParams& p, int N, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                     cudaStream_t stream, bool pdl) {
    return launch_sparse_attn<false, true>(p, N, kmap, vmap, stream, pdl);
}

int attention_max_clusters(int splits) {
    // how many clusters of `splits` blocks (one block per SM at this shared-memory size)
    // the GPCs hold at once; asked once per (device, size)
    static std::atomic<int> cached[64][kAttnMaxCluster + 1];
    if (splits < 2 || splits > kAttnMaxCluster) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int have = cached[dev][splits].load(std::memory_order_acquire);
    if (have != 0) return have - 1;  // stored plus one (0 = not asked yet)
    auto kern = sparse_attn_kernel<false, true>;
    int n = 0;
    bool ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem_bytes(true)) ==
                  cudaSuccess &&
              cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    if (ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)splits, 1, 1);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = attn_smem_bytes(true);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)splits;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    (void)cudaGetLastError();
    cached[dev][splits].store(n + 1, std::memory_order_release);
    return n;
}

}  // namespace step5
