// qmm_mma_inst_q4k.cu -- tensor-core kernel instances for Q4_K (raw super-block tiles by TMA) and the cluster-count query.
#include "qmm_mma_kernel.cuh"

namespace qmm {

// Clusters of two CTAs (one CTA per SM) that can be resident at once: every
// instance of the kernel has the same footprint class, so one query serves all.
int mma_clusters(const DeviceInfo &dev) {
    static std::once_flag once;
    static int n = 0;
    std::call_once(once, [&] {
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(2 * (unsigned)(dev.sm_count / 2));
        q.blockDim = dim3(kMmaThreads);
        q.dynamicSmemBytes = MmaCfg<256, kRawBytes, kEpiStageBytes>::kSmem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        q.attrs = attr;
        q.numAttrs = 1;
        int v = 0;
        if (cudaFuncSetAttribute(mma_kernel<F_Q4_K, 256, 2>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)MmaCfg<256, kRawBytes, kEpiStageBytes>::kSmem) != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&v, mma_kernel<F_Q4_K, 256, 2>, &q) != cudaSuccess ||
            v <= 0) {
            (void)cudaGetLastError();
            v = dev.sm_count / 2;
        }
        n = v;
    });
    return n;
}

QMM_MMA_INSTANTIATE(F_Q4_K);

}  // namespace qmm
