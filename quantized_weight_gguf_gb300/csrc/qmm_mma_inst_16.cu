// qmm_mma_inst_16.cu -- tensor-core kernel instances for BF16, F16 and Q4_0.
#include "qmm_mma_kernel.cuh"

namespace qmm {

QMM_MMA_INSTANTIATE(F_BF16);
QMM_MMA_INSTANTIATE(F_F16);
QMM_MMA_INSTANTIATE(F_Q4_0);

}  // namespace qmm
