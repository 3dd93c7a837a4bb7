// qmm_mma_inst_q.cu -- tensor-core kernel instances for Q6_K, Q8_0 and Q5_0.
#include "qmm_mma_kernel.cuh"

namespace qmm {

QMM_MMA_INSTANTIATE(F_Q6_K);
QMM_MMA_INSTANTIATE(F_Q8_0);
QMM_MMA_INSTANTIATE(F_Q5_0);

}  // namespace qmm
