// qmm_mma_inst_grp.cu -- tensor-core kernel instances of the expert-grouped
// N-token product (x split, GGUF formats).
#include "qmm_mma_kernel.cuh"

namespace qmm {

QMM_MMA_INSTANTIATE_GROUPED(F_BF16);
QMM_MMA_INSTANTIATE_GROUPED(F_F16);
QMM_MMA_INSTANTIATE_GROUPED(F_Q4_0);
QMM_MMA_INSTANTIATE_GROUPED(F_Q4_K);
QMM_MMA_INSTANTIATE_GROUPED(F_Q6_K);
QMM_MMA_INSTANTIATE_GROUPED(F_Q8_0);
QMM_MMA_INSTANTIATE_GROUPED(F_Q5_0);

}  // namespace qmm
