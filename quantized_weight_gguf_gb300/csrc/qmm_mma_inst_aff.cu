// qmm_mma_inst_aff.cu -- tensor-core kernel instances for the MLX-style affine 4- and 8-bit formats.
#include "qmm_mma_kernel.cuh"

namespace qmm {

QMM_MMA_INSTANTIATE(F_AFF4);
QMM_MMA_INSTANTIATE(F_AFF8);

}  // namespace qmm
