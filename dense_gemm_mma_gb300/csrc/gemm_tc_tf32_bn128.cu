// Tensor-core GEMM kernel with TF32 operands, 128-column output tiles: one CTA
// per tile, a CTA pair per 256-row tile, and a K pair.
#include "gemm_tc.cuh"

namespace dg {
#define DG_INST(MODE)                                                                                  \
  template cudaError_t launch_gemm_tc_bn<128, MODE, true>(const CUtensorMap&, const CUtensorMap&,       \
                                                         const CUtensorMap&, const CUtensorMap&,       \
                                                         const TcParams&, int, cudaStream_t);
DG_INST(TC_SOLO)
DG_INST(TC_PAIR)
DG_INST(TC_KPAIR)
#undef DG_INST
}  // namespace dg
