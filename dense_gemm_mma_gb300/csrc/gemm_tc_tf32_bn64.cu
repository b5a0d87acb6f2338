// Tensor-core GEMM kernel with TF32 operands, 64-column output tiles.
#include "gemm_tc.cuh"

namespace dg {
template cudaError_t launch_gemm_tc_bn<64, TC_SOLO, true>(const CUtensorMap&, const CUtensorMap&,
                                                         const CUtensorMap&, const CUtensorMap&, const TcParams&,
                                                         int, cudaStream_t);
}  // namespace dg
