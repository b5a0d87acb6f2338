// Tensor-core GEMM kernel instantiated for 128-column output tiles.
#include "gemm_tc.cuh"

namespace dg {
template cudaError_t launch_gemm_tc_bn<128, false>(const CUtensorMap&, const CUtensorMap&,
                                                  const CUtensorMap&, const TcParams&, int, cudaStream_t);
template cudaError_t launch_gemm_tc_bn<128, true>(const CUtensorMap&, const CUtensorMap&,
                                                 const CUtensorMap&, const TcParams&, int, cudaStream_t);
template int max_pairs<128>();
}  // namespace dg
