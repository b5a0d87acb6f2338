// Selects the tensor-core kernel instantiation for a tile width.
#include "gemm_tc.cuh"

namespace dg {

extern template cudaError_t launch_gemm_tc_bn<64>(const CUtensorMap&, const CUtensorMap&,
                                                  const CUtensorMap&, const TcParams&, int,
                                                  cudaStream_t);
extern template cudaError_t launch_gemm_tc_bn<128>(const CUtensorMap&, const CUtensorMap&,
                                                   const CUtensorMap&, const TcParams&, int,
                                                   cudaStream_t);
extern template cudaError_t launch_gemm_tc_bn<256>(const CUtensorMap&, const CUtensorMap&,
                                                   const CUtensorMap&, const TcParams&, int,
                                                   cudaStream_t);

int tc_smem_bytes(int bn) {
  switch (bn) {
    case 64: return TcCfg<64>::SMEM_BYTES;
    case 128: return TcCfg<128>::SMEM_BYTES;
    case 256: return TcCfg<256>::SMEM_BYTES;
    default: return -1;
  }
}

int tc_stages(int bn) {
  switch (bn) {
    case 64: return TcCfg<64>::STAGES;
    case 128: return TcCfg<128>::STAGES;
    case 256: return TcCfg<256>::STAGES;
    default: return -1;
  }
}

cudaError_t launch_gemm_tc(int bn, const CUtensorMap& a, const CUtensorMap& b,
                           const CUtensorMap& c, const TcParams& p, int grid, cudaStream_t s) {
  switch (bn) {
    case 64: return launch_gemm_tc_bn<64>(a, b, c, p, grid, s);
    case 128: return launch_gemm_tc_bn<128>(a, b, c, p, grid, s);
    case 256: return launch_gemm_tc_bn<256>(a, b, c, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dg
