// Selects the tensor-core kernel instantiation for a tile shape.
#include "gemm_tc.cuh"

namespace dg {

#define DG_EXTERN(BN, PAIR)                                                                   \
  extern template cudaError_t launch_gemm_tc_bn<BN, PAIR>(const CUtensorMap&, const CUtensorMap&, \
                                                          const CUtensorMap&, const TcParams&, int, \
                                                          cudaStream_t);
DG_EXTERN(64, false)
DG_EXTERN(128, false)
DG_EXTERN(256, false)
DG_EXTERN(128, true)
DG_EXTERN(256, true)
#undef DG_EXTERN
extern template int max_pairs<128>();
extern template int max_pairs<256>();

int tc_smem_bytes(int bn, bool pair) {
  if (pair) return bn == 256 ? TcCfg<256, true>::SMEM_BYTES : (bn == 128 ? TcCfg<128, true>::SMEM_BYTES : -1);
  switch (bn) {
    case 64: return TcCfg<64>::SMEM_BYTES;
    case 128: return TcCfg<128>::SMEM_BYTES;
    case 256: return TcCfg<256>::SMEM_BYTES;
    default: return -1;
  }
}

int tc_stages(int bn, bool pair) {
  if (pair) return bn == 256 ? TcCfg<256, true>::STAGES : (bn == 128 ? TcCfg<128, true>::STAGES : -1);
  switch (bn) {
    case 64: return TcCfg<64>::STAGES;
    case 128: return TcCfg<128>::STAGES;
    case 256: return TcCfg<256>::STAGES;
    default: return -1;
  }
}

int tc_max_pairs(int bn) {
  if (bn == 256) return max_pairs<256>();
  if (bn == 128) return max_pairs<128>();
  return 0;
}

cudaError_t launch_gemm_tc(int bn, bool pair, const CUtensorMap& a, const CUtensorMap& b,
                           const CUtensorMap& c, const TcParams& p, int grid, cudaStream_t s) {
  if (pair) {
    if (bn == 256) return launch_gemm_tc_bn<256, true>(a, b, c, p, grid, s);
    if (bn == 128) return launch_gemm_tc_bn<128, true>(a, b, c, p, grid, s);
    return cudaErrorInvalidValue;
  }
  switch (bn) {
    case 64: return launch_gemm_tc_bn<64, false>(a, b, c, p, grid, s);
    case 128: return launch_gemm_tc_bn<128, false>(a, b, c, p, grid, s);
    case 256: return launch_gemm_tc_bn<256, false>(a, b, c, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dg
