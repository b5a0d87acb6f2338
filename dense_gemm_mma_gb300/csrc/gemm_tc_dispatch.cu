// Selects the tensor-core kernel instantiation for a tile shape and mode.
#include "gemm_tc.cuh"

namespace dg {

#define DG_EXTERN(BN, MODE, TF32)                                                                    \
  extern template cudaError_t launch_gemm_tc_bn<BN, MODE, TF32>(const CUtensorMap&, const CUtensorMap&, \
                                                                const CUtensorMap&, const CUtensorMap&, \
                                                                const TcParams&, int, cudaStream_t);
#define DG_EXTERN_BOTH(BN, MODE) DG_EXTERN(BN, MODE, false) DG_EXTERN(BN, MODE, true)
DG_EXTERN_BOTH(64, TC_SOLO)
DG_EXTERN_BOTH(128, TC_SOLO)
DG_EXTERN_BOTH(256, TC_SOLO)
DG_EXTERN_BOTH(128, TC_PAIR)
DG_EXTERN_BOTH(256, TC_PAIR)
DG_EXTERN_BOTH(128, TC_KPAIR)
DG_EXTERN_BOTH(256, TC_KPAIR)
#undef DG_EXTERN_BOTH
#undef DG_EXTERN
extern template int max_clusters<128, TC_PAIR>();
extern template int max_clusters<256, TC_PAIR>();
extern template int max_clusters<128, TC_KPAIR>();
extern template int max_clusters<256, TC_KPAIR>();

namespace {
template <int MODE>
int cfg_value(int bn, bool stages) {
  if (bn == 128) return stages ? TcCfg<128, MODE>::STAGES : TcCfg<128, MODE>::SMEM_BYTES;
  if (bn == 256) return stages ? TcCfg<256, MODE>::STAGES : TcCfg<256, MODE>::SMEM_BYTES;
  if (bn == 64 && MODE == TC_SOLO) return stages ? TcCfg<64>::STAGES : TcCfg<64>::SMEM_BYTES;
  return -1;
}

int cfg_of(int bn, int mode, bool stages) {
  switch (mode) {
    case TC_SOLO: return cfg_value<TC_SOLO>(bn, stages);
    case TC_PAIR: return cfg_value<TC_PAIR>(bn, stages);
    case TC_KPAIR: return cfg_value<TC_KPAIR>(bn, stages);
    default: return -1;
  }
}
}  // namespace

int tc_smem_bytes(int bn, int mode) { return cfg_of(bn, mode, false); }
int tc_ring_bytes(int bn, int mode) {
  const int st = cfg_of(bn, mode, true);
  if (st <= 0) return -1;
  const int b_cols = mode == TC_PAIR ? bn / 2 : bn;
  return st * (TC_BM + b_cols) * TC_BK * 2;
}
int tc_stages(int bn, int mode) { return cfg_of(bn, mode, true); }

int tc_max_clusters(int bn, int mode) {
  if (mode == TC_PAIR) return bn == 256 ? max_clusters<256, TC_PAIR>() : (bn == 128 ? max_clusters<128, TC_PAIR>() : 0);
  if (mode == TC_KPAIR)
    return bn == 256 ? max_clusters<256, TC_KPAIR>() : (bn == 128 ? max_clusters<128, TC_KPAIR>() : 0);
  return 0;
}

namespace {
template <bool TF32>
cudaError_t launch_kind(int bn, int mode, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                        const CUtensorMap& ws, const TcParams& p, int grid, cudaStream_t s) {
  if (mode == TC_PAIR) {
    if (bn == 256) return launch_gemm_tc_bn<256, TC_PAIR, TF32>(a, b, c, ws, p, grid, s);
    if (bn == 128) return launch_gemm_tc_bn<128, TC_PAIR, TF32>(a, b, c, ws, p, grid, s);
    return cudaErrorInvalidValue;
  }
  if (mode == TC_KPAIR) {
    if (bn == 256) return launch_gemm_tc_bn<256, TC_KPAIR, TF32>(a, b, c, ws, p, grid, s);
    if (bn == 128) return launch_gemm_tc_bn<128, TC_KPAIR, TF32>(a, b, c, ws, p, grid, s);
    return cudaErrorInvalidValue;
  }
  switch (bn) {
    case 64: return launch_gemm_tc_bn<64, TC_SOLO, TF32>(a, b, c, ws, p, grid, s);
    case 128: return launch_gemm_tc_bn<128, TC_SOLO, TF32>(a, b, c, ws, p, grid, s);
    case 256: return launch_gemm_tc_bn<256, TC_SOLO, TF32>(a, b, c, ws, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_gemm_tc(int bn, int mode, const CUtensorMap& a, const CUtensorMap& b,
                           const CUtensorMap& c, const CUtensorMap& ws, const TcParams& p, int grid,
                           cudaStream_t s) {
  return p.tf32 ? launch_kind<true>(bn, mode, a, b, c, ws, p, grid, s)
                : launch_kind<false>(bn, mode, a, b, c, ws, p, grid, s);
}

}  // namespace dg
