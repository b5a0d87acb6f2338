// noalloc.cu -- gemm_gemv_noalloc: the column-stream GEMV with its scratch in a
// fixed device array of this library instead of plan workspace, so that the
// call allocates nothing.
//
// Who needs it: code that may not call cudaMalloc at the point where it runs
// a GEMV -- for instance a plugin inside an inference server or training
// framework that owns all device memory through its own pool allocator and
// forbids plugins from allocating behind its back (a raw cudaMalloc would
// fragment the pool, break its memory accounting and synchronise the device),
// or a latency-critical decode loop that cannot afford cudaMalloc's implicit
// device synchronisation.  gemm_run cannot serve them: gemm_plan_create
// allocates, and a plan grows its workspace on demand.
//
// The scratch (arrival counters + fp32 partial sums of the K slices) is one
// file-scope __device__ array of kScratchBytes.  CUDA loads a library's
// device code lazily, per device: this file's module, and with it the array,
// is loaded on a device by the first call there (cudaGetSymbolAddress), which
// takes the 4 MiB from that device's free memory and keeps it until the
// process exits.  A caller whose pool allocator reserves the device's memory
// should therefore make one call on each device before the pool takes the
// rest; later calls allocate nothing.  All calls on a device share the array
// and it keeps the last call's contents, so:
//  - each call zeroes the counters it uses (cudaMemsetAsync on its stream)
//    before the kernel, since the kernel needs them at zero on entry;
//  - calls whose kernels may overlap on the GPU (different streams without
//    ordering between them) race on the array and give wrong results; callers
//    must order such calls (one stream, or events).
// On the first call on a device the entry point looks the array's device
// address up with cudaGetSymbolAddress (host code cannot use the symbol
// itself: on the host it names a stand-in, not device memory).  That first
// call should come before any stream capture.  If the device has no room left
// for the array at that point, the call returns GEMM_ERR_OUT_OF_MEMORY.
#include <cuda_runtime.h>

#include <mutex>

#include "gemm.h"
#include "kernels.h"

namespace {

constexpr int kMaxPanels = 4096;                   // => N (or M) <= 2,097,152
constexpr size_t kScratchBytes = size_t(4) << 20;  // 4 MiB per device
constexpr size_t kCounterBytes = size_t(kMaxPanels) * sizeof(unsigned);
constexpr size_t kPartialFloats = (kScratchBytes - kCounterBytes) / sizeof(float);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

// Once per device, with that device current: device address of the scratch
// array and the SM count.
gemm_status_t device_setup(int dev, void** addr, int* sms) {
  if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    int major = 0, count = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        major != 10 ||
        cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_NO_DEVICE;
    }
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // loads the module here
    if (err != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return err == cudaErrorMemoryAllocation ? GEMM_ERR_OUT_OF_MEMORY : GEMM_ERR_CUDA;
    }
    g_sms[dev] = count;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  *sms = g_sms[dev];
  return GEMM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" gemm_status_t gemm_gemv_noalloc(int64_t M, int64_t N, int64_t K, const void* A,
                                           int64_t lda, const void* B, int64_t ldb, void* C,
                                           int64_t ldc, float alpha, float beta,
                                           gemm_dtype_t dtype, gemm_op_t transA, gemm_op_t transB,
                                           gemm_epilogue_t epilogue, void* stream) {
  gemm_status_t st = gemm_check_args(M, N, K, A, lda, B, ldb, C, ldc, alpha, dtype, transA,
                                     transB, epilogue);
  if (st != GEMM_OK) return st;
  if (M == 0 || N == 0) return GEMM_OK;
  if (K == 0 || alpha == 0.f) return GEMM_ERR_UNSUPPORTED;

  // The shapes gemm_run sends to the column-stream kernel: the matrix operand
  // is stored K x R with R contiguous.
  dg::GemvArgs g{};
  g.K = int(K);
  g.in_f16 = (dtype == GEMM_F16_F32 || dtype == GEMM_F16_F16) ? 1 : 0;
  g.out = C;
  const int kind = dtype == GEMM_BF16_F32 || dtype == GEMM_F16_F32
                       ? dg::OUT_F32
                       : (dtype == GEMM_BF16_BF16 ? dg::OUT_BF16 : dg::OUT_F16);
  g.e = dg::EpiParams{alpha, beta, epilogue.slope, epilogue.act, kind, kind};  // beta scales C itself
  if (N == 1 && transA == GEMM_OP_T) {
    g.R = int(M);
    g.inc_out = ldc;
    g.x = B;
    g.incx = transB == GEMM_OP_N ? ldb : 1;
    g.W = A;
    g.ldw = lda;
  } else if (M == 1 && N > 1 && transB == GEMM_OP_N) {
    g.R = int(N);
    g.inc_out = 1;
    g.x = A;
    g.incx = transA == GEMM_OP_N ? 1 : lda;
    g.W = B;
    g.ldw = ldb;
  } else {
    return GEMM_ERR_UNSUPPORTED;
  }
  g.cin = C;
  g.inc_cin = g.inc_out;
#ifdef DG_DEBUG
  // (debug build) no plan to report through: every byte range is allowed
  g.dbg.lo[0] = 0;
  g.dbg.hi[0] = ~uint64_t(0);
#endif
  if (!aligned16(g.W) || ((g.ldw * 2) % 16 != 0 && K != 1)) return GEMM_ERR_UNSUPPORTED;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  void* scratch = nullptr;
  int sms = 0;
  st = device_setup(dev, &scratch, &sms);
  if (st != GEMM_OK) return st;

  dg::ColstreamPlan cp = dg::plan_gemv_colstream(g.R, g.K, sms);
  if (cp.panels > kMaxPanels) return GEMM_ERR_UNSUPPORTED;  // R beyond the fixed scratch
  const int64_t per_split = int64_t(cp.panels) * cp.cols;
  const int64_t max_split = int64_t(kPartialFloats) / per_split;
  if (cp.ksplit > 1 && max_split < 2) {
    cp.ksplit = 1;  // no room for two slices: one slice, no partials
    cp.kc = g.K;
  } else if (cp.ksplit > max_split) {
    cp.kc = int((K + max_split - 1) / max_split);
    cp.ksplit = int((K + cp.kc - 1) / cp.kc);
  }
  cp.ws_bytes = cp.ksplit > 1 ? int64_t(cp.ksplit) * per_split * 4 : 0;

  unsigned* counters = static_cast<unsigned*>(scratch);
  float* partials = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + kCounterBytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cp.ksplit > 1 &&
      cudaMemsetAsync(counters, 0, size_t(cp.panels) * sizeof(unsigned), s) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (dg::launch_gemv_colstream(g, cp, partials, counters, s) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return GEMM_OK;
}
