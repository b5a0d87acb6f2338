// kernels.h -- parameter blocks and launchers shared by the host planner
// (api.cpp) and the CUDA kernels.  Internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dg {

// Output kinds of the tensor-core epilogue and of the GEMV / reduction kernels.
enum OutKind : int {
  OUT_F32 = 0,
  OUT_BF16 = 1,
  OUT_F16 = 2
};

// Debug build (compiled with DG_DEBUG into libdgemm_gb300_debug.so): every
// kernel checks each plain global load and store against the byte ranges of
// the call's own buffers (operands, output, the C that beta scales, plan
// workspace and counters), and each TMA copy's coordinates against the copy
// rules (innermost coordinate times the element size a multiple of 16 bytes;
// a store starts at non-negative coordinates), before the access.  A failed
// check skips the access and ORs DBG_FLAG and the site's bit (bit
// DBG_SITE_SHIFT + site) into the plan's error word, where
// gemm_plan_poll_error finds it.  A skipped TMA load never completes its
// barrier, so the waits behind it run out and add their own codes.  The
// release build compiles every check out.
enum DbgSite : int {
  DBG_TMA = 0,        // a TMA copy's coordinates break the copy rules
  DBG_EPI_STORE = 1,  // tensor-core epilogue: plain or bulk store of outputs
  DBG_EPI_LOAD = 2,   // tensor-core epilogue: plain load of the C that beta scales
  DBG_SPLIT = 3,      // K slices reduced inside the tensor-core kernel: partials, counters
  DBG_REDUCE = 4,     // tile reduction kernel
  DBG_GEMV = 5,       // GEMV kernels: matrix, vector, output, partials, counters
  DBG_SCALE = 6,      // the K == 0 / alpha == 0 kernel
  DBG_TRANSPOSE = 7   // the TF32 operand transpose
};
constexpr int DBG_SITE_SHIFT = 16;
constexpr int DBG_FLAG = 1 << 30;
constexpr int kDbgSpans = 6;
struct DbgSpans {
  uint64_t lo[kDbgSpans], hi[kDbgSpans];  // [lo, hi) byte ranges; unused entries have lo == hi
  int* err;                               // the plan's error word
};
#ifdef DG_DEBUG
#define DG_DEBUG_FIELD DbgSpans dbg;
#else
#define DG_DEBUG_FIELD
#endif

// Codes OR-ed into the plan's error word by a wait that ran out.
enum WaitCode : int {
  WAIT_PRODUCER_EMPTY = 1,
  WAIT_MMA_FULL = 2,
  WAIT_MMA_TMEM_EMPTY = 4,
  WAIT_EPI_TMEM_FULL = 8,
  WAIT_EPI_C_LOAD = 16,
  WAIT_DRAIN = 32,
  WAIT_SELFTEST = 64,
  WAIT_EPI_EXCHANGE = 128,  // K pair: the peer CTA's partial sums or its free buffers
  WAIT_SPLIT_PEERS = 256,   // split-K reduced in the GEMM kernel: the tile's other K slices
  WAIT_SPLIT_LOAD = 512     // ... or the bulk loads of the published slices
};

// Variants of the tensor-core kernel.
enum TcMode : int {
  TC_SOLO = 0,  // one CTA per 128-row tile (K optionally split over units + reduction kernel)
  TC_PAIR = 1,  // a cluster of two CTAs computes one 256-row tile with .cta_group::2 MMAs
  TC_KPAIR = 2  // a cluster of two CTAs splits the K loop of one 128-row tile in halves;
                // the halves' partial sums are exchanged through distributed shared
                // memory and each CTA finishes half of the tile's columns
};

constexpr int TC_BM = 128;       // output rows per tile (one tcgen05.mma M=128)
constexpr int TC_BK = 64;        // 16-bit K elements per stage: 64 x 2 B = one 128-B swizzle row
constexpr int TC_BK_TF32 = 32;   // TF32 (fp32 word) K elements per stage: the same 128 bytes
constexpr int TC_THREADS = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int TC_EPI_WARPS = 4;

// Output tile t (raster order) -> (m_blk, n_blk): groups of `group` tile rows,
// each group walked column by column, so that tiles running at the same time
// share A row-panels and B column-panels in L2.
__host__ __device__ inline void tile_coords(int t, int num_m_blocks, int num_n_blocks, int group,
                                            int* m_blk, int* n_blk) {
  const int per_group = group * num_n_blocks;
  const int g = t / per_group;
  const int first_m = g * group;
  const int rows = num_m_blocks - first_m < group ? num_m_blocks - first_m : group;
  const int r = t - g * per_group;
  *m_blk = first_m + r % rows;
  *n_blk = r / rows;
}

struct TcParams {
  int M, N, K;
  int num_m_blocks, num_n_blocks;
  int k_blocks;      // ceil(K / k-block elements): TC_BK (bf16/fp16) or TC_BK_TF32 per k-block
  int tf32;          // operands are TF32 (the kind::tf32 instantiation; both K-major)
  int raster_group;  // output-tile rows per rasterisation group
  // Work units, in this order: dp_units whole tiles (raster positions
  // 0 .. dp_units-1, all of K, final output); then `splitk` K slices of each of
  // the tail_tiles remaining tiles, slice-major, written as raw fp32 partial
  // sums to the workspace, tile-major [slice][tail tile][TILE_M rows][BN
  // columns], and summed in slice order by the tile reduction kernel.  Plain
  // split-K is dp_units = 0; no split is tail_tiles = 0.
  int dp_units;
  int tail_tiles;
  int splitk;        // K slices of a tail tile
  // fused_reduce (GEMM_FUSED_REDUCE=1): the slices are summed inside this
  // kernel instead of by the tile reduction kernel.  Then every partial unit is the last unit of its
  // CTA (tail_tiles * splitk <= CTAs or clusters) and all are resident at
  // once; the unit publishes its partials, arrives on the tile's counter
  // (counters[tail tile], zero on entry and left zero on exit), waits for
  // all splitk * CTAs-per-unit arrivals, then sums one share of the tile's
  // elements over slices 0 .. splitk-1 in order and applies the epilogue.
  int fused_reduce;
  unsigned* counters;
  const float* ws;   // the partial workspace (the memory tmW maps)
  int kb_per_split;  // k-blocks per slice (the last one may be shorter); a K pair: per half
  int units;         // dp_units + tail_tiles * splitk (a K pair: tiles)
  int out_kind;      // OutKind of C
  int n_tma;         // columns [0, n_tma) of the output go through TMA (a 16-byte multiple per row)
  void* c_ptr;       // the output (C, or D of gemm_run_ex), for columns [n_tma, N) written directly
  int64_t ldc;
  // The C that beta scales: the output itself (cin == c_ptr, read through the
  // output's tensor map) or, with cin_direct, a separate matrix of kind
  // cin_kind read with plain loads.
  const void* cin;
  int64_t ldcin;
  int cin_kind;
  int cin_direct;
  int a_mn_major;    // A stored K x M (M contiguous)
  int b_mn_major;    // B stored K x N (N contiguous)
  uint32_t idesc;    // tcgen05 instruction descriptor
  float alpha, beta, slope;
  int act;
  int* err;          // plan error word
  uint64_t timeout_ns;
  int pdl;           // launch as a programmatic dependent of the stream's previous kernel
  DG_DEBUG_FIELD     // (debug build) the byte ranges this launch may touch
};

// Shared-memory footprint and ring depth of the tensor-core kernel for a tile
// width and TcMode (TC_PAIR and TC_KPAIR exist for bn 128 and 256); -1 if none.
int tc_smem_bytes(int bn, int mode);
int tc_stages(int bn, int mode);
// Bytes of the operand ring (A and B stages) of one CTA.
int tc_ring_bytes(int bn, int mode);
// Clusters of two CTAs of a TC_PAIR / TC_KPAIR kernel that fit on the device at once.
int tc_max_clusters(int bn, int mode);

// TC_KPAIR: p.units counts tiles (one per cluster), p.kb_per_split is half the
// k-blocks (rounded up), and no unit is a tail slice (tail_tiles = 0).
// c: C (box 32 rows x 128 bytes); ws: the fp32 partial workspace (box 32 x 32),
// used only when p.tail_tiles > 0.
// p.tf32 selects the TF32 instantiation (kind::tf32, 32 K elements per k-block).
cudaError_t launch_gemm_tc(int bn, int mode, const CUtensorMap& a, const CUtensorMap& b,
                           const CUtensorMap& c, const CUtensorMap& ws, const TcParams& p, int grid,
                           cudaStream_t s);



#ifdef __CUDACC__
// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may be scheduled before the previous kernel
// in its stream has finished (once that kernel's CTAs have all started and
// signalled, or exited), so its launch and prologue overlap that kernel's
// tail.  It must call wait_prior_grid() before it reads or writes global
// memory: that returns once the previous kernel has completed and its writes
// are visible.  In a kernel launched normally it returns at once.
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Debug-build checks (see DbgSite): true when the access may go ahead.
#ifdef DG_DEBUG
__device__ __forceinline__ bool dbg_in(const DbgSpans& d, const void* ptr, int64_t bytes, int site) {
  const uint64_t a = reinterpret_cast<uint64_t>(ptr);
#pragma unroll
  for (int i = 0; i < kDbgSpans; ++i)
    if (a >= d.lo[i] && a + uint64_t(bytes) <= d.hi[i]) return true;
  atomicOr(d.err, DBG_FLAG | (1 << (DBG_SITE_SHIFT + site)));
  return false;
}
__device__ __forceinline__ bool dbg_tma(const DbgSpans& d, int x, int y, int esize, bool store) {
  if ((x * esize) % 16 == 0 && (!store || (x >= 0 && y >= 0))) return true;
  atomicOr(d.err, DBG_FLAG | (1 << (DBG_SITE_SHIFT + DBG_TMA)));
  return false;
}
#define DG_IN(spans, ptr, bytes, site) ::dg::dbg_in(spans, ptr, bytes, site)
#define DG_TMA(spans, x, y, esize, store) ::dg::dbg_tma(spans, x, y, esize, store)
#else
#define DG_IN(spans, ptr, bytes, site) true
#define DG_TMA(spans, x, y, esize, store) true
#endif

// kern<<<grid, block, smem, s>>>(args...), as a programmatic dependent if pdl.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Output transform (gemm_act_t), in fp32: 1 LeakyReLU, 2 ReLU, 3 GELU
// (x * Phi(x), Phi through erfc so the negative tail keeps its relative
// accuracy), 4 SiLU; anything else is the identity.
__device__ __forceinline__ float apply_act(float v, int act, float slope) {
  switch (act) {
    case 1: return v < 0.f ? v * slope : v;
    case 2: return v < 0.f ? 0.f : v;
    case 3: return 0.5f * v * erfcf(-v * 0.70710678118654752f);
    case 4: return v / (1.f + expf(-v));
    default: return v;
  }
}
#endif

struct EpiParams {
  float alpha, beta, slope;
  int act;
  int out_kind;  // OUT_F32 / OUT_BF16 / OUT_F16 of the output
  int cin_kind;  // of the C that beta scales
};

// Fixed-order sum of the K slices of the tail tiles of a tensor-core call
// (workspace layout: see TcParams), then the epilogue into C.
struct TileReduceArgs {
  const float* ws;
  int tail_tiles, splits;
  int tile0;  // raster position of the first tail tile (= dp_units)
  int tile_m, tile_n;
  int num_m_blocks, num_n_blocks, raster_group;
  int M, N;
  void* C;  // output
  int64_t ldc;
  const void* Cin;  // the C that beta scales (may be the output)
  int64_t ldcin;
  EpiParams e;
  int pdl;  // launch as a programmatic dependent of the GEMM that writes the partials
  DG_DEBUG_FIELD
};
cudaError_t launch_tile_reduce(const TileReduceArgs& a, cudaStream_t s, int sms);

// out (cols x rows, row stride ld_out) <- transpose of in (rows x cols, row
// stride ld_in), 32-bit elements: makes a TF32 operand K-major.
cudaError_t launch_transpose32(const void* in, int64_t ld_in, int rows, int cols, void* out, int64_t ld_out,
                               cudaStream_t s, const DbgSpans& dbg);

// D <- act(beta * C) (K == 0 or alpha == 0); C may be D.
// dbg: the byte ranges the kernel may touch (checked by the debug build only).
cudaError_t launch_scale(int M, int N, void* D, int64_t ldd, const void* C, int64_t ldc, EpiParams e,
                         cudaStream_t s, int sms, const DbgSpans& dbg);

// GEMV, operand type in_f16 (0 = bf16, 1 = fp16).
// rowdot:    out[r*inc_out] = epi(sum_k W[r*ldw + k] * x[k*incx]),  r < R
// colstream: out[c*inc_out] = epi(sum_k W[k*ldw + c] * x[k*incx]),  c < R
// generic:   out[r*inc_out] = epi(sum_k W[r*w_rs + k*w_cs] * x[k*incx])
struct GemvArgs {
  const void* W;
  int64_t ldw;
  int64_t w_rs, w_cs;  // generic strides (elements)
  int R, K;
  const void* x;
  int64_t incx;
  void* out;
  int64_t inc_out;
  const void* cin;  // the C that beta scales, element r at cin[r * inc_cin] (may be out)
  int64_t inc_cin;
  int in_f16;
  EpiParams e;
  int pdl;  // launch as a programmatic dependent of the stream's previous kernel
  DG_DEBUG_FIELD
};

int gemv_rowdot_max_k();
// grid_out (optional): the CTAs launched (one wave, sized from the occupancy query).
cudaError_t launch_gemv_rowdot(const GemvArgs& g, cudaStream_t s, int sms, int* grid_out = nullptr);

// Plan of the column-stream kernel: `ksplit` K slices of `kc` rows each.
struct ColstreamPlan {
  int cols;    // columns per CTA (panel width)
  int panels;  // ceil(R / cols)
  int ksplit;
  int kc;
  int64_t ws_bytes;  // fp32 partials, ksplit x panels x cols (0 when ksplit == 1)
};
ColstreamPlan plan_gemv_colstream(int R, int K, int sms);
// counters: `panels` words that are zero on entry and are left zero on exit.
cudaError_t launch_gemv_colstream(const GemvArgs& g, const ColstreamPlan& cp, void* ws,
                                  unsigned* counters, cudaStream_t s);

cudaError_t launch_gemv_generic(const GemvArgs& g, cudaStream_t s, int sms, int* grid_out = nullptr);

// One CTA waits on a barrier that nothing arrives on; gives up after timeout_ns.
cudaError_t launch_watchdog_selftest(int* err, uint64_t timeout_ns, cudaStream_t s);

}  // namespace dg
