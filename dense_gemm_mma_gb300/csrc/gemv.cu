// gemv.cu -- memory-bound kernels: GEMV (M == 1 or N == 1), the fixed-order
// split-K reduction, C <- act(beta*C), and the watchdog self-test.
//
// "Matrix Multiplication Background User's Guide", section 2: a
// matrix-vector product (M == 1 or N == 1) has an arithmetic intensity below
// one FLOP per byte and is always memory-bound, so these kernels use no tensor
// cores: they stream the matrix once with 128-bit loads, coalesced across the
// warp ("Learning Triton One Kernel at a Time: Matrix Multiplication", section
// Memory coalescing: consecutive threads read consecutive addresses), and
// reduce with warp shuffles.  Every sum is taken in a fixed order, so results
// do not depend on scheduling.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>

#include "kernels.h"
#include "ptx.cuh"

namespace dg {

namespace {

constexpr int kRowdotThreads = 256;
constexpr int kRowdotCtasPerSm = 8;
constexpr int kRowdotMaxK = 32768;  // x staged in shared memory: 64 KB of 16-bit values
constexpr int kColThreads = 512;  // 64 warps per SM at four CTAs per SM
constexpr int kColGroups = 8;             // K-interleaved thread groups per CTA
constexpr int kColCols = 8 * (kColThreads / kColGroups);  // 512 columns per CTA
constexpr int kColMaxKc = 2048;           // rows of x staged in shared memory at a time
static_assert(kColThreads % (kColCols / 4) == 0, "the last-CTA reduction gives every thread one column quad");
static_assert(kColMaxKc % kColGroups == 0, "a chunk of x keeps every row with its group");

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

template <bool F16>
__device__ __forceinline__ float2 to_f2(uint32_t w) {
  if (F16) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
  }
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
  return __bfloat1622float2(h);
}

template <bool F16>
__device__ __forceinline__ float to_f(uint16_t v) {
  if (F16) return __half2float(__ushort_as_half(v));
  return __bfloat162float(__ushort_as_bfloat16(v));
}

// acc += dot of 8 packed elements
template <bool F16>
__device__ __forceinline__ float dot8(uint4 a, uint4 b, float acc) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 fa = to_f2<F16>(aw[t]);
    const float2 fb = to_f2<F16>(bw[t]);
    acc = fmaf(fa.x, fb.x, acc);
    acc = fmaf(fa.y, fb.y, acc);
  }
  return acc;
}

__device__ __forceinline__ float load_c(const void* C, int64_t idx, int kind) {
  if (kind == OUT_F32) return static_cast<const float*>(C)[idx];
  const uint16_t v = static_cast<const uint16_t*>(C)[idx];
  if (kind == OUT_BF16) return __bfloat162float(__ushort_as_bfloat16(v));
  return __half2float(__ushort_as_half(v));
}

__device__ __forceinline__ void store_c(void* C, int64_t idx, float v, int kind) {
  if (kind == OUT_F32) {
    static_cast<float*>(C)[idx] = v;
  } else if (kind == OUT_BF16) {
    static_cast<__nv_bfloat16*>(C)[idx] = __float2bfloat16_rn(v);
  } else {
    static_cast<__half*>(C)[idx] = __float2half_rn(v);
  }
}

// alpha*acc + beta*C[idx] (C, of kind e.cin_kind, not read when beta == 0),
// then the activation.
__device__ __forceinline__ float epilogue(float acc, const void* C, int64_t idx, const EpiParams& e) {
  float v = e.alpha * acc;
  if (e.beta != 0.f) v = fmaf(e.beta, load_c(C, idx, e.cin_kind), v);
  v = apply_act(v, e.act, e.slope);
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Output r of a GEMV: the epilogue of acc (reading C[r * inc_cin] when beta
// != 0) stored at out[r * inc_out].
__device__ __forceinline__ void gemv_store(const GemvArgs& g, int64_t r, float acc) {
  const int64_t oi = r * g.inc_out, ci = r * g.inc_cin;
#ifdef DG_DEBUG
  const int os = g.e.out_kind == OUT_F32 ? 4 : 2, cs = g.e.cin_kind == OUT_F32 ? 4 : 2;
  if (g.e.beta != 0.f && !DG_IN(g.dbg, static_cast<const char*>(g.cin) + ci * cs, cs, DBG_GEMV)) return;
  if (!DG_IN(g.dbg, static_cast<char*>(g.out) + oi * os, os, DBG_GEMV)) return;
#endif
  store_c(g.out, oi, epilogue(acc, g.cin, ci, g.e), g.e.out_kind);
}

// ------------------------------------------------------------------ rowdot
// One warp per row of W (row-contiguous, 16-byte aligned rows).  Each lane
// keeps kRowU 16-byte loads of its row in flight; registers are held to 32 a
// thread so that eight CTAs (64 warps) fit on an SM and 8192 rows run as one
// wave at one row per warp (27.3 us for 1 x 8192 x 8192, against 29.3 with
// eight loads in flight, six CTAs per SM and two rows per warp).  x is read
// with 16-byte loads through L1 when it is contiguous and aligned (kXDirect),
// else it is first gathered into shared memory.
constexpr int kRowU = 4;

template <bool F16>
__device__ __forceinline__ uint4 load_x_vec(const uint16_t* x, const uint16_t* xs, int v, bool direct) {
  if (direct) return __ldg(reinterpret_cast<const uint4*>(x) + v);
  return reinterpret_cast<const uint4*>(xs)[v];
}

template <bool F16, bool kXDirect>
__global__ void __launch_bounds__(kRowdotThreads, kRowdotCtasPerSm)
    gemv_rowdot_kernel(const GemvArgs g) {
  wait_prior_grid();
  extern __shared__ __align__(16) uint16_t xs[];
  const uint16_t* x = static_cast<const uint16_t*>(g.x);
  const int K = g.K;
  if (!kXDirect) {
    const int K8 = (K + 7) & ~7;
    for (int k = threadIdx.x; k < K8; k += blockDim.x) {
      uint16_t v = 0;
      if (k < K && DG_IN(g.dbg, x + static_cast<int64_t>(k) * g.incx, 2, DBG_GEMV)) v = x[k * g.incx];
      xs[k] = v;
    }
    __syncthreads();
  }
#ifdef DG_DEBUG
  if (kXDirect && !DG_IN(g.dbg, x, int64_t(K) * 2, DBG_GEMV)) return;
#endif
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpb = kRowdotThreads / 32;
  const int nvec = K >> 3;
  for (int r = blockIdx.x * wpb + warp; r < g.R; r += gridDim.x * wpb) {
    const uint16_t* wrow = static_cast<const uint16_t*>(g.W) + static_cast<int64_t>(r) * g.ldw;
    const uint4* wv = reinterpret_cast<const uint4*>(wrow);
#ifdef DG_DEBUG
    if (!DG_IN(g.dbg, wrow, int64_t(K) * 2, DBG_GEMV)) continue;  // the whole row, once per warp
#endif
    float a0 = 0.f, a1 = 0.f;
    int v = lane;
    for (; v + 32 * (kRowU - 1) < nvec; v += 32 * kRowU) {
      uint4 w[kRowU];
#pragma unroll
      for (int u = 0; u < kRowU; ++u) w[u] = ldg_stream(wv + v + 32 * u);
#pragma unroll
      for (int u = 0; u < kRowU; u += 2) {
        a0 = dot8<F16>(w[u], load_x_vec<F16>(x, xs, v + 32 * u, kXDirect), a0);
        a1 = dot8<F16>(w[u + 1], load_x_vec<F16>(x, xs, v + 32 * (u + 1), kXDirect), a1);
      }
    }
    for (; v < nvec; v += 32) a0 = dot8<F16>(ldg_stream(wv + v), load_x_vec<F16>(x, xs, v, kXDirect), a0);
    for (int k = nvec * 8 + lane; k < K; k += 32)
      a1 = fmaf(to_f<F16>(wrow[k]), to_f<F16>(kXDirect ? x[k] : xs[k]), a1);
    const float acc = warp_sum(a0 + a1);
    if (lane == 0) gemv_store(g, r, acc);
  }
}

// --------------------------------------------------------------- colstream
// W is K x R with R contiguous.  CTA (panel, z) covers columns
// [panel*512, panel*512+512) and K rows [z*kc, z*kc+kc); its 512 threads form
// 8 groups of 64, each thread owning 8 adjacent columns (one 16-byte load per
// row, kColU rows in flight) and every 8th row of the slice; the slice of x is
// staged in shared memory as fp32.  The groups are summed in shared memory in
// a fixed order.  With ksplit > 1 each CTA writes its 512 partial sums to the
// workspace; the CTA that finishes a panel last (per-panel arrival counter,
// zero on entry) sums the slices -- four fixed ranges in slice order, then the
// ranges -- applies the epilogue and sets the counter back to zero.  Four CTAs
// of 512 threads at 32 registers fill an SM with 64 warps of loads for the
// same K split as 256-thread CTAs: 1 x 8192 x 8192 29.3 us (30.1-31.3 with
// 256 threads), 1 x 4096 x 4096 15.0 us (17.0 with 384).
constexpr int kColU = 4;

template <bool F16>
__device__ __forceinline__ void fma_row(float (&acc)[8], uint4 wv, float xf) {
  const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = to_f2<F16>(ww[q]);
    acc[2 * q] = fmaf(f.x, xf, acc[2 * q]);
    acc[2 * q + 1] = fmaf(f.y, xf, acc[2 * q + 1]);
  }
}

template <bool F16>
__global__ void __launch_bounds__(kColThreads, 4)
    gemv_colstream_kernel(const GemvArgs g, const ColstreamPlan cp, float* ws, unsigned* counters) {
  wait_prior_grid();
  __shared__ float red[kColGroups][kColCols];
  __shared__ float xsl[kColMaxKc];
  __shared__ unsigned ticket;
  const int panel = blockIdx.x, z = blockIdx.y;
  const int t = threadIdx.x % (kColThreads / kColGroups);
  const int grp = threadIdx.x / (kColThreads / kColGroups);
  const int col0 = panel * kColCols + t * 8;
  const int kb = z * cp.kc;
  const int ke = min(g.K, kb + cp.kc);
  const uint16_t* W = static_cast<const uint16_t*>(g.W);
  const uint16_t* x = static_cast<const uint16_t*>(g.x);
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
  // The slice is walked in chunks of kColMaxKc rows whose x values are staged
  // in shared memory (chunk starts are multiples of kColGroups rows past kb, so
  // row k stays with group (k - kb) % kColGroups).
  for (int cb = kb; cb < ke; cb += kColMaxKc) {
    const int ce = min(ke, cb + kColMaxKc);
    __syncthreads();  // the previous chunk's x is no longer read
    for (int k = cb + threadIdx.x; k < ce; k += kColThreads) {
      float xv = 0.f;
      if (DG_IN(g.dbg, x + static_cast<int64_t>(k) * g.incx, 2, DBG_GEMV)) xv = to_f<F16>(x[static_cast<int64_t>(k) * g.incx]);
      xsl[k - cb] = xv;
    }
    __syncthreads();
#ifdef DG_DEBUG
    // this thread's strip of the chunk: 8 columns of rows cb + grp, + 8, ... < ce
    const int k_last = cb + grp + ((ce - 1 - cb - grp) / kColGroups) * kColGroups;
    const bool strip_ok = col0 >= g.R || cb + grp >= ce ||
                          (DG_IN(g.dbg, W + static_cast<int64_t>(cb + grp) * g.ldw + col0, min(8, g.R - col0) * 2, DBG_GEMV) &&
                           DG_IN(g.dbg, W + static_cast<int64_t>(k_last) * g.ldw + col0, min(8, g.R - col0) * 2, DBG_GEMV));
    if (!strip_ok) continue;
#endif
    if (col0 + 8 <= g.R) {
      const uint16_t* wp = W + static_cast<int64_t>(cb + grp) * g.ldw + col0;
      const int64_t step = static_cast<int64_t>(kColGroups) * g.ldw;
      int k = cb + grp;
      for (; k + (kColU - 1) * kColGroups < ce; k += kColU * kColGroups) {
        uint4 wv[kColU];
#pragma unroll
        for (int i = 0; i < kColU; ++i) wv[i] = ldg_stream(wp + i * step);
#pragma unroll
        for (int i = 0; i < kColU; ++i) fma_row<F16>(acc, wv[i], xsl[k - cb + i * kColGroups]);
        wp += kColU * step;
      }
      for (; k < ce; k += kColGroups) {
        fma_row<F16>(acc, ldg_stream(wp), xsl[k - cb]);
        wp += step;
      }
    } else if (col0 < g.R) {
      const int nc = g.R - col0;
      for (int k = cb + grp; k < ce; k += kColGroups) {
        const float xf = xsl[k - cb];
        for (int j = 0; j < nc; ++j)
          acc[j] = fmaf(to_f<F16>(W[static_cast<int64_t>(k) * g.ldw + col0 + j]), xf, acc[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) red[grp][t * 8 + j] = acc[j];
  __syncthreads();

  const int rpad = cp.panels * kColCols;
  for (int c = threadIdx.x; c < kColCols; c += kColThreads) {
    const int col = panel * kColCols + c;
    float s = red[0][c];
#pragma unroll
    for (int q = 1; q < kColGroups; ++q) s += red[q][c];
    if (col < g.R) {
      if (cp.ksplit == 1) {
        gemv_store(g, col, s);
      } else if (DG_IN(g.dbg, ws + static_cast<int64_t>(z) * rpad + col, 4, DBG_GEMV)) {
        ws[static_cast<int64_t>(z) * rpad + col] = s;
      }
    }
  }
  if (cp.ksplit == 1) return;

  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    ticket = 0u;  // (the debug build's skipped arrival: not the last CTA)
    if (DG_IN(g.dbg, counters + panel, 4, DBG_GEMV)) ticket = atomicAdd(&counters[panel], 1u);
  }
  __syncthreads();
  if (ticket != static_cast<unsigned>(cp.ksplit - 1)) return;
  __threadfence();
  // Last CTA of the panel: thread (h, q) sums columns 4q..4q+3 over the h-th
  // of kParts consecutive ranges of slices.
  constexpr int kQuads = kColCols / 4;
  constexpr int kParts = kColThreads / kQuads;
  const int q = threadIdx.x % kQuads;
  const int h = threadIdx.x / kQuads;
  const int per = (cp.ksplit + kParts - 1) / kParts;
  const int z0 = min(cp.ksplit, h * per);
  int z1 = min(cp.ksplit, z0 + per);
  const float* src = ws + panel * kColCols + 4 * q;
  float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
  int zz = z0;
#ifdef DG_DEBUG
  if (z1 > z0 && !(DG_IN(g.dbg, src + static_cast<int64_t>(z0) * rpad, 16, DBG_GEMV) &&
                   DG_IN(g.dbg, src + static_cast<int64_t>(z1 - 1) * rpad, 16, DBG_GEMV)))
    z1 = z0;  // skip this thread's slices
#endif
  for (; zz + 7 < z1; zz += 8) {
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldcg(reinterpret_cast<const float4*>(src + static_cast<int64_t>(zz + i) * rpad));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s4.x += v[i].x;
      s4.y += v[i].y;
      s4.z += v[i].z;
      s4.w += v[i].w;
    }
  }
  for (; zz < z1; ++zz) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(src + static_cast<int64_t>(zz) * rpad));
    s4.x += v.x;
    s4.y += v.y;
    s4.z += v.z;
    s4.w += v.w;
  }
  float* half = &red[0][0];  // reuse: [kParts][kColCols]
  __syncthreads();
  half[h * kColCols + 4 * q + 0] = s4.x;
  half[h * kColCols + 4 * q + 1] = s4.y;
  half[h * kColCols + 4 * q + 2] = s4.z;
  half[h * kColCols + 4 * q + 3] = s4.w;
  __syncthreads();
  for (int c = threadIdx.x; c < kColCols; c += kColThreads) {
    const int col = panel * kColCols + c;
    if (col >= g.R) break;
    float s = half[c];
#pragma unroll
    for (int part = 1; part < kParts; ++part) s += half[part * kColCols + c];
    gemv_store(g, col, s);
  }
  if (threadIdx.x == 0 && DG_IN(g.dbg, counters + panel, 4, DBG_GEMV)) counters[panel] = 0u;
}

// ----------------------------------------------------------------- generic
// Any strides: one warp per output, lanes interleaved over K.
template <bool F16>
__global__ void __launch_bounds__(256) gemv_generic_kernel(const GemvArgs g) {
  wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const uint16_t* W = static_cast<const uint16_t*>(g.W);
  const uint16_t* x = static_cast<const uint16_t*>(g.x);
  for (int r = gw; r < g.R; r += nw) {
    float acc = 0.f;
    for (int k = lane; k < g.K; k += 32) {
      const uint16_t* wp = W + static_cast<int64_t>(r) * g.w_rs + static_cast<int64_t>(k) * g.w_cs;
      const uint16_t* xp = x + static_cast<int64_t>(k) * g.incx;
      if (DG_IN(g.dbg, wp, 2, DBG_GEMV) && DG_IN(g.dbg, xp, 2, DBG_GEMV))
        acc = fmaf(to_f<F16>(*wp), to_f<F16>(*xp), acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) gemv_store(g, r, acc);
  }
}

// ------------------------------------------------------------ split-K reduce
// One thread per 4 adjacent columns of a row of a tail tile: sums the tile's
// slices s = 0..S-1 in order (16-byte loads from the tile-major workspace),
// applies the epilogue and stores the outputs that lie inside C.
constexpr int kReduceThreads = 128;

__global__ void __launch_bounds__(kReduceThreads) tile_reduce_kernel(const TileReduceArgs a) {
  // Launched as a programmatic dependent of the GEMM that writes the partials:
  // this CTA may start before that grid ends, so wait for its results here.
  wait_prior_grid();
  const EpiParams& e = a.e;
  const int gpr = a.tile_n >> 2;
  const int64_t per_tile = static_cast<int64_t>(a.tile_m) * gpr;
  const int64_t total = per_tile * a.tail_tiles;
  const int64_t slice = static_cast<int64_t>(a.tail_tiles) * a.tile_m * a.tile_n;
  void* const C = a.C;
  const int N = a.N;
  // beta scales the output itself: 16- or 8-byte read-modify-write of 4 outputs
  const bool in_place = a.Cin == a.C && a.ldcin == a.ldc && e.cin_kind == e.out_kind;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / per_tile);
    const int rem = static_cast<int>(i - static_cast<int64_t>(t) * per_tile);
    const int r = rem / gpr;
    const int c4 = rem - r * gpr;
    int m_blk, n_blk;
    tile_coords(a.tile0 + t, a.num_m_blocks, a.num_n_blocks, a.raster_group, &m_blk, &n_blk);
    const int m = m_blk * a.tile_m + r;
    const int n = n_blk * a.tile_n + c4 * 4;
    if (m >= a.M || n >= N) continue;
    const float* src = a.ws + (static_cast<int64_t>(t) * a.tile_m + r) * a.tile_n + c4 * 4;
#ifdef DG_DEBUG
    // the first and the last slice of these four partial sums
    if (!DG_IN(a.dbg, src, 16, DBG_REDUCE) || !DG_IN(a.dbg, src + (a.splits - 1) * slice, 16, DBG_REDUCE)) continue;
#endif
    float4 s = __ldcs(reinterpret_cast<const float4*>(src));
    int sp = 1;
    // slices in order, eight loads in flight before their adds (the sum is
    // s0 + s1 + s2 + ... whatever the batching)
    for (; sp + 8 <= a.splits; sp += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcs(reinterpret_cast<const float4*>(src + (sp + u) * slice));
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        s.x += v[u].x;
        s.y += v[u].y;
        s.z += v[u].z;
        s.w += v[u].w;
      }
    }
    for (; sp < a.splits; ++sp) {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(src + sp * slice));
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    float sv[4] = {s.x, s.y, s.z, s.w};
    const int64_t base = static_cast<int64_t>(m) * a.ldc + n;
    const int nn = min(4, N - n);
    const int esz = e.out_kind == OUT_F32 ? 4 : 2;
    const bool vec = in_place && nn == 4 &&
                     ((reinterpret_cast<uintptr_t>(C) + base * esz) & (4 * esz - 1)) == 0;
    if (!vec) {
      const int64_t cbase = static_cast<int64_t>(m) * a.ldcin + n;
      for (int j = 0; j < nn; ++j) {
#ifdef DG_DEBUG
        const int cs = e.cin_kind == OUT_F32 ? 4 : 2;
        if (e.beta != 0.f && !DG_IN(a.dbg, static_cast<const char*>(a.Cin) + (cbase + j) * cs, cs, DBG_REDUCE)) continue;
        if (!DG_IN(a.dbg, static_cast<char*>(C) + (base + j) * esz, esz, DBG_REDUCE)) continue;
#endif
        store_c(C, base + j, epilogue(sv[j], a.Cin, cbase + j, e), e.out_kind);
      }
      continue;
    }
#ifdef DG_DEBUG
    if (!DG_IN(a.dbg, static_cast<char*>(C) + base * esz, 4 * esz, DBG_REDUCE)) continue;
#endif
    // Four adjacent outputs with one 16-byte (fp32) or 8-byte (16-bit) access.
    if (e.out_kind == OUT_F32) {
      float4* cp = reinterpret_cast<float4*>(static_cast<float*>(C) + base);
      float4 cv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e.beta != 0.f) cv = *cp;
      const float cin[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float v = e.alpha * sv[j];
        if (e.beta != 0.f) v = fmaf(e.beta, cin[j], v);
        v = apply_act(v, e.act, e.slope);
        sv[j] = v;
      }
      *cp = make_float4(sv[0], sv[1], sv[2], sv[3]);
    } else {
      uint2* cp = reinterpret_cast<uint2*>(static_cast<uint16_t*>(C) + base);
      uint2 cv = make_uint2(0u, 0u);
      if (e.beta != 0.f) cv = *cp;
      const uint16_t cin[4] = {uint16_t(cv.x), uint16_t(cv.x >> 16), uint16_t(cv.y), uint16_t(cv.y >> 16)};
      uint16_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float v = e.alpha * sv[j];
        if (e.beta != 0.f) {
          const float c = e.out_kind == OUT_BF16 ? __bfloat162float(__ushort_as_bfloat16(cin[j]))
                                                 : __half2float(__ushort_as_half(cin[j]));
          v = fmaf(e.beta, c, v);
        }
        v = apply_act(v, e.act, e.slope);
        o[j] = e.out_kind == OUT_BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v))
                                      : __half_as_ushort(__float2half_rn(v));
      }
      *cp = make_uint2(uint32_t(o[0]) | (uint32_t(o[1]) << 16), uint32_t(o[2]) | (uint32_t(o[3]) << 16));
    }
  }
}

// --------------------------------------------------------------- transpose
// out (cols x rows) <- in (rows x cols)^T for 32-bit words, in 64 x 64 tiles
// staged in shared memory (a padding column keeps the column-wise reads free
// of bank conflicts).  Each thread issues its 16 loads before any store, so
// enough bytes are in flight to stream from HBM; loads and stores are both
// row-contiguous (32 words per warp instruction).
constexpr int kTrTile = 64;
__global__ void __launch_bounds__(256) transpose32_kernel(const uint32_t* __restrict__ in, int64_t ld_in,
                                                          int rows, int cols, uint32_t* __restrict__ out,
                                                          int64_t ld_out, const DbgSpans dbg) {
  __shared__ uint32_t tile[kTrTile][kTrTile + 1];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 rows of 32 per pass
  for (int by = blockIdx.y * kTrTile; by < rows; by += gridDim.y * kTrTile) {
    for (int bx = blockIdx.x * kTrTile; bx < cols; bx += gridDim.x * kTrTile) {
      uint32_t v[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = by + ty + 8 * j, c = bx + tx + 32 * h;
          v[2 * j + h] = (r < rows && c < cols && DG_IN(dbg, in + static_cast<int64_t>(r) * ld_in + c, 4, DBG_TRANSPOSE))
                             ? in[static_cast<int64_t>(r) * ld_in + c]
                             : 0u;
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int h = 0; h < 2; ++h) tile[ty + 8 * j][tx + 32 * h] = v[2 * j + h];
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = bx + ty + 8 * j, c = by + tx + 32 * h;  // row of out = column of in
          if (r < cols && c < rows && DG_IN(dbg, out + static_cast<int64_t>(r) * ld_out + c, 4, DBG_TRANSPOSE))
            out[static_cast<int64_t>(r) * ld_out + c] = tile[tx + 32 * h][ty + 8 * j];
        }
      }
      __syncthreads();
    }
  }
}

// ------------------------------------------------------------------- scale
__global__ void __launch_bounds__(256) scale_kernel(int M, int N, void* D, int64_t ldd, const void* C,
                                                    int64_t ldc, const EpiParams e, const DbgSpans dbg) {
  const int64_t total = static_cast<int64_t>(M) * N;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(i / N);
    const int n = static_cast<int>(i - static_cast<int64_t>(m) * N);
    const int64_t ci = static_cast<int64_t>(m) * ldc + n, di = static_cast<int64_t>(m) * ldd + n;
#ifdef DG_DEBUG
    const int cs = e.cin_kind == OUT_F32 ? 4 : 2, ds = e.out_kind == OUT_F32 ? 4 : 2;
    const bool c_ok = DG_IN(dbg, static_cast<const char*>(C) + ci * cs, cs, DBG_SCALE);
    if (!DG_IN(dbg, static_cast<char*>(D) + di * ds, ds, DBG_SCALE)) continue;
#else
    constexpr bool c_ok = true;
#endif
    float v = e.beta != 0.f && c_ok ? e.beta * load_c(C, ci, e.cin_kind) : 0.f;
    v = apply_act(v, e.act, e.slope);
    store_c(D, di, v, e.out_kind);
  }
}

// --------------------------------------------------------- watchdog self-test
__global__ void watchdog_selftest_kernel(int* err, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const Watch w{&abort_flag, err, timeout_ns};
    wait_bar(smem_u32(&bar), 0, w, WAIT_SELFTEST);  // nothing ever arrives
  }
}

int grid_for(int64_t items, int per_block, int sms, int blocks_per_sm) {
  int64_t g = (items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(sms) * blocks_per_sm;
  if (g > cap) g = cap;
  return g < 1 ? 1 : static_cast<int>(g);
}

// Grid of a kernel whose warps take rows r, r + (warps in the grid), ...:
// one wave, every warp the same number of rows (within one).  A CTA that has
// to wait for a slot runs its rows after the others have finished, at a
// fraction of the bandwidth: in a 1 x 8192 x 8192 row-dot GEMV a second wave
// of 11% of the CTAs took 40% of the time.  `occ` caches the resident CTAs
// per SM of the kernel as smem << 16 | count (one word, so that threads see a
// matching pair).
template <typename Kern>
int resident_per_sm(Kern kern, std::atomic<int64_t>& occ, int threads, int smem) {
  int64_t c = occ.load(std::memory_order_relaxed);
  if (c < 0 || (c >> 16) != smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 1;
    }
    c = (static_cast<int64_t>(smem) << 16) | n;
    occ.store(c, std::memory_order_relaxed);
  }
  return static_cast<int>(c & 0xffff);
}

template <typename Kern>
int one_wave_grid(Kern kern, std::atomic<int64_t>& occ, int threads, int smem, int64_t rows, int sms) {
  const int wpb = threads / 32;
  const int64_t resident_warps = static_cast<int64_t>(sms) * resident_per_sm(kern, occ, threads, smem) * wpb;
  const int64_t rows_per_warp = (rows + resident_warps - 1) / resident_warps;
  const int64_t warps = (rows + rows_per_warp - 1) / rows_per_warp;
  const int64_t grid = (warps + wpb - 1) / wpb;
  return grid < 1 ? 1 : static_cast<int>(grid);
}

}  // namespace

int gemv_rowdot_max_k() { return kRowdotMaxK; }

cudaError_t launch_gemv_rowdot(const GemvArgs& g, cudaStream_t s, int sms, int* grid_out) {
  const bool direct = g.incx == 1 && (reinterpret_cast<uintptr_t>(g.x) & 15u) == 0;
  const int smem = direct ? 0 : ((g.K + 7) & ~7) * 2;
  cudaError_t err = cudaSuccess;
  auto go = [&](auto kern) {
    if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    static std::atomic<int64_t> occ{-1};
    const int grid = one_wave_grid(kern, occ, kRowdotThreads, smem, g.R, sms);
    if (grid_out) *grid_out = grid;
    err = launch_k(kern, dim3(grid), dim3(kRowdotThreads), smem, s, g.pdl != 0, g);
  };
  if (g.in_f16) {
    if (direct) go(gemv_rowdot_kernel<true, true>); else go(gemv_rowdot_kernel<true, false>);
  } else {
    if (direct) go(gemv_rowdot_kernel<false, true>); else go(gemv_rowdot_kernel<false, false>);
  }
  return err;
}

ColstreamPlan plan_gemv_colstream(int R, int K, int sms) {
  ColstreamPlan cp;
  cp.cols = kColCols;
  cp.panels = (R + kColCols - 1) / kColCols;
  const int target = sms * 4;  // four CTAs per SM, each thread with kColU rows in flight
  // at most `target` CTAs: more would leave a few of them for a second wave
  int ksplit = target / cp.panels;
  const int max_split = (K + 63) / 64;  // at least 64 rows (16 per thread) per slice
  if (ksplit > max_split) ksplit = max_split;
  if (const char* f = std::getenv("GEMM_FORCE_GEMV_SPLITK")) {  // tests and sweeps
    const int v = std::atoi(f);
    if (v > 0) ksplit = v < K ? v : K;
  }
  if (ksplit < 1) ksplit = 1;
  cp.kc = (K + ksplit - 1) / ksplit;
  cp.ksplit = (K + cp.kc - 1) / cp.kc;
  if (cp.ksplit < 1) cp.ksplit = 1;
  cp.ws_bytes = cp.ksplit > 1 ? static_cast<int64_t>(cp.ksplit) * cp.panels * kColCols * 4 : 0;
  return cp;
}

cudaError_t launch_gemv_colstream(const GemvArgs& g, const ColstreamPlan& cp, void* ws,
                                  unsigned* counters, cudaStream_t s) {
  float* part = static_cast<float*>(ws);
  const dim3 grid(cp.panels, cp.ksplit);
  auto kern = g.in_f16 ? gemv_colstream_kernel<true> : gemv_colstream_kernel<false>;
  return launch_k(kern, grid, dim3(kColThreads), 0, s, g.pdl != 0, g, cp, part, counters);
}

cudaError_t launch_gemv_generic(const GemvArgs& g, cudaStream_t s, int sms, int* grid_out) {
  auto kern = g.in_f16 ? gemv_generic_kernel<true> : gemv_generic_kernel<false>;
  static std::atomic<int64_t> occ[2] = {{-1}, {-1}};
  const int grid = one_wave_grid(kern, occ[g.in_f16 ? 1 : 0], 256, 0, g.R, sms);
  if (grid_out) *grid_out = grid;
  return launch_k(kern, dim3(grid), dim3(256), 0, s, g.pdl != 0, g);
}

cudaError_t launch_tile_reduce(const TileReduceArgs& a, cudaStream_t s, int sms) {
  const int64_t items = static_cast<int64_t>(a.tail_tiles) * a.tile_m * (a.tile_n / 4);
  // Programmatic dependent launch: the reduction's launch overlaps the tail of
  // the GEMM; its griddepcontrol.wait orders it after the GEMM's writes.
  // (a grid-stride kernel: no more CTAs than are resident at once, so none
  // waits for a slot and runs its share after the others)
  // (128-thread CTAs: a split-K call has few tiles, and smaller CTAs spread
  // its items over more SMs)
  static std::atomic<int64_t> occ{-1};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_for(items, kReduceThreads, sms,
                              resident_per_sm(tile_reduce_kernel, occ, kReduceThreads, 0)));
  cfg.blockDim = dim3(kReduceThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tile_reduce_kernel, a);
}

cudaError_t launch_transpose32(const void* in, int64_t ld_in, int rows, int cols, void* out, int64_t ld_out,
                               cudaStream_t s, const DbgSpans& dbg) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(std::min(65535, (cols + kTrTile - 1) / kTrTile)),
                  static_cast<unsigned>(std::min(65535, (rows + kTrTile - 1) / kTrTile)));
  transpose32_kernel<<<grid, 256, 0, s>>>(static_cast<const uint32_t*>(in), ld_in, rows, cols,
                                          static_cast<uint32_t*>(out), ld_out, dbg);
  return cudaGetLastError();
}

cudaError_t launch_scale(int M, int N, void* D, int64_t ldd, const void* C, int64_t ldc, EpiParams e,
                         cudaStream_t s, int sms, const DbgSpans& dbg) {
  const int64_t items = static_cast<int64_t>(M) * N;
  static std::atomic<int64_t> occ{-1};
  scale_kernel<<<grid_for(items, 256, sms, resident_per_sm(scale_kernel, occ, 256, 0)), 256, 0, s>>>(
      M, N, D, ldd, C, ldc, e, dbg);
  return cudaGetLastError();
}

cudaError_t launch_watchdog_selftest(int* err, uint64_t timeout_ns, cudaStream_t s) {
  watchdog_selftest_kernel<<<1, 32, 0, s>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace dg
