// gemm_tc.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// What it computes ("Matrix Multiplication Background User's Guide", section
// 2.1, GPU Implementation, Fig. 1): the output is cut into TC_BM x BN tiles;
// each tile walks K in TC_BK steps, loading the A and B blocks it needs and
// accumulating their products ("Learning Triton One Kernel at a Time: Matrix
// Multiplication", section Tiled GEMM: partial dot products over blocks of the
// shared dimension sum to the same result).  Blocks are staged on chip and
// reused by every output of the tile ("GEMM kernels", section Improving the
// naive matrix multiplier: shared-memory tiles; register coarsening becomes
// the 128 x BN fp32 accumulator held in tensor memory).
//
// GB300 mapping:
//  - warp 0, one lane: TMA producer.  For each k-block it waits for a free
//    stage of an S-deep shared-memory ring (mbarrier "empty"), arms "full"
//    with the expected byte count and issues 2-D tensor-map loads of the A
//    and B blocks (128-byte swizzle, out-of-range elements read as zero, which
//    handles every ragged M/N/K edge -- the zero padding of the block-pointer
//    loads in "Learning Triton ...", section Triton implementation).
//  - warp 1, one lane: MMA issuer.  Waits for "full", issues TC_BK/16
//    tcgen05.mma (M=128, N=BN, K=16, kind::f16) into an fp32 accumulator in
//    tensor memory, and commits to "empty" so the stage is refilled as soon
//    as the tensor core is done with it.  At the end of a tile it commits to
//    "tmem_full".  Tensor memory holds two accumulators (2*BN columns), so the
//    epilogue of one tile overlaps the main loop of the next.
//  - warps 2-5: epilogue.  Each warp owns the 32 tensor-memory lanes (output
//    rows) that its warp index allows, reads 32-column slices with
//    tcgen05.ld, applies alpha/beta/LeakyReLU, converts with round-to-nearest-
//    even, writes a 32 x 128-byte swizzled box to shared memory and stores it
//    with one TMA store (coalesced 128-byte rows, clipped at the matrix edge).
//    With beta != 0 the same box of C is first TMA-loaded into that buffer.
//  - persistence: gridDim.x <= #SMs CTAs walk the work units
//    u = blockIdx.x, blockIdx.x + gridDim.x, ... ("GEMM kernels", section
//    Understanding the naive matrix multiplier: blocks are queued onto SMs and
//    stay there; here the queue is explicit).  Units are ordered slice-major,
//    then in groups of `raster_group` tile rows so that concurrently running
//    tiles share A and B blocks in L2.
//  - split-K: a unit may cover only a K slice of a tile; then the epilogue
//    writes raw fp32 partials to the workspace and a separate kernel sums the
//    slices in a fixed order ("Matrix Multiplication Background User's Guide",
//    section 2.3: splitting along K needs a final reduction).  The split may
//    cover every tile, or only the tiles of the last, partly filled wave: the
//    first whole waves then run whole tiles, and the tail tiles' slices fill
//    one more wave (section 3.2: a partial last wave leaves SMs idle).
//  - K pair (TC_KPAIR): the same reduction done on chip for two slices.  A
//    cluster of two CTAs takes one tile; CTA r runs the r-th half of the K
//    loop into its own tensor memory.  In the epilogue each CTA sends its
//    partial sums of the other CTA's half of the columns straight into that
//    CTA's staging buffers (st.async into distributed shared memory, counted
//    on the receiver's mbarrier), adds the partials it receives to its own
//    and finishes its half of the columns.  fp32 addition is commutative, so
//    both halves are summed in the same, fixed way, and the result equals the
//    two-slice reduction kernel's.
#pragma once

#include <atomic>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dg {

// TC_PAIR: a cluster of two CTAs computes one 256-row tile with .cta_group::2
// MMAs; each CTA stages its own 128 rows of A and half of the tile's BN columns
// of B, and holds its 128 rows of the accumulator in its tensor memory.
// TC_KPAIR: each CTA of a cluster of two stages whole 128 x BN tiles' blocks of
// one half of K; the exchange of partials goes through the staging buffers.
template <int BN, int MODE = TC_SOLO>
struct TcCfg {
  static constexpr bool PAIR = MODE == TC_PAIR;
  static constexpr bool KPAIR = MODE == TC_KPAIR;
  static constexpr int TILE_M = PAIR ? 2 * TC_BM : TC_BM;
  static constexpr int BN_CTA = PAIR ? BN / 2 : BN;   // B columns staged by one CTA
  static constexpr int A_STAGE = TC_BM * TC_BK * 2;  // 16 KB
  static constexpr int B_STAGE = BN_CTA * TC_BK * 2;
  static constexpr int STAGES = (192 * 1024) / (A_STAGE + B_STAGE);
  static constexpr int STG_BYTES = 32 * 128;         // one 32-row x 128-byte epilogue box
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
  static constexpr int OFF_STG = OFF_B + STAGES * B_STAGE;
  static constexpr int OFF_BAR = OFF_STG + TC_EPI_WARPS * 2 * STG_BYTES;
  // full[S], empty[S], tmem_full[2], tmem_empty[2], c_load[4], drain[1],
  // K pair: xfull[4] (the peer's partials have landed), xfree[4] (the peer's
  // staging buffers may be written)
  static constexpr int NUM_BARS = 2 * STAGES + 4 + TC_EPI_WARPS + 1 + 2 * TC_EPI_WARPS;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;  // tmem address, abort flag
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1024-B alignment
  static constexpr int TMEM_COLS = 2 * BN;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(TMEM_COLS <= 512, "tensor memory budget");
  static_assert(BN_CTA % 64 == 0, "B is staged in 64-column pieces");
  // K pair: each CTA finishes BN/2 columns, 64 per exchange round (the two
  // staging buffers of a warp hold 32 rows x 64 fp32 partials).
  static constexpr int KP_ROUNDS = BN / 128;
  static_assert(!KPAIR || BN >= 128, "a K pair finishes 64-column pieces");
  // On a cluster's last tile the A ring is idle once the accumulator is
  // complete: it holds the outgoing partials of every warp and round.
  static_assert(!KPAIR || KP_ROUNDS * TC_EPI_WARPS * 2 * STG_BYTES <= STAGES * A_STAGE, "send buffer");
  // ... and it holds one staging buffer per fp32 chunk of every epilogue warp
  // (the epilogue of a CTA's last unit).
  static_assert(TC_EPI_WARPS * (BN / 32) * STG_BYTES <= STAGES * (A_STAGE + B_STAGE), "last-unit staging");
};

struct Unit {
  int m_blk, n_blk, split, kb_begin, kb_end;
  int ws_tile;   // tail tile index (partial units)
  bool partial;  // a K slice of a tail tile: raw fp32 partials to the workspace
};

// Work unit u -> (tile, K range).  Units [0, dp_units) are whole tiles in
// raster order; the rest are K slices of the tail tiles, slice-major.
__device__ __forceinline__ Unit decode_unit(int u, const TcParams& p) {
  Unit x;
  int t;
  if (u < p.dp_units) {
    t = u;
    x.split = 0;
    x.ws_tile = 0;
    x.partial = false;
    x.kb_begin = 0;
    x.kb_end = p.k_blocks;
  } else {
    const int v = u - p.dp_units;
    x.split = v / p.tail_tiles;
    x.ws_tile = v - x.split * p.tail_tiles;
    x.partial = true;
    t = p.dp_units + x.ws_tile;
    x.kb_begin = x.split * p.kb_per_split;
    x.kb_end = min(p.k_blocks, x.kb_begin + p.kb_per_split);
  }
  tile_coords(t, p.num_m_blocks, p.num_n_blocks, p.raster_group, &x.m_blk, &x.n_blk);
  return x;
}

__device__ __forceinline__ uint32_t pack2(float a, float b, int out_kind) {
  if (out_kind == OUT_BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack2(uint32_t w, int out_kind) {
  if (out_kind == OUT_BF16) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
    return __bfloat1622float2(h);
  }
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}

// Four consecutive values of the C that beta scales, at (row, col .. col+3),
// as fp32; zero outside the matrix.  One 16- or 8-byte load when aligned.
__device__ __forceinline__ float4 load_cin4(const TcParams& p, int row, int col) {
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (row < p.M && col < p.N) {
    const int es = p.cin_kind == OUT_F32 ? 4 : 2;
    const uint8_t* src = static_cast<const uint8_t*>(p.cin) + (int64_t(row) * p.ldcin + col) * es;
#ifdef DG_DEBUG
    if (!DG_IN(p.dbg, src, min(4, p.N - col) * es, DBG_EPI_LOAD)) return make_float4(0.f, 0.f, 0.f, 0.f);
#endif
    if (col + 4 <= p.N && (reinterpret_cast<uintptr_t>(src) & uintptr_t(4 * es - 1)) == 0) {
      if (es == 4) return *reinterpret_cast<const float4*>(src);
      const uint2 w = *reinterpret_cast<const uint2*>(src);
      const float2 lo = unpack2(w.x, p.cin_kind), hi = unpack2(w.y, p.cin_kind);
      return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (col + i < p.N) {
        if (es == 4) {
          v[i] = reinterpret_cast<const float*>(src)[i];
        } else {
          const uint32_t h = reinterpret_cast<const uint16_t*>(src)[i];
          v[i] = unpack2(h, p.cin_kind).x;
        }
      }
    }
  }
  return make_float4(v[0], v[1], v[2], v[3]);
}

// Where the C that beta scales comes from, for one row segment.
enum CSource : int {
  C_NONE = 0,    // beta == 0: C is not read
  C_STAGED = 1,  // C is the output, TMA-loaded into the lane's staging line
  C_DIRECT = 2   // a separate C (or a K pair's), read from global memory
};

// Epilogue variants, compiled separately so that a tile's epilogue loop holds
// only the code its call can take: EPI_PLAIN (beta == 0; identity, LeakyReLU
// or ReLU), EPI_BETA (any C source; those activations), EPI_ALL (GELU, SiLU).
// With every variant inlined into one loop, the fp32 path of a 256-column
// chunk crossed tens of KB of code that it skipped, missed the instruction
// cache on every chunk (~0.5 us a chunk) and evicted the producer's and MMA
// issuer's code, which share the cache.
enum EpiVariant : int { EPI_PLAIN = 0, EPI_BETA = 1, EPI_ALL = 2 };

__device__ __forceinline__ int epi_variant(const TcParams& p, bool has_beta) {
  if (p.act >= 3) return EPI_ALL;
  return has_beta ? EPI_BETA : EPI_PLAIN;
}

// v <- alpha * v + beta * C (C_STAGED or C_DIRECT).
__device__ __forceinline__ void epi_beta(float (&v)[32], const TcParams& p, int csrc, const uint8_t* row_p,
                                         int sw, int chunk0, int esize, int row, int col0) {
  if (csrc == C_STAGED && esize == 4) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 c = *reinterpret_cast<const float4*>(row_p + (((chunk0 + j) ^ sw) << 4));
      v[4 * j + 0] = fmaf(p.beta, c.x, p.alpha * v[4 * j + 0]);
      v[4 * j + 1] = fmaf(p.beta, c.y, p.alpha * v[4 * j + 1]);
      v[4 * j + 2] = fmaf(p.beta, c.z, p.alpha * v[4 * j + 2]);
      v[4 * j + 3] = fmaf(p.beta, c.w, p.alpha * v[4 * j + 3]);
    }
  } else if (csrc == C_STAGED) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 c = *reinterpret_cast<const uint4*>(row_p + (((chunk0 + j) ^ sw) << 4));
      const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 cc = unpack2(w[t], p.out_kind);
        v[8 * j + 2 * t] = fmaf(p.beta, cc.x, p.alpha * v[8 * j + 2 * t]);
        v[8 * j + 2 * t + 1] = fmaf(p.beta, cc.y, p.alpha * v[8 * j + 2 * t + 1]);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 c = load_cin4(p, row, col0 + 4 * j);
      v[4 * j + 0] = fmaf(p.beta, c.x, p.alpha * v[4 * j + 0]);
      v[4 * j + 1] = fmaf(p.beta, c.y, p.alpha * v[4 * j + 1]);
      v[4 * j + 2] = fmaf(p.beta, c.z, p.alpha * v[4 * j + 2]);
      v[4 * j + 3] = fmaf(p.beta, c.w, p.alpha * v[4 * j + 3]);
    }
  }
}

// v <- act(v): identity, LeakyReLU and ReLU in every variant, GELU and SiLU in EPI_ALL.
template <int V>
__device__ __forceinline__ void epi_act(float (&v)[32], const TcParams& p) {
  if (p.act == 1) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = v[i] < 0.f ? v[i] * p.slope : v[i];
  } else if (p.act == 2) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = v[i] < 0.f ? 0.f : v[i];
  } else if constexpr (V == EPI_ALL) {
    if (p.act == 3) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = apply_act(v[i], 3, 0.f);
    } else if (p.act == 4) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = apply_act(v[i], 4, 0.f);
    }
  }
}

// v <- act(alpha * v + beta * C) on the 32 consecutive columns [col0, col0+32)
// of output row `row`.  C_STAGED: the 32 values start at 16-byte chunk
// `chunk0` of the lane's swizzled 128-byte staging line, in the output's
// format (esize bytes each).  Every run-time choice is taken once, outside
// the unrolled loops, so the path a launch takes is straight-line code.
template <int V>
__device__ __forceinline__ void epi32(float (&v)[32], const TcParams& p, int csrc, const uint8_t* row_p,
                                      int sw, int chunk0, int esize, int row, int col0) {
  if (V == EPI_PLAIN || csrc == C_NONE) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] *= p.alpha;
    return epi_act<V>(v, p);
  }
  if constexpr (V != EPI_PLAIN) epi_beta(v, p, csrc, row_p, sw, chunk0, esize, row, col0);
  epi_act<V>(v, p);
}

// The epilogue's inputs, read from the kernel parameters once into registers
// (the in-kernel split-K reduction applies the epilogue to many outputs per
// thread).
struct Fin {
  const void* cin;
  int64_t ldcin;
  int cin_kind;
  void* c;
  int64_t ldc;
  int out_kind;
  int M, N;
  float alpha, beta, slope;
  int act;
#ifdef DG_DEBUG
  const DbgSpans* dbg;
#endif
};

__device__ __forceinline__ Fin fin_of(const TcParams& p) {
#ifdef DG_DEBUG
  return Fin{p.cin, p.ldcin, p.cin_kind, p.c_ptr, p.ldc, p.out_kind, p.M, p.N, p.alpha, p.beta, p.slope, p.act, &p.dbg};
#else
  return Fin{p.cin, p.ldcin, p.cin_kind, p.c_ptr, p.ldc, p.out_kind, p.M, p.N, p.alpha, p.beta, p.slope, p.act};
#endif
}

// The four values of the C that beta scales at (row, col .. col+3), zero
// outside the matrix.
__device__ __forceinline__ float4 fin_c4(const Fin& f, int row, int col) {
  float c[4] = {0.f, 0.f, 0.f, 0.f};
  if (row < f.M && col < f.N) {
    const int nn = min(4, f.N - col);
    const int es = f.cin_kind == OUT_F32 ? 4 : 2;
    const uint8_t* src = static_cast<const uint8_t*>(f.cin) + (int64_t(row) * f.ldcin + col) * es;
#ifdef DG_DEBUG
    if (!DG_IN(*f.dbg, src, nn * es, DBG_SPLIT)) return make_float4(0.f, 0.f, 0.f, 0.f);
#endif
    if (nn == 4 && (reinterpret_cast<uintptr_t>(src) & uintptr_t(4 * es - 1)) == 0) {
      if (es == 4) return *reinterpret_cast<const float4*>(src);
      const uint2 w = *reinterpret_cast<const uint2*>(src);
      const float2 lo = unpack2(w.x, f.cin_kind), hi = unpack2(w.y, f.cin_kind);
      return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    for (int j = 0; j < nn; ++j)
      c[j] = es == 4 ? reinterpret_cast<const float*>(src)[j]
                     : unpack2(reinterpret_cast<const uint16_t*>(src)[j], f.cin_kind).x;
  }
  return make_float4(c[0], c[1], c[2], c[3]);
}

// v <- act(alpha * v + beta * C) for 16 values (four groups of four columns),
// with the arithmetic of the tile reduction kernel so that both give the same
// bits.  Every run-time choice is taken once for the 16 values: with the
// activation switch inside an unrolled per-value loop, the executed path was
// spread over tens of KB of code and every batch missed the instruction cache.
__device__ __forceinline__ void fin_epilogue16(float (&v)[16], const Fin& f, const int (&row)[4],
                                               const int (&col)[4]) {
  if (f.beta != 0.f) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 c = fin_c4(f, row[j], col[j]);
      v[4 * j + 0] = fmaf(f.beta, c.x, f.alpha * v[4 * j + 0]);
      v[4 * j + 1] = fmaf(f.beta, c.y, f.alpha * v[4 * j + 1]);
      v[4 * j + 2] = fmaf(f.beta, c.z, f.alpha * v[4 * j + 2]);
      v[4 * j + 3] = fmaf(f.beta, c.w, f.alpha * v[4 * j + 3]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = f.alpha * v[i];
  }
  switch (f.act) {
    case 0:
      break;
    case 1:
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = v[i] < 0.f ? v[i] * f.slope : v[i];
      break;
    case 2:
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = v[i] < 0.f ? 0.f : v[i];
      break;
    case 3:
      for (int i = 0; i < 16; ++i) v[i] = apply_act(v[i], 3, 0.f);
      break;
    default:
      for (int i = 0; i < 16; ++i) v[i] = apply_act(v[i], 4, 0.f);
      break;
  }
}

// Split-K reduced inside the GEMM kernel ("Matrix Multiplication Background
// User's Guide", section 2.3: K slices need a final reduction), run by the
// four epilogue warps of a CTA after the last unit it computes, a K slice of
// tail tile `tile`, whose raw fp32 partials it has stored (TMA) into the
// workspace.  The CTA publishes them (their stores complete, a proxy fence,
// a release add on the tile's counter), waits until all `parts` = slices x
// CTAs per unit have done so, then takes share `part` of the tile's
// elements: one bulk load per slice brings that share of every slice into
// its idle operand ring, and each output is summed over slices 0 .. S-1 in
// order -- the order of the tile reduction kernel -- before the epilogue.
// Each thread carries four outputs at a time (independent chains of shared
// memory loads and adds).  The results, in the output's type, go back into
// the ring (fp32 in place of slice 0, which each thread has read; 16-bit after
// the slices) at addresses that share the 16-byte alignment of their place
// in C, and one thread writes every row segment of the share with a 1-D bulk
// store (plain stores for the unaligned ends): a few warps' plain global
// stores, on an SM whose shared memory is almost all carved out, measured
// ~5 GB/s per SM.  The counter goes back to zero once all parts have seen it
// complete.  `gather` counts one arrival per epilogue warp (phase 0 before the
// release, phase 1 once the results are in the ring); `bar` takes the bulk
// loads.  Both are fresh and every wait is bounded.
template <int TILE_M, int BN>
__device__ __forceinline__ void fused_split_reduce(const TcParams& p, int tile, int part, int parts, int m_blk,
                                                   int n_blk, uint32_t ring, uint32_t gather, uint32_t bar,
                                                   const Watch& w) {
  const int ept = int(threadIdx.x) - 2 * 32;  // 0 .. 127 over the epilogue warps
  const int lane = int(threadIdx.x) & 31;
  constexpr uint32_t kAll = 0xffffffffu;
  // Every wait is taken by the whole warp through __all_sync (the lanes leave
  // it together, converged), and single-lane work is followed by __syncwarp()
  // before the warp waits: lanes that left a bounded wait at different times,
  // or that spin while one lane works, make the warp run its lanes' paths one
  // after another.
  if (lane == 0) {
    bulk_wait<0>();              // this warp's partial stores have been written ...
    fence_proxy_async_global();  // ... and come before the release below
    mbar_arrive(gather);
  }
  __syncwarp();
  const Fin fin = fin_of(p);
  unsigned* const cnt = p.counters + tile;
  const float* const ws = p.ws;
  const int tail_tiles = p.tail_tiles;
  if (!__all_sync(kAll, wait_bar(gather, 0, w, WAIT_SPLIT_PEERS))) return;  // all four warps' stores
  const unsigned target = unsigned(parts);
  constexpr int F = TILE_M * BN / 4;  // float4s in the tile
  const int share = (F + parts - 1) / parts;
  const int f0 = min(F, part * share), f1 = min(F, f0 + share);
  const uint32_t share_bytes = uint32_t(f1 - f0) * 16u;
  const int splits = parts / (TILE_M / TC_BM);
#ifdef DG_DEBUG
  if (!DG_IN(p.dbg, cnt, 4, DBG_SPLIT)) return;  // (the peers' waits for this part run out)
#endif
  if (ept < 32) {
    if (lane == 0) {
      __threadfence();
      red_release_add(cnt, 1u);
      if (wait_counter(cnt, target, w, WAIT_SPLIT_PEERS)) {
        fence_proxy_async_global();  // the bulk loads read what the releases published
        mbar_arrive_expect_tx(bar, share_bytes * uint32_t(splits));
        if (share_bytes > 0) {
          const int64_t slice = int64_t(tail_tiles) * TILE_M * BN;
          const float* src = ws + int64_t(tile) * TILE_M * BN + int64_t(f0) * 4;
          for (int sl = 0; sl < splits; ++sl)
            if (DG_IN(p.dbg, src + sl * slice, share_bytes, DBG_SPLIT))
              bulk_load_1d(ring + sl * share_bytes, src + sl * slice, share_bytes, bar);
        }
      }
    }
    __syncwarp();
  }
  if (!__all_sync(kAll, wait_bar(bar, 0, w, WAIT_SPLIT_LOAD))) return;  // (also when lane 0 gave up: abort flag)
  const int es = fin.out_kind == OUT_F32 ? 4 : 2;
  const int e0 = 4 * f0, e1 = 4 * f1;  // the share's tile elements
  // results: element e of the tile at out + (e - e0) * es, out = e0 * es (mod 16)
  const uint32_t out = (es == 4 ? ring : ((ring + uint32_t(splits) * share_bytes + 15u) & ~15u)) +
                       (uint32_t(e0 * es) & 15u);
  constexpr int T = TC_EPI_WARPS * 32;
  for (int fb = f0 + ept; fb < f1; fb += 4 * T) {
    float4 acc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int f = min(fb + j * T, f1 - 1);  // (a clamped duplicate is summed but not stored)
      acc[j] = ld_shared_f4(ring + uint32_t(f - f0) * 16u);
    }
    for (int sl = 1; sl < splits; ++sl) {
      const uint32_t src = ring + uint32_t(sl) * share_bytes;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int f = min(fb + j * T, f1 - 1);
        const float4 v = ld_shared_f4(src + uint32_t(f - f0) * 16u);
        acc[j].x += v.x;
        acc[j].y += v.y;
        acc[j].z += v.z;
        acc[j].w += v.w;
      }
    }
    float v[16];
    int rows[4], cols[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * (fb + j * T);
      const int r = e / BN;
      rows[j] = m_blk * TILE_M + r;
      cols[j] = n_blk * BN + (e - r * BN);
      v[4 * j + 0] = acc[j].x;
      v[4 * j + 1] = acc[j].y;
      v[4 * j + 2] = acc[j].z;
      v[4 * j + 3] = acc[j].w;
    }
    fin_epilogue16(v, fin, rows, cols);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int f = fb + j * T;
      if (f < f1) {
        const uint32_t dst = out + uint32_t(4 * f - e0) * uint32_t(es);
        if (es == 4)
          st_shared_f4(dst, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
        else
          st_shared_u2(dst, pack2(v[4 * j], v[4 * j + 1], fin.out_kind), pack2(v[4 * j + 2], v[4 * j + 3], fin.out_kind));
      }
    }
  }
  fence_proxy_async_smem();  // the bulk stores read these results through the async proxy
  __syncwarp();
  if (lane == 0) mbar_arrive(gather);
  __syncwarp();
  if (!__all_sync(kAll, wait_bar(gather, 1, w, WAIT_SPLIT_LOAD))) return;  // every warp's results are in
  // One row segment of C per tile row the share touches, rows spread over the
  // 128 threads: a 1-D bulk store for its 16-byte aligned part, plain stores
  // for the ends.
  const int epb = 16 / es;  // elements per 16 bytes
  for (int r = e0 / BN + ept; r * BN < e1; r += T) {
    const int row = m_blk * TILE_M + r;
    if (row >= fin.M) break;
    const int c_lo = max(e0, r * BN) - r * BN, c_hi = min(e1, (r + 1) * BN) - r * BN;
    const int g_lo = n_blk * BN + c_lo, g_hi = min(n_blk * BN + c_hi, fin.N);
    if (g_lo >= g_hi) continue;
    const int a_lo = min(g_hi, (g_lo + epb - 1) / epb * epb);
    const int a_hi = max(a_lo, g_hi / epb * epb);
    uint8_t* const crow = static_cast<uint8_t*>(fin.c) + int64_t(row) * fin.ldc * es;
    auto src_of = [&](int g) { return out + uint32_t(r * BN + (g - n_blk * BN) - e0) * uint32_t(es); };
    if (a_lo < a_hi && DG_IN(p.dbg, crow + int64_t(a_lo) * es, int64_t(a_hi - a_lo) * es, DBG_SPLIT))
      bulk_store_1d(crow + int64_t(a_lo) * es, src_of(a_lo), uint32_t(a_hi - a_lo) * uint32_t(es));
    for (int g = g_lo; g < g_hi; ++g) {  // the unaligned ends, element by element
      if (g == a_lo) g = a_hi;
      if (g >= g_hi) break;
      if (!DG_IN(p.dbg, crow + int64_t(g) * es, es, DBG_SPLIT)) continue;
      if (es == 4)
        *reinterpret_cast<uint32_t*>(crow + int64_t(g) * 4) = ld_shared_u32(src_of(g));
      else
        *reinterpret_cast<uint16_t*>(crow + int64_t(g) * 2) = uint16_t(ld_shared_u16(src_of(g)));
    }
  }
  bulk_commit();
  bulk_wait_read<0>();  // this thread's bulk stores have read the ring before the CTA exits
  __syncwarp();
  if (ept == 0) {
    const unsigned old = atomicAdd(cnt, 1u);
    if (old == 2u * target - 1u) atomicExch(cnt, 0u);  // every part has seen the count complete
  }
}

// The TC_BK/16 MMAs of one ring stage (each reads 32 bytes of K per row:
// 16 bf16/fp16 or 8 TF32 elements), accumulating unless this is the first
// stage of the unit.
template <bool PAIR, bool TF32>
__device__ __forceinline__ void issue_stage(uint32_t d_tmem, uint32_t sa, uint32_t sb, uint32_t lbo_a,
                                            uint32_t lbo_b, uint32_t kstep_a, uint32_t kstep_b, uint32_t lay_a,
                                            uint32_t lay_b, uint32_t idesc, bool first) {
#pragma unroll
  for (int kk = 0; kk < TC_BK / 16; ++kk) {
    // (32-byte swizzle atoms are four 128-byte rows deep, 16-byte ones eight)
    const uint64_t ad = smem_desc_sw128(sa + kk * kstep_a, lbo_a, lay_a == SMEM_SW128_ATOM32 ? 512 : 1024, lay_a);
    const uint64_t bd = smem_desc_sw128(sb + kk * kstep_b, lbo_b, lay_b == SMEM_SW128_ATOM32 ? 512 : 1024, lay_b);
    const uint32_t accum = (!first || kk > 0) ? 1u : 0u;
    if constexpr (PAIR && TF32)
      tc_mma_tf32_pair(d_tmem, ad, bd, idesc, accum);
    else if constexpr (PAIR)
      tc_mma_f16_pair(d_tmem, ad, bd, idesc, accum);
    else if constexpr (TF32)
      tc_mma_tf32(d_tmem, ad, bd, idesc, accum);
    else
      tc_mma_f16(d_tmem, ad, bd, idesc, accum);
  }
}

// TF32: operands are TF32 (fp32 words; kind::tf32 MMAs, 32 K elements per
// k-block); a compile-time choice, so the 16-bit kernels carry none of it.
template <int BN, int MODE, bool TF32 = false>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ TcParams p) {
  using Cfg = TcCfg<BN, MODE>;
  constexpr bool PAIR = Cfg::PAIR;
  constexpr bool KPAIR = Cfg::KPAIR;
  constexpr bool CLUSTER = MODE != TC_SOLO;
  constexpr int S = Cfg::STAGES;
  constexpr int BNC = Cfg::BN_CTA;
  const uint32_t rank = CLUSTER ? cluster_ctarank() : 0u;
  const bool leader = !PAIR || rank == 0;  // issues MMAs (only CTA 0 of a 256-row pair)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = base + Cfg::OFF_BAR;
  const uint32_t full0 = bar0, empty0 = bar0 + 8 * S;
  const uint32_t tfull0 = bar0 + 16 * S, tempty0 = tfull0 + 16;
  const uint32_t cload0 = tempty0 + 16, drain_bar = cload0 + 8 * TC_EPI_WARPS;
  const uint32_t xfull0 = drain_bar + 8, xfree0 = xfull0 + 8 * TC_EPI_WARPS;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sbase + Cfg::OFF_MISC);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(sbase + Cfg::OFF_MISC + 4);

  // Units: a cluster walks tiles; a K pair's CTA r takes the r-th K half.
  const int cta0 = CLUSTER ? int(blockIdx.x) / 2 : int(blockIdx.x);
  const int ncta = CLUSTER ? int(gridDim.x) / 2 : int(gridDim.x);
  auto unit_of = [&](int u) {
    Unit x = decode_unit(u, p);
    if constexpr (KPAIR) {
      x.split = int(rank);
      x.kb_begin = int(rank) * p.kb_per_split;
      x.kb_end = min(p.k_blocks, x.kb_begin + p.kb_per_split);
    }
    return x;
  };
  // One ring stage's loads (producer thread): this CTA's rows of A and
  // columns of B for k-block kb of unit x.  A pair's loads complete on the
  // leader's barrier, which the leader arms with both CTAs' bytes.
  auto issue_loads = [&](int stage, const Unit& x, int kb) {
    constexpr int kbe = TF32 ? TC_BK_TF32 : TC_BK;
    const int m0 = x.m_blk * Cfg::TILE_M + (PAIR ? int(rank) * TC_BM : 0);
    const int n0 = x.n_blk * BN + (PAIR ? int(rank) * BNC : 0);
    const uint32_t fb = full0 + 8 * stage;
    const uint32_t sa = base + Cfg::OFF_A + stage * Cfg::A_STAGE;
    const uint32_t sb = base + Cfg::OFF_B + stage * Cfg::B_STAGE;
    const int k0 = kb * kbe;
    uint32_t fbc = fb;
    if constexpr (PAIR) fbc = mapa_shared(fb, 0);
    if (leader) mbar_arrive_expect_tx(fb, (PAIR ? 2 : 1) * (Cfg::A_STAGE + Cfg::B_STAGE));
    auto load = [&](uint32_t dst, const CUtensorMap* m, int cx, int cy) {
      if (!DG_TMA(p.dbg, cx, cy, TF32 ? 4 : 2, false)) return;  // (its barrier never completes)
      if constexpr (PAIR)
        tma_load_2d_pair(dst, m, fbc, cx, cy);
      else
        tma_load_2d(dst, m, fb, cx, cy);
    };
    // K-major: one box of the tile's rows x one 128-byte row of K.  M/N-major:
    // boxes of kbe K rows x kbe elements of M or N (128 bytes), one per
    // 128-byte piece of the tile's rows, each a column of swizzle atoms.
    if (!p.a_mn_major) {
      load(sa, &tmA, k0, m0);  // 128 rows x kbe K
    } else {
#pragma unroll
      for (int j = 0; j < TC_BM / kbe; ++j) load(sa + j * kbe * 128, &tmA, m0 + kbe * j, k0);
    }
    if (!p.b_mn_major) {
      load(sb, &tmB, k0, n0);  // BNC rows x kbe K
    } else {
#pragma unroll
      for (int j = 0; j < BNC / kbe; ++j) load(sb + j * kbe * 128, &tmB, n0 + kbe * j, k0);
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, PAIR ? 2 * TC_EPI_WARPS : TC_EPI_WARPS);  // both CTAs' epilogues
    }
    for (int e = 0; e < TC_EPI_WARPS; ++e) {
      mbar_init(cload0 + 8 * e, 1);
      mbar_init(xfull0 + 8 * e, 1);  // own arrive.expect_tx; the peer's bytes complete it
      // one arrival from the peer per exchange round; outside a K pair, xfree[0]
      // gathers the epilogue warps before an in-kernel split-K reduction
      mbar_init(xfree0 + 8 * e, (KPAIR || e > 0) ? 1 : TC_EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
    if (p.tail_tiles > 0) prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), Cfg::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (CLUSTER)
    cluster_sync();  // both CTAs' barriers exist before either signals the other
  else
    __syncthreads();
  tc_fence_after();
  // Launched as a programmatic dependent, the prologue above overlapped the
  // previous kernel's tail; its results are needed from here on.
  wait_prior_grid();
  const uint32_t tmem_base = *tmem_slot;
  // A dependent grid (the split-K reduction) may be scheduled now; it waits
  // for this grid's completion before it reads anything.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const Watch w{abort_flag, p.err, p.timeout_ns};
  // Bounded wait; cluster-scope acquire when the peer CTA signals (a pair's
  // shared pipeline).  A K pair's pipeline is its own; only its exchange
  // barriers hear from the peer.
  auto wait = [&](uint32_t bar, uint32_t parity, int code) {
    if constexpr (PAIR) return wait_bar_cluster(bar, parity, w, code);
    return wait_bar(bar, parity, w, code);
  };
  auto wait_peer = [&](uint32_t bar, uint32_t parity, int code) {
    return wait_bar_cluster(bar, parity, w, code);
  };
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int u = cta0; u < p.units && ok; u += ncta) {
        const Unit x = unit_of(u);
        for (int kb = x.kb_begin; kb < x.kb_end; ++kb) {
          if (!wait(empty0 + 8 * stage, phase ^ 1u, WAIT_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          issue_loads(stage, x, kb);
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let the loads already in flight land before the CTA can exit.
        for (int s = 0; s < S; ++s) {
          const int n_s = issued > s ? (issued - s + S - 1) / S : 0;
          if (n_s > 0 && leader) wait(full0 + 8 * s, (uint32_t)((n_s - 1) & 1), 0);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && leader) {
      // M/N-major operands: the next column of swizzle atoms along M or N is
      // one box (kbe K rows of 128 bytes) further, and one MMA's K (16
      // elements, 8 for TF32) spans that many 128-byte rows; TF32 tiles stored
      // M/N-major are swizzled in 32-byte units.  K-major: the MMA's K is 32
      // bytes of each row.
      constexpr uint32_t kbe = TF32 ? TC_BK_TF32 : TC_BK;
      constexpr uint32_t mma_k = TF32 ? 8 : 16;
      const uint32_t lbo_a = p.a_mn_major ? kbe * 128 : 16;
      const uint32_t lbo_b = p.b_mn_major ? kbe * 128 : 16;
      const uint32_t kstep_a = p.a_mn_major ? mma_k * 128 : 32;
      const uint32_t kstep_b = p.b_mn_major ? mma_k * 128 : 32;
      const uint32_t lay_a = TF32 && p.a_mn_major ? SMEM_SW128_ATOM32 : SMEM_SW128;
      const uint32_t lay_b = TF32 && p.b_mn_major ? SMEM_SW128_ATOM32 : SMEM_SW128;
      const uint32_t idesc = p.idesc;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = cta0; u < p.units && ok; u += ncta) {
        const Unit x = unit_of(u);
        if (!wait(tempty0 + 8 * acc, acc_phase ^ 1u, WAIT_MMA_TMEM_EMPTY)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = x.kb_begin; kb < x.kb_end; ++kb) {
          if (!wait(full0 + 8 * stage, phase, WAIT_MMA_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + Cfg::OFF_A + stage * Cfg::A_STAGE;
          const uint32_t sb = base + Cfg::OFF_B + stage * Cfg::B_STAGE;
          issue_stage<PAIR, TF32>(d_tmem, sa, sb, lbo_a, lbo_b, kstep_a, kstep_b, lay_a, lay_b, idesc,
                                  kb == x.kb_begin);
          // stage free (in both CTAs of a pair) once these MMAs finish
          if constexpr (PAIR)
            tc_commit_pair_multicast(empty0 + 8 * stage, 0x3);
          else
            tc_commit(empty0 + 8 * stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // accumulator ready for the epilogue (of both CTAs of a pair)
        if constexpr (PAIR)
          tc_commit_pair_multicast(tfull0 + 8 * acc, 0x3);
        else
          tc_commit(tfull0 + 8 * acc);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Every MMA issued by this thread completes before tensor memory is freed.
      if constexpr (PAIR)
        tc_commit_pair_multicast(drain_bar, 0x1);
      else
        tc_commit(drain_bar);
      wait(drain_bar, 0, WAIT_DRAIN);
    }
  } else if constexpr (KPAIR) {
    // ------------------------------------------------- epilogue of a K pair
    // Warp e of each CTA reads tensor-memory lanes 32q..32q+31 (tile rows) and
    // trades with warp e of the peer.  Per round: my two staging buffers are
    // free (my stores from them are done) -> tell the peer and arm my receive;
    // send my partials of the peer's 64 columns into the peer's buffers once
    // the peer says they are free; wait for the peer's partials of my 64
    // columns, add, apply the epilogue in place and store with TMA.
    const int e = warp - 2;
    const int q = warp & 3;
    const uint32_t peer = rank ^ 1u;
    const bool has_beta = p.beta != 0.f;
    const int esize = p.out_kind == OUT_F32 ? 4 : 2;
    const uint32_t stg0 = base + Cfg::OFF_STG + e * 2 * Cfg::STG_BYTES;
    uint8_t* const stg_p0 = sbase + Cfg::OFF_STG + e * 2 * Cfg::STG_BYTES;
    const uint32_t xfull = xfull0 + 8 * e, xfree = xfree0 + 8 * e;
    const uint32_t peer_stg0 = mapa_shared(stg0, peer);
    const uint32_t peer_stg = peer_stg0 + lane * 128;
    const uint32_t peer_xfull = mapa_shared(xfull, peer);
    const uint32_t peer_xfree = mapa_shared(xfree, peer);
    const int sw = lane & 7;  // 128-byte swizzle: 16-byte chunk j of row r lives at j ^ (r % 8)
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t xphase = 0;
    bool ok = true;
    // My staging buffers are free once my earlier stores from them have read
    // them: tell the peer and arm my receive.  (The peer can only send for the
    // next round after this warp has waited for the peer's data of this one,
    // so no arrival ever runs a phase ahead.)
    auto free_and_arm = [&]() {
      if (lane == 0) {
        bulk_wait_read<0>();
        mbar_arrive_cluster(peer_xfree);
        mbar_arrive_expect_tx(xfull, 2 * Cfg::STG_BYTES);
      }
      __syncwarp();
    };
    for (int u = cta0; u < p.units && ok; u += ncta) {
      const Unit x = unit_of(u);
      // Round 0's handshake does not need the accumulator: it overlaps the
      // tile's last MMAs instead of following them.
      free_and_arm();
      if (!__all_sync(0xffffffffu, wait(tfull0 + 8 * acc, acc_phase, WAIT_EPI_TMEM_FULL))) break;
      tc_fence_after();
      const int y0 = x.m_blk * TC_BM + 32 * q;
      const int row = y0 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                             static_cast<uint32_t>(acc * BN);
      // one compiled copy of the exchange rounds per epilogue variant, chosen per tile
      auto rounds = [&](auto variant) {
      constexpr int V = decltype(variant)::value;
      for (int rd = 0; rd < Cfg::KP_ROUNDS; ++rd) {
        const int own_c = int(rank) * (BN / 2) + rd * 64;  // tile columns finished here
        const int peer_c = int(peer) * (BN / 2) + rd * 64;
        if (rd > 0) free_and_arm();
        {
          uint32_t r0[32], r1[32];
          tmem_ld_32x32b_x32(t_row + peer_c, r0);
          tmem_ld_32x32b_x32(t_row + peer_c + 32, r1);
          tmem_ld_wait(r0);
          tmem_ld_wait(r1);
          // The cluster's last tile: no stage will be refilled, so the partials
          // go through this warp's 8 KB of the idle A ring and move as one
          // bulk copy (faster over distributed shared memory than 16-byte
          // stores); an earlier tile sends them with st.async.
          const bool last = u + ncta >= p.units;
          const uint32_t snd = base + Cfg::OFF_A + (rd * TC_EPI_WARPS + e) * 2 * Cfg::STG_BYTES;
          if (last) {
            uint8_t* const snd_p = sbase + Cfg::OFF_A + (rd * TC_EPI_WARPS + e) * 2 * Cfg::STG_BYTES + lane * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int off = (j ^ sw) << 4;
              *reinterpret_cast<uint4*>(snd_p + off) = make_uint4(r0[4 * j], r0[4 * j + 1], r0[4 * j + 2], r0[4 * j + 3]);
              *reinterpret_cast<uint4*>(snd_p + Cfg::STG_BYTES + off) =
                  make_uint4(r1[4 * j], r1[4 * j + 1], r1[4 * j + 2], r1[4 * j + 3]);
            }
            fence_proxy_async_smem();  // the copy reads them through the async proxy
          }
          if (!__all_sync(0xffffffffu, wait_peer(xfree, xphase, WAIT_EPI_EXCHANGE))) {
            ok = false;
            break;
          }
          if (last) {
            if (lane == 0) bulk_copy_to_cluster(peer_stg0, snd, 2 * Cfg::STG_BYTES, peer_xfull);
            __syncwarp();  // the copy is issued before any lane of this warp waits
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t off = uint32_t((j ^ sw) << 4);
              st_async_v4(peer_stg + off, r0[4 * j], r0[4 * j + 1], r0[4 * j + 2], r0[4 * j + 3], peer_xfull);
              st_async_v4(peer_stg + Cfg::STG_BYTES + off, r1[4 * j], r1[4 * j + 1], r1[4 * j + 2],
                          r1[4 * j + 3], peer_xfull);
            }
          }
        }
        if (!__all_sync(0xffffffffu, wait_peer(xfull, xphase, WAIT_EPI_EXCHANGE))) {
          ok = false;
          break;
        }
        xphase ^= 1u;
        if (esize == 4) {
          for (int c = 0; c < 2; ++c) {
            const int x0 = x.n_blk * BN + own_c + 32 * c;
            uint8_t* const row_p = stg_p0 + c * Cfg::STG_BYTES + lane * 128;
            uint32_t r[32];
            tmem_ld_32x32b_x32(t_row + own_c + 32 * c, r);
            tmem_ld_wait(r);
            float v[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {  // own partial sums + the peer's
              const float4 pv = *reinterpret_cast<const float4*>(row_p + ((j ^ sw) << 4));
              v[4 * j + 0] = __uint_as_float(r[4 * j + 0]) + pv.x;
              v[4 * j + 1] = __uint_as_float(r[4 * j + 1]) + pv.y;
              v[4 * j + 2] = __uint_as_float(r[4 * j + 2]) + pv.z;
              v[4 * j + 3] = __uint_as_float(r[4 * j + 3]) + pv.w;
            }
            epi32<V>(v, p, has_beta ? C_DIRECT : C_NONE, row_p, sw, 0, 4, row, x0);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<float4*>(row_p + ((j ^ sw) << 4)) =
                  make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            const int tail_lo = max(x0, p.n_tma), tail_hi = min(x0 + 32, p.N);
            if (tail_lo < tail_hi && row < p.M) {
              for (int col = tail_lo; col < tail_hi; ++col) {
                const int b = (col - x0) * 4;
                uint8_t* const dst = static_cast<uint8_t*>(p.c_ptr) + (int64_t(row) * p.ldc + col) * 4;
                if (!DG_IN(p.dbg, dst, 4, DBG_EPI_STORE)) continue;
                *reinterpret_cast<float*>(dst) = *reinterpret_cast<const float*>(row_p + (((b >> 4) ^ sw) << 4) + (b & 15));
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (x0 < p.n_tma && DG_TMA(p.dbg, x0, y0, 4, true)) tma_store_2d(&tmC, stg0 + c * Cfg::STG_BYTES, x0, y0);
              bulk_commit();
            }
          }
        } else {
          const int x0 = x.n_blk * BN + own_c;
          uint32_t r0[32], r1[32];
          tmem_ld_32x32b_x32(t_row + own_c, r0);
          tmem_ld_32x32b_x32(t_row + own_c + 32, r1);
          tmem_ld_wait(r0);
          tmem_ld_wait(r1);
          // the peer's partials of my 64 columns, whole row first (the bf16 /
          // fp16 result is then written over the first buffer)
          float pv[64];
          uint8_t* const row_p = stg_p0 + lane * 128;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float4 v = *reinterpret_cast<const float4*>(row_p + (j >> 3) * Cfg::STG_BYTES +
                                                              (((j & 7) ^ sw) << 4));
            pv[4 * j] = v.x;
            pv[4 * j + 1] = v.y;
            pv[4 * j + 2] = v.z;
            pv[4 * j + 3] = v.w;
          }
          float v0[32], v1[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {  // own partial sums + the peer's
            v0[i] = __uint_as_float(r0[i]) + pv[i];
            v1[i] = __uint_as_float(r1[i]) + pv[32 + i];
          }
          const int csrc = has_beta ? C_DIRECT : C_NONE;
          epi32<V>(v0, p, csrc, row_p, sw, 0, 2, row, x0);
          epi32<V>(v1, p, csrc, row_p, sw, 4, 2, row, x0 + 32);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float* h = j < 4 ? &v0[8 * (j & 3)] : &v1[8 * (j & 3)];
            *reinterpret_cast<uint4*>(row_p + ((j ^ sw) << 4)) =
                make_uint4(pack2(h[0], h[1], p.out_kind), pack2(h[2], h[3], p.out_kind),
                           pack2(h[4], h[5], p.out_kind), pack2(h[6], h[7], p.out_kind));
          }
          const int tail_lo = max(x0, p.n_tma), tail_hi = min(x0 + 64, p.N);
          if (tail_lo < tail_hi && row < p.M) {
            for (int col = tail_lo; col < tail_hi; ++col) {
              const int b = (col - x0) * 2;
              uint8_t* const dst = static_cast<uint8_t*>(p.c_ptr) + (int64_t(row) * p.ldc + col) * 2;
              if (!DG_IN(p.dbg, dst, 2, DBG_EPI_STORE)) continue;
              *reinterpret_cast<uint16_t*>(dst) = *reinterpret_cast<const uint16_t*>(row_p + (((b >> 4) ^ sw) << 4) + (b & 15));
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (x0 < p.n_tma && DG_TMA(p.dbg, x0, y0, 2, true)) tma_store_2d(&tmC, stg0, x0, y0);
            bulk_commit();
          }
        }
      }
      };
      const int variant = epi_variant(p, has_beta);
      if (variant == EPI_PLAIN)
        rounds(std::integral_constant<int, EPI_PLAIN>{});
      else if (variant == EPI_BETA)
        rounds(std::integral_constant<int, EPI_BETA>{});
      else
        rounds(std::integral_constant<int, EPI_ALL>{});
      if (!ok) break;
      // this warp's reads of the accumulator are complete: release it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    // Every partial sum the peer sends this warp has arrived (or the warp gave
    // up): its side of the exchange is over.
    cluster_arrive();
    // The stores must have read the staging buffers before the CTA exits; the
    // grid's completion covers their writes to global memory.
    if (lane == 0) bulk_wait_read<0>();
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - 2;  // staging buffers / C-load barrier of this warp
    const int q = warp & 3;  // tensor-memory lane quarter this warp may read
    const uint32_t stg0 = base + Cfg::OFF_STG + e * 2 * Cfg::STG_BYTES;
    uint8_t* const stg_p0 = sbase + Cfg::OFF_STG + e * 2 * Cfg::STG_BYTES;
    int acc = 0;
    uint32_t acc_phase = 0;
    int sbuf = 0;
    uint32_t cphase = 0;
    bool ok = true;
    Unit fused{};  // the K slice this CTA reduces in the kernel (fused_reduce: its last unit)
    fused.ws_tile = -1;
    for (int u = cta0; u < p.units && ok; u += ncta) {
      const Unit x = unit_of(u);
      if (x.partial && p.fused_reduce) fused = x;
      // All lanes wait; the warp leaves together if any lane gave up, because the
      // tcgen05.ld below must be executed by the whole warp.
      if (!__all_sync(0xffffffffu, wait(tfull0 + 8 * acc, acc_phase, WAIT_EPI_TMEM_FULL)))
        break;
      tc_fence_after();
      // A partial unit stores raw fp32 sums into its slice's copy of the tile
      // in the workspace (BN columns wide, no ragged edge); a whole tile
      // stores the epilogue's result into C.
      const bool partial = x.partial;
      const bool has_beta = !partial && p.beta != 0.f;
      // beta's C through the output's tensor map (it is the output), or with
      // plain loads (a separate C of its own type and leading dimension)
      const bool c_tma = has_beta && !p.cin_direct;
      const int csrc = c_tma ? C_STAGED : (has_beta ? C_DIRECT : C_NONE);
      const int esize = (partial || p.out_kind == OUT_F32) ? 4 : 2;
      const int cw = 128 / esize;  // columns per 128-byte box row
      const CUtensorMap* const out_map = partial ? &tmW : &tmC;
      const int n0 = partial ? 0 : x.n_blk * BN;
      const int row0 = x.m_blk * Cfg::TILE_M + int(rank) * TC_BM + 32 * q;  // rows of C
      const int y0 = partial ? (x.split * p.tail_tiles + x.ws_tile) * Cfg::TILE_M + int(rank) * TC_BM + 32 * q
                             : row0;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                             static_cast<uint32_t>(acc * BN);
      const int chunks = BN / cw;
      // On the CTA's last unit the operand ring is idle (every MMA of the unit
      // has completed, no load follows): each chunk gets a staging buffer of
      // its own there, so no store waits for an earlier one to have been read
      // (with one tile per CTA, two buffers per warp left the epilogue of a
      // 256x256 pair tile at ~5.6 us).
      const bool spread = u + ncta >= p.units;
      // One compiled copy of the chunk loop per epilogue variant (EpiVariant),
      // chosen once per tile.
      auto chunk_loop = [&](auto variant) {
      constexpr int V = decltype(variant)::value;
      for (int c = 0; c < chunks; ++c) {
        const uint32_t ring_buf = uint32_t(Cfg::OFF_A + (e * chunks + c) * Cfg::STG_BYTES);
        const uint32_t stg = spread ? base + ring_buf : stg0 + sbuf * Cfg::STG_BYTES;
        uint8_t* const stg_p = spread ? sbase + ring_buf : stg_p0 + sbuf * Cfg::STG_BYTES;
        const int x0 = n0 + c * cw;
        // A TMA store writes whole 16-byte pieces of a row, so columns past the
        // last 16-byte boundary inside C, [n_tma, N), are written by the threads.
        const bool tma_cols = partial || x0 < p.n_tma;
        const int tail_lo = max(x0, p.n_tma), tail_hi = min(x0 + cw, p.N);
        const int row = row0 + lane;
        const bool has_tail = !partial && tail_lo < tail_hi && row < p.M;
        if (lane == 0 && !spread) bulk_wait_read<1>();  // the store that last used this buffer has read it
        __syncwarp();
        if (V != EPI_PLAIN && c_tma && tma_cols) {
          if (lane == 0) {
            mbar_arrive_expect_tx(cload0 + 8 * e, Cfg::STG_BYTES);
            if (DG_TMA(p.dbg, x0, y0, esize, false)) tma_load_2d(stg, &tmC, cload0 + 8 * e, x0, y0);
          }
          __syncwarp();  // the load is issued before any lane of this warp waits for it
          if (!__all_sync(0xffffffffu, wait(cload0 + 8 * e, cphase, WAIT_EPI_C_LOAD))) {
            ok = false;
            break;
          }
          cphase ^= 1u;
        }
        __syncwarp();
        uint8_t* const row_p = stg_p + lane * 128;
        const int sw = lane & 7;  // 128-byte swizzle: 16-byte chunk j lives at j ^ (row % 8)
        if (V != EPI_PLAIN && c_tma && has_tail) {
          for (int col = tail_lo; col < tail_hi; ++col) {
            const int b = (col - x0) * esize;
            uint8_t* dst = row_p + ((((b >> 4) ^ sw)) << 4) + (b & 15);
            const uint8_t* src = static_cast<const uint8_t*>(p.c_ptr) + (int64_t(row) * p.ldc + col) * esize;
            if (!DG_IN(p.dbg, src, esize, DBG_EPI_LOAD)) continue;
            if (esize == 4)
              *reinterpret_cast<float*>(dst) = *reinterpret_cast<const float*>(src);
            else
              *reinterpret_cast<uint16_t*>(dst) = *reinterpret_cast<const uint16_t*>(src);
          }
        }
        if (esize == 4) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_row + c * 32, r);
          tmem_ld_wait(r);
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          if (!partial) epi32<V>(v, p, csrc, row_p, sw, 0, 4, row, x0);  // partials stay raw
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(row_p + ((j ^ sw) << 4)) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        } else {
          uint32_t r0[32], r1[32];
          tmem_ld_32x32b_x32(t_row + c * 64, r0);
          tmem_ld_32x32b_x32(t_row + c * 64 + 32, r1);
          tmem_ld_wait(r0);
          tmem_ld_wait(r1);
          float v0[32], v1[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v0[i] = __uint_as_float(r0[i]);
            v1[i] = __uint_as_float(r1[i]);
          }
          epi32<V>(v0, p, csrc, row_p, sw, 0, 2, row, x0);  // (16-bit output: never a partial unit)
          epi32<V>(v1, p, csrc, row_p, sw, 4, 2, row, x0 + 32);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float* h = j < 4 ? &v0[8 * (j & 3)] : &v1[8 * (j & 3)];
            *reinterpret_cast<uint4*>(row_p + ((j ^ sw) << 4)) =
                make_uint4(pack2(h[0], h[1], p.out_kind), pack2(h[2], h[3], p.out_kind),
                           pack2(h[4], h[5], p.out_kind), pack2(h[6], h[7], p.out_kind));
          }
        }
        if (has_tail) {
          for (int col = tail_lo; col < tail_hi; ++col) {
            const int b = (col - x0) * esize;
            const uint8_t* src = row_p + ((((b >> 4) ^ sw)) << 4) + (b & 15);
            uint8_t* dst = static_cast<uint8_t*>(p.c_ptr) + (int64_t(row) * p.ldc + col) * esize;
            if (!DG_IN(p.dbg, dst, esize, DBG_EPI_STORE)) continue;
            if (esize == 4)
              *reinterpret_cast<float*>(dst) = *reinterpret_cast<const float*>(src);
            else
              *reinterpret_cast<uint16_t*>(dst) = *reinterpret_cast<const uint16_t*>(src);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (tma_cols && DG_TMA(p.dbg, x0, y0, esize, true)) tma_store_2d(out_map, stg, x0, y0);
          bulk_commit();  // one group per chunk (possibly empty) keeps the buffer accounting exact
        }
        sbuf ^= 1;
      }
      };
      const int variant = partial ? int(EPI_PLAIN) : epi_variant(p, has_beta);
      if (variant == EPI_PLAIN)
        chunk_loop(std::integral_constant<int, EPI_PLAIN>{});
      else if (variant == EPI_BETA)
        chunk_loop(std::integral_constant<int, EPI_BETA>{});
      else
        chunk_loop(std::integral_constant<int, EPI_ALL>{});
      // This warp's reads of the accumulator are complete: release it (to the
      // leader, whose MMA warp waits for both CTAs of a pair).
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR)
          mbar_arrive_cluster(mapa_shared(tempty0 + 8 * acc, 0));
        else
          mbar_arrive(tempty0 + 8 * acc);
      }
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (ok && fused.ws_tile >= 0) {
      constexpr int CPU = PAIR ? 2 : 1;  // CTAs per unit
      // (the ring is idle: every MMA of this CTA's last unit has completed)
      fused_split_reduce<Cfg::TILE_M, BN>(p, fused.ws_tile, fused.split * CPU + int(rank), p.splitk * CPU,
                                          fused.m_blk, fused.n_blk, base + Cfg::OFF_A, xfree0, xfull0, w);
    }
    // The stores must have read the staging buffers before the CTA exits; the
    // grid's completion covers their writes to global memory.
    if (lane == 0) bulk_wait_read<0>();
  }

  // ------------------------------------------------------------- teardown
  // A cluster's CTAs stay until both are done: a pair leader's MMAs read the
  // peer's shared memory and write its tensor memory, so a pair synchronises
  // before it frees tensor memory.  A K pair's CTAs write partial sums into
  // each other's shared memory and arrive on each other's barriers: the
  // producer and MMA warps, done with the peer from the start, and the
  // epilogue warps, once their exchange is over, announce it; each CTA frees
  // its own tensor memory and waits for the peer's announcement only before
  // it exits.
  if constexpr (KPAIR) {
    if (warp < 2) cluster_arrive();
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
  if constexpr (KPAIR) cluster_wait();
}

template <int BN, int MODE, bool TF32 = false>
cudaError_t launch_gemm_tc_bn(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                              const CUtensorMap& ws, const TcParams& p, int grid, cudaStream_t s) {
  constexpr int smem = TcCfg<BN, MODE>::SMEM_BYTES;
  auto kern = gemm_tc_kernel<BN, MODE, TF32>;
  // The shared-memory limit is set once per device (bit d of `ready`), not on
  // every launch: it is host time in front of every call.
  static std::atomic<uint64_t> ready{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const uint64_t bit = dev < 64 ? uint64_t(1) << dev : 0;
  if (bit == 0 || (ready.load(std::memory_order_acquire) & bit) == 0) {
    const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    ready.fetch_or(bit, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (MODE != TC_SOLO) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 2;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (p.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, a, b, c, ws, p);
}

// Clusters of two that can be resident at once (the grid of a cluster kernel
// is twice this, at most).
template <int BN, int MODE>
int max_clusters() {
  constexpr int smem = TcCfg<BN, MODE>::SMEM_BYTES;
  auto kern = gemm_tc_kernel<BN, MODE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace dg
