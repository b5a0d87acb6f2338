// api.cpp -- the C ABI declared in include/gemm.h: argument checks, the
// tile-shape / split-K planner, tensor-map (TMA descriptor) encoding, the plan
// object and kernel dispatch.
#include "gemm.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "kernels.h"

namespace {

// A tensor-core call as far as planning and descriptors are concerned.
struct TcKey {
  int64_t M, N, K, lda, ldb, ldc;
  uintptr_t A, B, C;
  int32_t dtype, ta, tb, beta_nz;
  uintptr_t Cin;  // the C that beta scales (C itself unless gemm_run_ex got a separate one)
  int64_t ldcin;
  int32_t cin_kind;
  bool operator==(const TcKey& o) const {
    return M == o.M && N == o.N && K == o.K && lda == o.lda && ldb == o.ldb && ldc == o.ldc &&
           A == o.A && B == o.B && C == o.C && dtype == o.dtype && ta == o.ta && tb == o.tb &&
           beta_nz == o.beta_nz && Cin == o.Cin && ldcin == o.ldcin && cin_kind == o.cin_kind;
  }
};

struct TcKeyHash {
  size_t operator()(const TcKey& k) const {
    uint64_t h = 1469598103934665603ull;
    auto mix = [&](uint64_t v) { h = (h ^ v) * 1099511628211ull; };
    mix(uint64_t(k.M)); mix(uint64_t(k.N)); mix(uint64_t(k.K)); mix(uint64_t(k.lda));
    mix(uint64_t(k.ldb)); mix(uint64_t(k.ldc)); mix(k.A); mix(k.B); mix(k.C);
    mix(uint64_t(k.dtype) | (uint64_t(k.ta) << 8) | (uint64_t(k.tb) << 16) | (uint64_t(k.beta_nz) << 24) |
        (uint64_t(k.cin_kind) << 32));
    mix(k.Cin); mix(uint64_t(k.ldcin));
    return size_t(h);
  }
};

// One tensor-core plan: tile width, kernel variant, K slices, and whether
// only the tail wave's tiles are split.
struct TcChoice {
  int bn = 256, mode = dg::TC_SOLO, s = 1;
  bool tail = false;
  double t = 1e300;  // estimated seconds
};

// The C that beta scales: the output itself, or gemm_run_ex's separate C.
struct CinRef {
  const void* ptr;
  int64_t ld;
  int kind;  // dg::OutKind
};

// Planner decision, encoded tensor maps and kernel parameters of one call.
struct TcEntry {
  gemm_config_info_t info;
  CUtensorMap ma, mb, mc, mw;  // A, B, C, split-K partial workspace
  dg::TcParams p;
  size_t ws_bytes;
  void* ws_ptr;  // workspace the partial map was encoded for (split-K)
};

}  // namespace

struct gemm_plan {
  int device = 0;
  int sms = 0;
  int* err = nullptr;  // device word, OR of wait codes (and, debug build, failed-check sites)
  int64_t last_err_bits = 0;  // the word the last gemm_plan_poll_error read
  void* ws = nullptr;  // workspace (split-K partials, GEMV partials)
  size_t ws_bytes = 0;
  unsigned* counters = nullptr;  // GEMV per-panel arrival counters: zero between calls
  void* tws = nullptr;  // K-major copies of TF32 operands stored M/N-major
  size_t tws_bytes = 0;
  size_t counter_count = 0;
  uint64_t watchdog_ns = 2000000000ull;
  // Kernels launch as programmatic dependents of the stream's previous kernel
  // (their launch and prologue overlap its tail); GEMM_PDL=0 turns this off.
  bool pdl = true;
  gemm_config_info_t last{};
  // Repeated calls with the same shapes, pointers and flags skip planning and
  // descriptor encoding (host time that would otherwise sit in front of the
  // kernels on the stream).
  std::unordered_map<TcKey, TcEntry, TcKeyHash> tc_cache;
  // GEMM_LOG=1 (read at plan creation): one line per call on stderr.
  bool log = false;
  // GEMM_NVTX=1 (read at plan creation): every gemm_run / gemm_run_ex is an
  // NVTX range named after its shape and types, for profilers' timelines.
  bool nvtx = false;
  // Benchmark mode: the fastest measured choice per shape (key without pointers).
  bool autotune = false;
  std::unordered_map<TcKey, TcChoice, TcKeyHash> tuned;
};

namespace {

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

bool out_is_f32(gemm_dtype_t d) { return d == GEMM_BF16_F32 || d == GEMM_F16_F32 || d == GEMM_TF32_F32; }
bool in_is_f16(gemm_dtype_t d) { return d == GEMM_F16_F32 || d == GEMM_F16_F16; }
bool in_is_tf32(gemm_dtype_t d) { return d == GEMM_TF32_F32; }
int in_bytes(gemm_dtype_t d) { return in_is_tf32(d) ? 4 : 2; }

int out_kind(gemm_dtype_t d) {
  switch (d) {
    case GEMM_BF16_F32:
    case GEMM_F16_F32:
    case GEMM_TF32_F32: return dg::OUT_F32;
    case GEMM_BF16_BF16: return dg::OUT_BF16;
    default: return dg::OUT_F16;
  }
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------- validation

// Floor division for a positive divisor.
int64_t floor_div(int64_t a, int64_t b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// A row-major matrix as memory: `rows` rows of `width` bytes, `pitch` bytes
// apart, the first at byte address `base`.
struct Region {
  uint64_t base;
  int64_t rows, pitch, width;
};

Region region(const void* p, int64_t rows, int64_t cols, int64_t ld, int64_t esize) {
  return Region{uint64_t(reinterpret_cast<uintptr_t>(p)), rows, ld * esize, cols * esize};
}

// Byte ranges of a call's buffers for the debug build's device checks
// (kernels.h, DbgSpans).  The release build passes them to no kernel.
// GEMM_DEBUG_SHRINK=n (read by the debug build only, for its tests) makes the
// output's range n bytes shorter, so that the checks of the last output
// elements fail while every access stays inside the caller's buffer.
struct Spans {
  dg::DbgSpans s{};
  int n = 0;
  explicit Spans(int* err) { s.err = err; }
  Spans& bytes(const void* p, int64_t len) {
    if (p != nullptr && len > 0 && n < dg::kDbgSpans) {
      s.lo[n] = uint64_t(reinterpret_cast<uintptr_t>(p));
      s.hi[n] = s.lo[n] + uint64_t(len);
      ++n;
    }
    return *this;
  }
  // rows x cols elements of esize bytes, rows ld elements apart
  Spans& matrix(const void* p, int64_t rows, int64_t cols, int64_t ld, int64_t esize) {
    if (rows <= 0 || cols <= 0) return *this;
    return bytes(p, ((rows - 1) * ld + cols) * esize);
  }
  // count elements of esize bytes, inc elements apart
  Spans& vector(const void* p, int64_t count, int64_t inc, int64_t esize) {
    return count > 0 ? bytes(p, ((count - 1) * inc + 1) * esize) : *this;
  }
  // the output: its range less GEMM_DEBUG_SHRINK bytes
  Spans& out_matrix(const void* p, int64_t rows, int64_t cols, int64_t ld, int64_t esize) {
    const int at = n;
    matrix(p, rows, cols, ld, esize);
    return shrink(at);
  }
  Spans& out_vector(const void* p, int64_t count, int64_t inc, int64_t esize) {
    const int at = n;
    vector(p, count, inc, esize);
    return shrink(at);
  }
  Spans& shrink(int at) {
    static const int64_t cut = [] {
      const char* v = std::getenv("GEMM_DEBUG_SHRINK");
      return v ? std::max<int64_t>(0, std::atoll(v)) : int64_t(0);
    }();
    if (at < n) s.hi[at] -= std::min<uint64_t>(uint64_t(cut), s.hi[at] - s.lo[at]);
    return *this;
  }
};

// Do two matrices share a byte?  Row i of x and row k of y meet iff y's row
// starts before x's ends and ends after x's starts: -wy < d + k*Ly - i*Lx < wx
// with d = by - bx.  Exact in O(1) for equal pitches (row-interleaved slices
// of one parent, or a single row), where only t = k - i matters; with
// different pitches the rows of the shorter matrix are tested one by one, and
// past 2^20 such rows overlapping byte spans count as overlap.
bool overlaps(Region x, Region y) {
  if (x.rows <= 0 || y.rows <= 0 || x.width <= 0 || y.width <= 0) return false;
  const uint64_t xe = x.base + uint64_t(x.rows - 1) * uint64_t(x.pitch) + uint64_t(x.width);
  const uint64_t ye = y.base + uint64_t(y.rows - 1) * uint64_t(y.pitch) + uint64_t(y.width);
  if (xe <= y.base || ye <= x.base) return false;  // disjoint spans
  if (x.rows == 1) x.pitch = y.pitch;  // a single row fits any pitch
  if (y.rows == 1) y.pitch = x.pitch;
  if (x.pitch == y.pitch) {
    const int64_t L = x.pitch;
    const int64_t d = int64_t(y.base - x.base);  // the spans overlap: |d| < 2^63
    // integers t in the open interval ((-wy - d) / L, (wx - d) / L), and
    // t = k - i in [1 - rows_x, rows_y - 1] (each such t has a valid i, k)
    const int64_t lo = std::max<int64_t>(floor_div(-y.width - d, L) + 1, 1 - x.rows);
    const int64_t hi = std::min<int64_t>(-floor_div(d - x.width, L) - 1, y.rows - 1);
    return lo <= hi;
  }
  if (x.rows > y.rows) std::swap(x, y);
  if (x.rows > (int64_t(1) << 20)) return true;
  const int64_t d = int64_t(y.base - x.base);
  for (int64_t i = 0; i < x.rows; ++i) {
    // row i of x covers [s, s + wx) relative to y.base; rows k of y with
    // k*Ly < s + wx and k*Ly + wy > s
    const int64_t s = int64_t(i) * x.pitch - d;
    const int64_t k_lo = std::max<int64_t>(floor_div(s - y.width, y.pitch) + 1, 0);
    const int64_t k_hi = std::min<int64_t>(floor_div(s + x.width - 1, y.pitch), y.rows - 1);
    if (k_lo <= k_hi) return true;
  }
  return false;
}

gemm_status_t check(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                    int64_t ldb, const void* C, int64_t ldc, float alpha, gemm_dtype_t dtype,
                    gemm_op_t ta, gemm_op_t tb, gemm_epilogue_t epi) {
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (dtype < GEMM_BF16_F32 || dtype > GEMM_TF32_F32) return GEMM_ERR_INVALID_ARG;
  if ((ta != GEMM_OP_N && ta != GEMM_OP_T) || (tb != GEMM_OP_N && tb != GEMM_OP_T))
    return GEMM_ERR_INVALID_ARG;
  if (epi.act < GEMM_ACT_NONE || epi.act > GEMM_ACT_SILU) return GEMM_ERR_INVALID_ARG;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_UNSUPPORTED;
  const int64_t a_cols = ta == GEMM_OP_N ? K : M;
  const int64_t b_cols = tb == GEMM_OP_N ? N : K;
  if (lda < std::max<int64_t>(1, a_cols) || ldb < std::max<int64_t>(1, b_cols) ||
      ldc < std::max<int64_t>(1, N))
    return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  if (C == nullptr) return GEMM_ERR_INVALID_ARG;
  const bool reads_ab = K > 0 && alpha != 0.f;
  if (reads_ab && (A == nullptr || B == nullptr)) return GEMM_ERR_INVALID_ARG;
  const size_t ces = out_is_f32(dtype) ? 4 : 2;
  const int ies = in_bytes(dtype);
  if (reads_ab) {  // C is written while A and B are read: they must not share a byte
    const Region rc = region(C, M, N, ldc, int64_t(ces));
    const Region ra = ta == GEMM_OP_N ? region(A, M, K, lda, ies) : region(A, K, M, lda, ies);
    const Region rb = tb == GEMM_OP_N ? region(B, K, N, ldb, ies) : region(B, N, K, ldb, ies);
    if (overlaps(rc, ra) || overlaps(rc, rb)) return GEMM_ERR_INVALID_ARG;
  }
  if (!aligned(C, ces)) return GEMM_ERR_ALIGNMENT;
  if (reads_ab && (!aligned(A, ies) || !aligned(B, ies))) return GEMM_ERR_ALIGNMENT;
  if (in_is_tf32(dtype)) {  // always the tensor-core path
    if (reads_ab && (!aligned(A, 16) || !aligned(B, 16) || (lda * 4) % 16 || (ldb * 4) % 16))
      return GEMM_ERR_ALIGNMENT;
    if (N >= 4 && (!aligned(C, 16) || (ldc * 4) % 16)) return GEMM_ERR_ALIGNMENT;
    return GEMM_OK;
  }
  if (reads_ab && M >= 2 && N >= 2) {
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16)) return GEMM_ERR_ALIGNMENT;
    if ((lda * 2) % 16 || (ldb * 2) % 16 || (ldc * int64_t(ces)) % 16) return GEMM_ERR_ALIGNMENT;
  }
  return GEMM_OK;
}

// --------------------------------------------------------------- planner

void quantization(int64_t M, int64_t N, int tm, int tn, int splitk, int sms, int ctas_per_sm,
                  gemm_config_info_t* o) {
  o->tile_m = tm;
  o->tile_n = tn;
  o->splitk = splitk;
  o->sms = sms;
  o->tiles = ceil_div(M, tm) * ceil_div(N, tn);
  o->units = o->tiles * splitk;
  const int64_t wave = int64_t(sms) * ctas_per_sm;
  o->waves = double(o->units) / double(wave);
  const int64_t tail = o->units % wave;
  o->tail_fraction = double(tail) / double(wave);
  o->useful_fraction = o->tiles ? double(M) * double(N) / (double(o->tiles) * tm * tn) : 0.0;
}

// Cost model of the tensor-core path (seconds), calibrated on GB300 against
// measured times of every tile shape (128 x {64,128,256} on one CTA, 256 x 256
// on a CTA pair, the 128 x 128 K pair), K split and tail split for 204
// shapes: skinny M x {64,128,256} x {4096,8192} (M = 1024 ... 32768), the
// 2304 x N x 4096 and 27648 x N x 4096 sweeps and 14 cubes and long-K
// shapes.  Persistent CTAs take units round-robin, so the busiest SM runs
// ceil(units/SMs) units ("Matrix Multiplication Background User's Guide",
// section 3.2, wave quantization); every unit pays for a full tile whatever
// part of it lies inside C (section 3.1, tile quantization).
//
// A unit walks its k-blocks through a ring of `stages` shared-memory stages.
// A stage is refilled only after the MMAs that read it have finished, and
// its next block then arrives after the memory latency, so one k-block costs
// max(MMA time, (latency + MMA time) / stages): a latency-bound ring when the
// MMAs are short (skinny shapes), the tensor pipe when they are long.  The MMA
// rate of one SM is its own peak while few SMs run, and the GPU's sustained
// rate (power-limited) shared by the active SMs when many do.  The call is
// also bound by streaming its unique bytes from DRAM at ~80 GB/s per distinct
// A or B panel in flight, up to the copy bandwidth.  Split-K adds its partials
// (written, then read by the reduction launch) and that launch, whose threads
// load eight slices at a time, so every further eight slices add a round of
// memory latency.
struct Model {
  double peak_flops = 2.0e15;   // dense bf16 rate with every SM busy (power-limited)
  double peak_sm = 1.5e13;      // dense bf16 rate of one SM when the power limit does not bind
  double latency = 2.1e-6;      // from a stage's release to its next block's arrival, under load
  double stream_bw = 6.8e12;    // B/s DRAM rate reachable by TMA box streams (copy bandwidth)
  double panel_bw = 8.0e10;     // B/s of one streamed panel
  double part_bw = 4.5e12;      // B/s at which split-K partials are written and read back
  double fixed = 6.0e-6;        // launch, pipeline fill and last epilogue
  double wave = 3.0e-6;         // each further wave of units (refill after an epilogue)
  double reduce = 7.0e-6;       // split-K reduction launch and tail
  double reduce_round = 1.0e-6; // each further 8 K slices: the reduction's next round of dependent loads
  double fused = 4.5e-6;        // split-K reduced in the GEMM kernel (opt-in): arrival wait and tail
  double l2_bw = 1.0e13;        // B/s of the partials' round trip through L2 in that case
};

// GEMM_FUSED_REDUCE=1 sums K slices that all run at once inside the GEMM
// kernel instead of in the tile reduction kernel.  Measured on GB300 over the
// 2304 x N x 4096 and 27648 x N x 4096 sweeps and 256 x 256 x 65536, the two
// are within a few microseconds of each other (the reduction kernel, launched
// as a programmatic dependent, already overlaps the GEMM's tail) and the
// reduction kernel is ahead on most shapes, so it is the default.
bool fused_enabled() {
  const char* v = std::getenv("GEMM_FUSED_REDUCE");
  return v && *v && std::atoi(v) != 0;
}

double tile_efficiency(int bn) { return bn >= 128 ? 1.0 : 0.5; }

// Extra fixed cost of a CTA-pair (cluster) launch, fitted on GB300.
constexpr double kPairFixed = 6.0e-6;
// Cost of a K pair's on-chip exchange per 64-column round (bn/128 rounds):
// 32 KB of fp32 partials each way between two SMs (distributed shared memory
// moves ~15-27 GB/s per SM each way); fitted on GB300 to the K pair against
// one-CTA tiles at 256^3 ... 2048^3 and 8192 x 128 x 8192.
constexpr double kKPairRound = 1.2e-6;

// Distinct A row-panels and B column-panels among the first `count` units of
// the kernel's unit order (gemm_tc.cuh: decode_unit): slice-major, then groups
// of `group` tile rows walked column by column.
void distinct_panels(int64_t mb, int64_t nb, int64_t group, int64_t count, int64_t* da, int64_t* db) {
  const int64_t tiles = mb * nb;
  const int64_t full_slices = count / tiles, r = count % tiles;
  *da = full_slices * mb;
  *db = full_slices * nb;
  if (r == 0) return;
  const int64_t per = group * nb;
  const int64_t full_groups = r / per, rem = r % per;
  int64_t dm = std::min(full_groups * group, mb);
  int64_t dn = full_groups > 0 ? nb : 0;
  if (rem > 0) {
    const int64_t rows = std::min(mb - full_groups * group, group);
    dm += std::min(rows, rem);
    dn = std::max(dn, ceil_div(rem, rows));
  }
  *da += dm;
  *db += dn;
}

// One k-block of one unit: the MMAs of a 128 x bn tile (a pair's SM does the
// flops of 128 x bn as well) at the rate one SM gets while `active_sms` SMs
// run, or, when the ring waits on memory, the latency plus those MMAs spread
// over the ring's stages.
double kblock_time(int bn, int mode, int eb, int64_t active_sms, const Model& md) {
  const double scale = eb == 4 ? 0.5 : 1.0;  // TF32 runs at half the 16-bit rate
  const double rate = std::min(md.peak_sm * scale, md.peak_flops * scale / double(std::max<int64_t>(1, active_sms)));
  const double t_mma = 2.0 * dg::TC_BM * bn * double(128 / eb) / (rate * tile_efficiency(bn));
  const int stages = std::max(1, dg::tc_stages(bn, mode));
  return std::max(t_mma, (md.latency + t_mma) / stages);
}

// eb: operand element bytes (2: bf16/fp16, 4: TF32, whose tensor-core rate is
// half of the 16-bit one); a k-block is one 128-byte row of every operand.
double estimate(int64_t M, int64_t N, int64_t K, int bn, int mode, int splitk, int sms, int c_es,
                bool beta, int raster_group, const Model& md, int* splitk_eff, int eb) {
  const bool pair = mode == dg::TC_PAIR, kpair = mode == dg::TC_KPAIR;
  const int kbe = 128 / eb;
  const int64_t kb = ceil_div(K, kbe);
  const int64_t kbps = ceil_div(kb, splitk);
  const int s_eff = int(ceil_div(kb, kbps));
  *splitk_eff = s_eff;
  // A pair unit (256 x bn) runs on two SMs; each SM stages 128 rows of A and
  // bn/2 columns of B per k-block and does the flops of a 128 x bn tile.  A
  // K-pair tile is two CTA units (its K halves) that run side by side.
  const int tile_m = pair ? 2 * dg::TC_BM : dg::TC_BM;
  const int slots = pair ? sms / 2 : sms;
  const int64_t mb = ceil_div(M, tile_m), nb = ceil_div(N, bn);
  const int64_t group = std::max<int64_t>(1, std::min<int64_t>(raster_group, mb));
  const int64_t units = mb * nb * s_eff;
  const int64_t active = std::min<int64_t>(units, slots);
  const double waves = double(ceil_div(units, slots));
  // distinct A and B panels the first wave streams
  int64_t da = 0, db = 0;
  if (kpair) {
    distinct_panels(mb, nb, group, active / 2, &da, &db);
    da *= 2;  // both K halves of each panel stream at once
    db *= 2;
  } else {
    distinct_panels(mb, nb, group, active, &da, &db);
  }
  int64_t streams = da + db;
  const int64_t active_sms = pair ? 2 * active : active;
  const double makespan = waves * double(kbps) * kblock_time(bn, mode, eb, active_sms, md) + md.fixed +
                          (waves - 1.0) * md.wave + (pair ? kPairFixed : 0.0) +
                          (kpair ? kKPairRound * (bn / 128) * waves : 0.0);
  const double unique = double(M * K + K * N) * eb;
  double bytes = unique + double(M) * N * c_es * (beta ? 2.0 : 1.0);
  double t = 0.0;
  if (s_eff > 1 && !kpair) {
    const double part = double(s_eff) * double(mb * tile_m) * double(N) * 4.0;
    if (units <= slots && fused_enabled()) {  // reduced in the kernel, the partials stay in L2
      t += md.fused + 2.0 * part / md.l2_bw;
    } else {
      bytes += part;                          // partials written, read back by the reduction kernel
      t += md.reduce + double(ceil_div(s_eff, 8)) * md.reduce_round + part / md.part_bw;
    }
  }
  if (pair) streams *= 2;  // each CTA of a pair streams its own half of A and of B
  const double t_mem = bytes / std::min(md.stream_bw, md.panel_bw * double(streams));
  return std::max(makespan, t_mem) + t;
}

// Extra cost of a tail split's reduction over the model's split-K reduction
// (fitted on GB300 with the rest of the model, tail split on and off).
constexpr double kTailExtra = 0.0;

// Whole tiles for the W = tiles / slots full waves, then the T remaining
// tiles in S K slices each (one more wave, T*S <= slots), whose partials a
// reduction launch sums.  Same ingredients as estimate().
double estimate_tail(int64_t M, int64_t N, int64_t K, int bn, int mode, int S, int sms, int c_es,
                     bool beta, int raster_group, const Model& md, int eb) {
  const bool pair = mode == dg::TC_PAIR;
  const int tile_m = pair ? 2 * dg::TC_BM : dg::TC_BM;
  const int slots = pair ? sms / 2 : sms;
  const int64_t mb = ceil_div(M, tile_m), nb = ceil_div(N, bn), tiles = mb * nb;
  const int64_t W = tiles / slots, T = tiles - W * slots;
  const int kbe = 128 / eb;
  const int64_t kb = ceil_div(K, kbe), kbps = ceil_div(kb, S);
  const int64_t group = std::max<int64_t>(1, std::min<int64_t>(raster_group, mb));
  int64_t da = 0, db = 0;
  distinct_panels(mb, nb, group, std::min<int64_t>(tiles, slots), &da, &db);
  const int64_t streams = (da + db) * (pair ? 2 : 1);
  // every SM is busy in the full waves; the tail wave's slices fill the GPU as well
  const double tk = kblock_time(bn, mode, eb, sms, md);
  const double makespan = double(W) * (double(kb) * tk + md.wave) + double(kbps) * tk + md.fixed +
                          (pair ? kPairFixed : 0.0);
  const double unique = double(M * K + K * N) * eb;
  const double part = double(S) * double(T) * tile_m * bn * 4.0;
  const bool fused = fused_enabled();  // the tail's slices are one per CTA: reduced in the kernel
  const double bytes = unique + double(M) * N * c_es * (beta ? 2.0 : 1.0) + (fused ? 0.0 : part);
  const double t_mem = bytes / std::min(md.stream_bw, md.panel_bw * double(streams));
  if (fused) return std::max(makespan, t_mem) + md.fused + 2.0 * part / md.l2_bw;
  return std::max(makespan, t_mem) + md.reduce + double(ceil_div(S, 8)) * md.reduce_round + kTailExtra +
         part / md.part_bw;
}

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  return std::atoi(v);
}

// Every candidate the planner estimates, in the order it considers them
// (best estimate first after sorting); `best` is the planner's pick.
void tc_candidates(int64_t M, int64_t N, int64_t K, int sms, int c_es, bool beta, TcChoice* best,
                   std::vector<TcChoice>* all, int eb) {
  const Model md;
  TcChoice pick;
  int force_bn = 0;
  bool force_pair = false;
  if (const char* f = std::getenv("GEMM_FORCE_TILE")) {
    int fm = 0, fn = 0;
    if (std::sscanf(f, "%dx%d", &fm, &fn) == 2 && (fn == 64 || fn == 128 || fn == 256)) {
      if (fm == dg::TC_BM) force_bn = fn;
      if (fm == 2 * dg::TC_BM && fn >= 128) {  // 256-row tile on a CTA pair
        force_bn = fn;
        force_pair = true;
      }
    }
  }
  const int force_s = env_int("GEMM_FORCE_SPLITK", 0);
  // GEMM_SPLITK_CLUSTER: 0 never reduces K halves on chip, 1 only does (where
  // a two-slice split on a K pair exists), unset lets the model choose.
  const int kpair_env = env_int("GEMM_SPLITK_CLUSTER", -1);
  // GEMM_TAIL_SPLIT: 0 never splits only the tail wave; 1 only does (where a
  // partly filled last wave exists), with the slices the planner picks; S >= 2
  // only does, with S slices; unset lets the model choose.
  const int tail_env = env_int("GEMM_TAIL_SPLIT", -1);
  const bool only_tail = tail_env >= 1;
  const int raster = env_int("GEMM_RASTER_GROUP", 16);
  const int64_t kb = ceil_div(K, 128 / eb);
  // GEMM_PLAN_DEBUG=1 prints every candidate's estimate to stderr.
  const bool debug = env_int("GEMM_PLAN_DEBUG", 0) != 0;
  // candidates: 128-row tiles of width 256/128/64 on one CTA, 256 x 256 on a
  // CTA pair, 128 x 128 with K halves on a K pair.  The 128 x 256 K pair
  // (two exchange rounds, and a third of each ring stage for A instead of
  // half) measured no faster than the 256 x 256 CTA pair on any shape: it
  // runs only when that tile is forced.
  struct Cand { int bn; int mode; };
  const Cand cands[6] = {{256, dg::TC_PAIR}, {256, dg::TC_SOLO}, {128, dg::TC_SOLO}, {64, dg::TC_SOLO},
                         {256, dg::TC_KPAIR}, {128, dg::TC_KPAIR}};
  auto take = [&](double t, int bn, int mode, int s, bool tail) {
    if (debug)
      std::fprintf(stderr, "gemm plan %lldx%lldx%lld: bn %d mode %d split %d tail %d -> %.2f us\n",
                   (long long)M, (long long)N, (long long)K, bn, mode, s, int(tail), t * 1e6);
    TcChoice c;
    c.bn = bn;
    c.mode = mode;
    c.s = s;
    c.tail = tail;
    c.t = t;
    if (all) all->push_back(c);
    // prefer earlier candidates / fewer slices unless clearly faster (2%)
    if (t < pick.t * 0.98) pick = c;
  };
  for (const Cand& c : cands) {
    const bool kpair = c.mode == dg::TC_KPAIR;
    if (force_bn && (c.bn != force_bn || (c.mode == dg::TC_PAIR) != force_pair)) continue;
    if (kpair ? kpair_env == 0 : kpair_env == 1) continue;
    if (kpair && (only_tail || (c.bn == 256 && force_bn != 256))) continue;
    // A K pair pays its exchange on every tile.  Where its tiles take more
    // than one wave of clusters it measured faster only when the best other
    // choice needs more than one wave as well (27648 x 128 x 4096: 45.7
    // against 53.9 us); against a one-wave choice it lost by up to 32%.
    if (kpair && kpair_env != 1 && ceil_div(M, dg::TC_BM) * ceil_div(N, c.bn) > sms / 2) {
      bool pick_multi_wave = pick.tail || pick.t >= 1e300;  // (or nothing else was possible)
      if (!pick_multi_wave) {
        const int p_tm = pick.mode == dg::TC_PAIR ? 2 * dg::TC_BM : dg::TC_BM;
        const int p_slots = pick.mode == dg::TC_PAIR ? sms / 2 : sms;
        pick_multi_wave = ceil_div(M, p_tm) * ceil_div(N, pick.bn) * pick.s > p_slots;
      }
      if (!pick_multi_wave) continue;
    }
    const int tile_m = c.mode == dg::TC_PAIR ? 2 * dg::TC_BM : dg::TC_BM;
    const int slots = c.mode == dg::TC_PAIR ? sms / 2 : sms;
    if (c.mode != dg::TC_SOLO && sms < 2) continue;
    const int64_t tiles = ceil_div(M, tile_m) * ceil_div(N, c.bn);
    for (int s = kpair ? 2 : 1; s <= (kpair ? 2 : 64) && !only_tail; ++s) {
      if (force_s > 0 && s != force_s) continue;
      if (s > kb) break;
      if (s > 1 && tiles * s > 4 * int64_t(slots)) break;
      int s_eff = 1;
      const double t = estimate(M, N, K, c.bn, c.mode, s, sms, c_es, beta, raster, md, &s_eff, eb);
      if (s_eff != s) continue;
      take(t, c.bn, c.mode, s, false);
    }
    // Tail split: whole tiles for the full waves, the last wave's tiles in
    // K slices that fill one more wave ("Matrix Multiplication Background
    // User's Guide", section 3.2: the tail wave is what a tile choice alone
    // cannot fill).
    if (!kpair && tail_env != 0 && (force_s <= 0 || only_tail)) {
      const int64_t W = tiles / slots, T = tiles - W * slots;
      if (W >= 1 && T > 0) {
        // slices: as many as fill the wave at most, fewer when the partials'
        // traffic and reduction cost more than the shorter slices save
        static const int kTry[] = {2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64};
        for (int st0 : kTry) {
          if (tail_env >= 2 && st0 != 2) break;
          int64_t st = tail_env >= 2 ? tail_env : st0;
          if (tail_env < 2 && st * T > slots) break;
          st = std::min<int64_t>(st, kb);
          if (st >= 2) st = ceil_div(kb, ceil_div(kb, st));  // no empty slice
          if (st < 2) break;
          const double t = estimate_tail(M, N, K, c.bn, c.mode, int(st), sms, c_es, beta, raster, md, eb);
          take(t, c.bn, c.mode, int(st), true);
        }
      }
    }
  }
  if (pick.t == 1e300) {  // forced choices not reachable exactly: take the nearest valid
    pick.s = force_s > 0 ? int(std::min<int64_t>(force_s, kb)) : 1;
    pick.bn = force_bn ? force_bn : 256;
    pick.mode = force_pair ? dg::TC_PAIR : dg::TC_SOLO;
    pick.tail = false;
  }
  *best = pick;
}

// Can a call's K slices be summed inside the GEMM kernel?  Every partial unit
// must be the last unit of its CTA (or cluster) -- the last `ncta` units are --
// and one share of every slice, plus the share's results in a 16-bit type,
// must fit the CTA's idle operand ring.
bool fused_fits(const gemm_config_info_t& info, int mode, int grid) {
  if (info.tail_tiles <= 0 || mode == dg::TC_KPAIR || !fused_enabled()) return false;
  const int cpu = mode == dg::TC_PAIR ? 2 : 1;
  const int64_t ncta = grid / cpu;
  if (int64_t(info.tail_tiles) * info.splitk > ncta) return false;
  const int64_t parts = int64_t(info.splitk) * cpu;
  const int64_t f = int64_t(info.tile_m) * info.tile_n / 4;
  const int64_t share = (f + parts - 1) / parts;
  return int64_t(info.splitk) * share * 16 + share * 8 + 32 <= dg::tc_ring_bytes(info.tile_n, mode);
}

// The configuration record of one choice.
void fill_info(int64_t M, int64_t N, int64_t K, int sms, const TcChoice& c, gemm_config_info_t* out,
               int eb) {
  const int64_t kb = ceil_div(K, 128 / eb);
  const int best_s = int(ceil_div(kb, ceil_div(kb, c.s)));
  const bool pair = c.mode == dg::TC_PAIR, kpair = c.mode == dg::TC_KPAIR;
  const int tile_m = pair ? 2 * dg::TC_BM : dg::TC_BM;
  const int pairs = sms / 2;
  const int slots = pair ? pairs : sms;
  std::memset(out, 0, sizeof(*out));
  quantization(M, N, tile_m, c.bn, best_s, slots, 1, out);
  out->sms = sms;
  if (kpair) {
    out->path = GEMM_PATH_TC_SPLITK_CLUSTER;
  } else if (c.tail && out->tiles % slots != 0) {
    out->path = GEMM_PATH_TC_TAIL_SPLIT;
    out->tail_tiles = int32_t(out->tiles % slots);
    out->units = (out->tiles - out->tail_tiles) + int64_t(out->tail_tiles) * best_s;
    out->waves = double(out->units) / double(slots);
    out->tail_fraction = double(out->units % slots) / double(slots);
  } else if (best_s > 1) {
    out->path = GEMM_PATH_TC_SPLITK;
    out->tail_tiles = int32_t(out->tiles);
  } else {
    out->path = GEMM_PATH_TC;
  }
  out->tile_k = 128 / eb;
  out->cta_per_tile = c.mode == dg::TC_SOLO ? 1 : 2;
  out->stages = dg::tc_stages(c.bn, c.mode);
  const int64_t mblocks = ceil_div(M, tile_m);
  out->raster_group = int(std::max<int64_t>(1, std::min<int64_t>(env_int("GEMM_RASTER_GROUP", 16), mblocks)));
  if (pair)
    out->grid = int(2 * std::min<int64_t>(out->units, pairs));
  else if (kpair)
    out->grid = int(2 * std::min<int64_t>(out->tiles, pairs));
  else
    out->grid = int(std::min<int64_t>(out->units, sms));
  out->workspace_bytes = int64_t(out->tail_tiles) * best_s * tile_m * c.bn * 4;
  out->launches = out->tail_tiles > 0 && !fused_fits(*out, c.mode, out->grid) ? 2 : 1;
}

void choose_tc(int64_t M, int64_t N, int64_t K, int sms, int c_es, bool beta, gemm_config_info_t* out,
               int eb) {
  TcChoice best;
  tc_candidates(M, N, K, sms, c_es, beta, &best, nullptr, eb);
  fill_info(M, N, K, sms, best, out, eb);
}

// ------------------------------------------------------------ tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D row-major tensor: `inner` contiguous elements per row, `outer` rows,
// `ld` elements between rows; boxes of box_inner x box_outer with 128-byte
// swizzling (box_inner * esize == 128).  Out-of-range reads give zero.
bool make_map(CUtensorMap* m, CUtensorMapDataType t, int esize, const void* ptr, int64_t inner,
              int64_t outer, int64_t ld, int box_inner, int box_outer,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
  cuuint64_t strides[1] = {cuuint64_t(ld) * cuuint64_t(esize)};
  cuuint32_t box[2] = {cuuint32_t(box_inner), cuuint32_t(box_outer)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, t, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// TF32 operands stored M/N-major: read by the MMAs where they are (tiles
// swizzled in 32-byte units), or first copied K-major into plan workspace?
// Measured on GB300 (8192^3 ... 512^3, skinny and GEMV-like shapes, L2
// flushed): in place, the MMAs of a call run ~10% longer with one such
// operand and ~44% longer with both; a copy reads and writes the operand at
// the copy bandwidth plus ~3 us of launch.  Each choice (copy none, the
// smaller, or both) is estimated and the cheapest taken: copies pay off only
// for large, compute-bound calls (8192^3 and 4096^3 with both operands
// M/N-major).  GEMM_TF32_TRANSPOSE=1 (read at every call) copies every
// M/N-major operand, =0 none.
void tf32_copies(int64_t M, int64_t N, int64_t K, gemm_op_t ta, gemm_op_t tb, bool* copy_a, bool* copy_b) {
  const bool a_mn = ta == GEMM_OP_T, b_mn = tb == GEMM_OP_N;
  *copy_a = *copy_b = false;
  const int force = env_int("GEMM_TF32_TRANSPOSE", -1);
  if (force >= 0) {
    *copy_a = a_mn && force != 0;
    *copy_b = b_mn && force != 0;
    return;
  }
  const double t_mma = 2.0 * double(M) * double(N) * double(K) / 1.0e15;  // TF32 at ~1 PFLOP/s
  const double copy_a_t = 2.0 * double(M) * double(K) * 4.0 / 6.8e12 + 3e-6;
  const double copy_b_t = 2.0 * double(N) * double(K) * 4.0 / 6.8e12 + 3e-6;
  auto penalty = [&](bool a_in_place, bool b_in_place) {
    const int n = int(a_in_place) + int(b_in_place);
    return t_mma * (n == 2 ? 0.44 : n == 1 ? 0.10 : 0.0);
  };
  double best = penalty(a_mn, b_mn);
  for (int c = 1; c < 4; ++c) {  // bit 0: copy A, bit 1: copy B
    const bool ca = (c & 1) != 0, cb = (c & 2) != 0;
    if ((ca && !a_mn) || (cb && !b_mn)) continue;
    const double t = penalty(a_mn && !ca, b_mn && !cb) + (ca ? copy_a_t : 0.0) + (cb ? copy_b_t : 0.0);
    if (t < best) {
      best = t;
      *copy_a = ca;
      *copy_b = cb;
    }
  }
}

// tcgen05 instruction descriptor, kind::f16 with fp32 accumulation:
// bits 4-5 D type (1 = f32), 7-9 A type and 10-12 B type (0 = f16, 1 = bf16),
// 15/16 A/B major (0 = K-major, 1 = M/N-major), 17-22 N>>3, 24-28 M>>4.
// kind::tf32 takes the same descriptor with A and B type 2 (TF32).
uint32_t make_idesc(int in_type, bool a_mn, bool b_mn, int n, int m) {
  const uint32_t ab = uint32_t(in_type);  // 0 fp16, 1 bf16, 2 TF32
  return (1u << 4) | (ab << 7) | (ab << 10) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
         (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

// ------------------------------------------------------------- workspace

// Grow a plan buffer to at least `bytes` (1 MiB steps, stream-ordered,
// zero-filled).
gemm_status_t ensure_buffer(void** buf, size_t* have, size_t bytes, cudaStream_t s) {
  if (bytes <= *have) return GEMM_OK;
  size_t nb = std::max<size_t>(bytes, size_t(1) << 20);
  nb = (nb + (size_t(1) << 20) - 1) & ~((size_t(1) << 20) - 1);
  if (*buf) cudaFreeAsync(*buf, s);
  *buf = nullptr;
  *have = 0;
  if (cudaMallocAsync(buf, nb, s) != cudaSuccess) {
    cudaGetLastError();
    *buf = nullptr;
    return GEMM_ERR_OUT_OF_MEMORY;
  }
  if (cudaMemsetAsync(*buf, 0, nb, s) != cudaSuccess) return GEMM_ERR_CUDA;
  *have = nb;
  return GEMM_OK;
}

gemm_status_t ensure_ws(gemm_plan* plan, size_t bytes, cudaStream_t s) {
  return ensure_buffer(&plan->ws, &plan->ws_bytes, bytes, s);
}

// The counters are zeroed once when allocated; every kernel that uses one
// leaves it at zero again.
gemm_status_t ensure_counters(gemm_plan* plan, size_t count, cudaStream_t s) {
  if (count <= plan->counter_count) return GEMM_OK;
  size_t nc = std::max<size_t>(count, 4096);
  if (plan->counters) cudaFreeAsync(plan->counters, s);
  plan->counters = nullptr;
  plan->counter_count = 0;
  if (cudaMallocAsync(reinterpret_cast<void**>(&plan->counters), nc * sizeof(unsigned), s) != cudaSuccess) {
    cudaGetLastError();
    plan->counters = nullptr;
    return GEMM_ERR_OUT_OF_MEMORY;
  }
  if (cudaMemsetAsync(plan->counters, 0, nc * sizeof(unsigned), s) != cudaSuccess) return GEMM_ERR_CUDA;
  plan->counter_count = nc;
  return GEMM_OK;
}

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// --------------------------------------------------------------- dispatch

gemm_status_t run_gemv(gemm_plan* plan, int64_t M, int64_t N, int64_t K, const void* A,
                       int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                       gemm_dtype_t dtype, gemm_op_t ta, gemm_op_t tb, const dg::EpiParams& e,
                       const CinRef& cin, cudaStream_t s, gemm_config_info_t* info) {
  dg::GemvArgs g{};
  g.K = int(K);
  g.in_f16 = in_is_f16(dtype);
  g.out = C;
  g.cin = cin.ptr;
  g.inc_cin = N == 1 ? cin.ld : 1;  // output r is C(r, 0) (N == 1) or C(0, r) (M == 1)
  g.e = e;
  g.pdl = plan->pdl;
  bool row_major_w;  // true: W rows run along K (rowdot); false: W rows run along R (colstream)
  if (N == 1) {      // C(i,0) = sum_k op(A)(i,k) op(B)(k,0)
    g.R = int(M);
    g.inc_out = ldc;
    g.x = B;
    g.incx = tb == GEMM_OP_N ? ldb : 1;
    g.W = A;
    g.ldw = lda;
    row_major_w = ta == GEMM_OP_N;
    g.w_rs = row_major_w ? lda : 1;
    g.w_cs = row_major_w ? 1 : lda;
  } else {           // M == 1: C(0,j) = sum_k op(A)(0,k) op(B)(k,j)
    g.R = int(N);
    g.inc_out = 1;
    g.x = A;
    g.incx = ta == GEMM_OP_N ? 1 : lda;
    g.W = B;
    g.ldw = ldb;
    row_major_w = tb == GEMM_OP_T;
    g.w_rs = row_major_w ? ldb : 1;
    g.w_cs = row_major_w ? 1 : ldb;
  }
  const bool vec_ok = aligned(g.W, 16) && (g.ldw * 2) % 16 == 0;
  // (debug build) the output, beta's C, the matrix and the vector; the plan's
  // workspace and counters once they exist
  auto set_spans = [&]() {
#ifdef DG_DEBUG
    Spans sp(plan->err);
    sp.out_vector(C, g.R, g.inc_out, e.out_kind == dg::OUT_F32 ? 4 : 2);
    if (e.beta != 0.f) sp.vector(g.cin, g.R, g.inc_cin, e.cin_kind == dg::OUT_F32 ? 4 : 2);
    sp.matrix(g.W, row_major_w ? g.R : K, row_major_w ? K : g.R, g.ldw, 2);
    sp.vector(g.x, K, g.incx, 2);
    sp.bytes(plan->ws, int64_t(plan->ws_bytes)).bytes(plan->counters, int64_t(plan->counter_count) * 4);
    g.dbg = sp.s;
#endif
  };
  cudaError_t err;
  info->path = GEMM_PATH_GEMV_GENERIC;
  info->splitk = 1;
  info->launches = 1;
  if (row_major_w && (vec_ok || g.R == 1) && aligned(g.W, 16) && K <= dg::gemv_rowdot_max_k()) {
    info->path = GEMM_PATH_GEMV_ROWDOT;
    set_spans();
    err = dg::launch_gemv_rowdot(g, s, plan->sms, &info->grid);
  } else if (!row_major_w && (vec_ok || K == 1) && aligned(g.W, 16)) {
    const dg::ColstreamPlan cp = dg::plan_gemv_colstream(g.R, g.K, plan->sms);
    if (cp.ws_bytes > 0) {
      gemm_status_t st = ensure_ws(plan, size_t(cp.ws_bytes), s);
      if (st == GEMM_OK) st = ensure_counters(plan, size_t(cp.panels), s);
      if (st != GEMM_OK) return st;
    }
    info->path = GEMM_PATH_GEMV_COLSTREAM;
    info->splitk = cp.ksplit;
    info->grid = cp.panels * cp.ksplit;
    info->workspace_bytes = cp.ws_bytes;
    set_spans();
    err = dg::launch_gemv_colstream(g, cp, plan->ws, plan->counters, s);
  } else {
    set_spans();
    err = dg::launch_gemv_generic(g, s, plan->sms, &info->grid);
  }
  return err == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// Kernel variant of a tensor-core plan.
int tc_mode(const gemm_config_info_t& info) {
  if (info.path == GEMM_PATH_TC_SPLITK_CLUSTER) return dg::TC_KPAIR;
  return info.cta_per_tile == 2 ? dg::TC_PAIR : dg::TC_SOLO;
}

bool planner_overridden() {
  static const char* vars[] = {"GEMM_FORCE_TILE", "GEMM_FORCE_SPLITK", "GEMM_RASTER_GROUP",
                               "GEMM_SPLITK_CLUSTER", "GEMM_TAIL_SPLIT", "GEMM_FUSED_REDUCE"};
  for (const char* v : vars) {
    const char* x = std::getenv(v);
    if (x && *x) return true;
  }
  return false;
}

// Plan a tensor-core call and encode its descriptors (cache miss).
gemm_status_t build_tc_entry(gemm_plan* plan, int64_t M, int64_t N, int64_t K, const void* A,
                             int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                             const CinRef& cin, bool beta_nz, gemm_dtype_t dtype, gemm_op_t ta,
                             gemm_op_t tb, const TcChoice* forced, TcEntry* e) {
  gemm_config_info_t* info = &e->info;
  const int c_es = out_is_f32(dtype) ? 4 : 2;
  const int eb = in_bytes(dtype);
  if (forced)
    fill_info(M, N, K, plan->sms, *forced, info, eb);
  else
    choose_tc(M, N, K, plan->sms, c_es, beta_nz, info, eb);
  const int bn = info->tile_n;
  const int S = info->splitk;
  const int mode = tc_mode(*info);
  const bool pair = mode == dg::TC_PAIR, kpair = mode == dg::TC_KPAIR;
  const int tile_m = info->tile_m;
  if (mode != dg::TC_SOLO) {  // the grid holds whole clusters that fit at once
    const int mc = dg::tc_max_clusters(bn, mode);
    if (mc <= 0) return GEMM_ERR_UNSUPPORTED;
    info->grid = int(2 * std::min<int64_t>(pair ? info->units : info->tiles, mc));
  }
  const bool f16 = in_is_f16(dtype), tf32 = in_is_tf32(dtype);
  const CUtensorMapDataType in_t = tf32  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                         : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int kbe = 128 / eb;  // K elements in one 128-byte swizzle row
  const bool a_mn = ta == GEMM_OP_T, b_mn = tb == GEMM_OP_N;
  // K-major: boxes of tile rows x one 128-byte row of K; M/N-major: boxes of
  // kbe K rows x one 128-byte row of M or N (kbe elements), swizzled in
  // 32-byte units for TF32, as the M/N-major kind::tf32 MMAs read them
  const CUtensorMapSwizzle mn_sw = tf32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B;
  bool ok = a_mn ? make_map(&e->ma, in_t, eb, A, M, K, lda, kbe, kbe, mn_sw)
                 : make_map(&e->ma, in_t, eb, A, K, M, lda, kbe, dg::TC_BM);
  ok = ok && (b_mn ? make_map(&e->mb, in_t, eb, B, N, K, ldb, kbe, kbe, mn_sw)
                   : make_map(&e->mb, in_t, eb, B, K, N, ldb, kbe, pair ? bn / 2 : bn));
  dg::TcParams& p = e->p;
  p = dg::TcParams{};
  p.M = int(M);
  p.N = int(N);
  p.K = int(K);
  p.num_m_blocks = int(ceil_div(M, tile_m));
  p.num_n_blocks = int(ceil_div(N, bn));
  p.k_blocks = int(ceil_div(K, kbe));
  p.tf32 = tf32;
  p.raster_group = info->raster_group;
  // units: whole tiles first, then the K slices of the tail tiles (all tiles
  // for split-K, the last wave's for a tail split, none otherwise)
  const int64_t tiles = int64_t(p.num_m_blocks) * p.num_n_blocks;
  const int tail = kpair ? 0 : info->tail_tiles;
  p.dp_units = int(tiles - tail);
  p.tail_tiles = tail;
  p.splitk = S;
  p.kb_per_split = int(ceil_div(p.k_blocks, S));
  p.units = kpair ? int(tiles) : p.dp_units + tail * S;
  p.out_kind = out_kind(dtype);
  p.a_mn_major = a_mn;
  p.b_mn_major = b_mn;
  p.idesc = make_idesc(tf32 ? 2 : (f16 ? 0 : 1), a_mn, b_mn, bn, tile_m);
  p.c_ptr = C;
  p.ldc = ldc;
  p.cin = cin.ptr;
  p.ldcin = cin.ld;
  p.cin_kind = cin.kind;
  // a C other than the output is read with plain loads in the epilogue
  p.cin_direct = beta_nz && (cin.ptr != C || cin.ld != ldc || cin.kind != p.out_kind);
  p.err = plan->err;
  // TMA stores write whole 16-byte pieces of a row: the map covers only the
  // 16-byte-aligned prefix of each row of C; the kernel writes the rest.
  p.n_tma = int((N * c_es) / 16 * 16 / c_es);
  const CUtensorMapDataType ct = out_is_f32(dtype) ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : in_t;
  if (p.n_tma > 0)
    ok = ok && make_map(&e->mc, ct, c_es, C, p.n_tma, M, ldc, 128 / c_es, 32);
  else  // every column is written (and read for beta) by the threads: a placeholder map
    ok = ok && make_map(&e->mc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, plan->err, 32, 32, 32, 32, 32);
  e->mw = e->mc;  // replaced by the workspace map before a launch that has tail tiles
  e->ws_ptr = nullptr;
  // fp32 partials, tile-major: [slice][tail tile][tile_m rows][bn columns]
  e->ws_bytes = size_t(tail) * size_t(S) * size_t(tile_m) * size_t(bn) * 4;
  info->workspace_bytes = int64_t(e->ws_bytes);
  p.fused_reduce = fused_fits(*info, mode, info->grid);
  info->launches = tail > 0 && !p.fused_reduce ? 2 : 1;
  return ok ? GEMM_OK : GEMM_ERR_CUDA;
}

// Launch the kernels of a planned call (the plan's workspace may grow).
gemm_status_t launch_entry(gemm_plan* plan, TcEntry* e, int64_t M, int64_t N, void* C, int64_t ldc,
                           float alpha, float beta, gemm_dtype_t dtype, gemm_epilogue_t epi,
                           cudaStream_t s) {
  // (the C that beta scales travels in e->p: cin, ldcin, cin_kind)
  dg::TcParams p = e->p;  // per-call fields below
  p.alpha = alpha;
  p.beta = beta;
  p.act = epi.act;
  p.slope = epi.slope;
  p.timeout_ns = plan->watchdog_ns;
  p.pdl = plan->pdl;
  const int mode = tc_mode(e->info);
  const int tail = e->p.tail_tiles;  // tiles whose K slices a second launch reduces
  if (tail > 0) {
    gemm_status_t st = ensure_ws(plan, e->ws_bytes, s);
    if (st == GEMM_OK && p.fused_reduce) st = ensure_counters(plan, size_t(tail), s);
    if (st != GEMM_OK) return st;
    p.ws = static_cast<const float*>(plan->ws);
    p.counters = plan->counters;
    if (e->ws_ptr != plan->ws) {  // (re-)encode the partial map for the current workspace
      const int64_t rows = int64_t(e->p.splitk) * tail * e->info.tile_m;
      if (!make_map(&e->mw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, plan->ws, e->info.tile_n, rows,
                    e->info.tile_n, 32, 32))
        return GEMM_ERR_CUDA;
      e->ws_ptr = plan->ws;
    }
  }
#ifdef DG_DEBUG
  {  // what the kernels touch with plain or bulk accesses: the output, beta's C, workspace, counters
    Spans sp(plan->err);
    sp.out_matrix(C, M, N, ldc, p.out_kind == dg::OUT_F32 ? 4 : 2);
    if (beta != 0.f) sp.matrix(p.cin, M, N, p.ldcin, p.cin_kind == dg::OUT_F32 ? 4 : 2);
    if (tail > 0) sp.bytes(plan->ws, int64_t(plan->ws_bytes)).bytes(plan->counters, int64_t(plan->counter_count) * 4);
    p.dbg = sp.s;
  }
#endif
  if (dg::launch_gemm_tc(e->info.tile_n, mode, e->ma, e->mb, e->mc, e->mw, p, e->info.grid, s) !=
      cudaSuccess)
    return GEMM_ERR_CUDA;
  if (tail > 0 && !p.fused_reduce) {
    dg::TileReduceArgs r{};
    r.ws = static_cast<const float*>(plan->ws);
    r.tail_tiles = tail;
    r.splits = e->p.splitk;
    r.tile0 = e->p.dp_units;
    r.tile_m = e->info.tile_m;
    r.tile_n = e->info.tile_n;
    r.num_m_blocks = e->p.num_m_blocks;
    r.num_n_blocks = e->p.num_n_blocks;
    r.raster_group = e->p.raster_group;
    r.M = int(M);
    r.N = int(N);
    r.C = C;
    r.ldc = ldc;
    r.Cin = e->p.cin;
    r.ldcin = e->p.ldcin;
    r.e = dg::EpiParams{alpha, beta, epi.slope, epi.act, out_kind(dtype), e->p.cin_kind};
    r.pdl = plan->pdl;
#ifdef DG_DEBUG
    r.dbg = p.dbg;
#endif
    if (dg::launch_tile_reduce(r, s, plan->sms) != cudaSuccess) return GEMM_ERR_CUDA;
  }
  return GEMM_OK;
}

// Benchmark mode ("Matrix Multiplication Background User's Guide", section
// 2.3: some frameworks time every implementation option once and keep the
// fastest): time the planner's leading candidates on this call's stream,
// writing into a scratch copy of C, and return the fastest.  Falls back to
// the planner's pick if anything fails.
TcChoice autotune(gemm_plan* plan, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                  const void* B, int64_t ldb, const void* C, int64_t ldc, const CinRef& cin, float alpha,
                  float beta, gemm_dtype_t dtype, gemm_op_t ta, gemm_op_t tb, gemm_epilogue_t epi,
                  cudaStream_t s) {
  const int c_es = out_is_f32(dtype) ? 4 : 2;
  std::vector<TcChoice> all;
  TcChoice best;
  tc_candidates(M, N, K, plan->sms, c_es, beta != 0.f, &best, &all, in_bytes(dtype));
  std::stable_sort(all.begin(), all.end(), [](const TcChoice& x, const TcChoice& y) { return x.t < y.t; });
  std::vector<TcChoice> trial{best};
  for (const TcChoice& c : all) {
    if (trial.size() >= 6 || c.t > 1.15 * all.front().t) break;
    bool dup = false;
    for (const TcChoice& d : trial) dup |= d.bn == c.bn && d.mode == c.mode && d.s == c.s && d.tail == c.tail;
    if (!dup) trial.push_back(c);
  }
  if (trial.size() < 2) return best;
  const size_t c_bytes = (size_t(M - 1) * size_t(ldc) + size_t(N)) * size_t(c_es);
  void* scratch = nullptr;
  if (cudaMallocAsync(&scratch, c_bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return best;
  }
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  // The trials write the scratch; when beta scales the output itself they
  // read the scratch copy of it too, else the separate C (never written).
  const bool in_place = cin.ptr == C;
  const CinRef cin_trial = in_place ? CinRef{scratch, ldc, cin.kind} : cin;
  bool ok = (!in_place || beta == 0.f ||
             cudaMemcpyAsync(scratch, C, c_bytes, cudaMemcpyDeviceToDevice, s) == cudaSuccess) &&
            cudaEventCreate(&e0) == cudaSuccess && cudaEventCreate(&e1) == cudaSuccess;
  TcChoice fastest = best;
  float fastest_ms = 1e30f;
  constexpr int kReps = 3;
  for (size_t i = 0; ok && i < trial.size(); ++i) {
    TcEntry ent;
    if (build_tc_entry(plan, M, N, K, A, lda, B, ldb, scratch, ldc, cin_trial, beta != 0.f, dtype, ta, tb,
                       &trial[i], &ent) != GEMM_OK)
      continue;
    if (launch_entry(plan, &ent, M, N, scratch, ldc, alpha, beta, dtype, epi, s) != GEMM_OK) continue;
    bool run_ok = cudaEventRecord(e0, s) == cudaSuccess;
    for (int r = 0; r < kReps && run_ok; ++r)
      run_ok = launch_entry(plan, &ent, M, N, scratch, ldc, alpha, beta, dtype, epi, s) == GEMM_OK;
    float ms = 0.f;
    run_ok = run_ok && cudaEventRecord(e1, s) == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess &&
             cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess;
    if (!run_ok) {
      cudaGetLastError();
      ok = false;
      break;
    }
    if (ms < fastest_ms * 0.99f) {  // the earlier (planner-ranked) choice unless clearly faster
      fastest_ms = ms;
      fastest = trial[i];
    }
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaFreeAsync(scratch, s);
  return ok ? fastest : best;
}

gemm_status_t run_tc(gemm_plan* plan, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                     const void* B, int64_t ldb, void* C, int64_t ldc, const CinRef& cin, float alpha,
                     float beta, gemm_dtype_t dtype, gemm_op_t ta, gemm_op_t tb, gemm_epilogue_t epi,
                     cudaStream_t s, gemm_config_info_t* info) {
  const TcKey key{M, N, K, lda, ldb, ldc, reinterpret_cast<uintptr_t>(A), reinterpret_cast<uintptr_t>(B),
                  reinterpret_cast<uintptr_t>(C), int32_t(dtype), int32_t(ta), int32_t(tb),
                  int32_t(beta != 0.f), reinterpret_cast<uintptr_t>(cin.ptr), cin.ld, int32_t(cin.kind)};
  const bool use_cache = !planner_overridden();
  TcEntry local;
  TcEntry* e = nullptr;
  if (use_cache) {
    auto it = plan->tc_cache.find(key);
    if (it != plan->tc_cache.end()) e = &it->second;
  }
  if (e == nullptr) {
    const TcChoice* forced = nullptr;
    TcChoice tuned;
    // Benchmark mode synchronizes on its trials: not while the stream is
    // being captured into a CUDA graph (the planner's estimate decides then).
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (plan->autotune && cudaStreamIsCapturing(s, &capture) != cudaSuccess) {
      cudaGetLastError();
      capture = cudaStreamCaptureStatusActive;
    }
    if (plan->autotune && use_cache && capture == cudaStreamCaptureStatusNone) {
      TcKey shape = key;
      shape.A = shape.B = shape.C = shape.Cin = 0;
      shape.cin_kind = cin.ptr == C ? -1 : cin.kind;  // in place, or a separate C of this kind
      auto t = plan->tuned.find(shape);
      if (t == plan->tuned.end())
        t = plan->tuned.emplace(shape, autotune(plan, M, N, K, A, lda, B, ldb, C, ldc, cin, alpha, beta,
                                                dtype, ta, tb, epi, s)).first;
      tuned = t->second;
      forced = &tuned;
      if (plan->tuned.size() > 4096) plan->tuned.clear();  // bounded; re-tuned on next use
    }
    const gemm_status_t st = build_tc_entry(plan, M, N, K, A, lda, B, ldb, C, ldc, cin, beta != 0.f, dtype,
                                            ta, tb, forced, &local);
    if (st != GEMM_OK) return st;
    if (use_cache) {
      if (plan->tc_cache.size() >= 256) plan->tc_cache.clear();
      e = &plan->tc_cache.emplace(key, local).first->second;
    } else {
      e = &local;
    }
  }
  *info = e->info;
  return launch_entry(plan, e, M, N, C, ldc, alpha, beta, dtype, epi, s);
}

}  // namespace

// =================================================================== C ABI

extern "C" {

const char* gemm_status_string(gemm_status_t st) {
  switch (st) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG: invalid argument";
    case GEMM_ERR_ALIGNMENT: return "GEMM_ERR_ALIGNMENT: pointer or leading dimension misaligned";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED: size not supported";
    case GEMM_ERR_NO_DEVICE: return "GEMM_ERR_NO_DEVICE: no compute capability 10.x CUDA device";
    case GEMM_ERR_OUT_OF_MEMORY: return "GEMM_ERR_OUT_OF_MEMORY: workspace allocation failed";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: CUDA call or kernel launch failed";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT: a kernel wait ran out (watchdog)";
    case GEMM_ERR_DEBUG_CHECK: return "GEMM_ERR_DEBUG_CHECK: a kernel's bounds or copy-rule check failed (debug build)";
  }
  return "unknown gemm_status_t";
}

gemm_status_t gemm_plan_create(gemm_plan_t* plan, int device) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  *plan = nullptr;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || device < 0 || device >= count) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess || prop.major != 10) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  if (!encode_fn()) return GEMM_ERR_NO_DEVICE;
  DeviceGuard guard(device);
  gemm_plan* p = new gemm_plan();
  p->device = device;
  p->sms = prop.multiProcessorCount;
  p->autotune = env_int("GEMM_AUTOTUNE", 0) != 0;
  p->pdl = env_int("GEMM_PDL", 1) != 0;
  p->log = env_int("GEMM_LOG", 0) != 0;
  p->nvtx = env_int("GEMM_NVTX", 0) != 0;
  if (const char* w = std::getenv("GEMM_WATCHDOG_NS")) {
    const unsigned long long v = std::strtoull(w, nullptr, 10);
    if (v >= 1000) p->watchdog_ns = v;
  }
  if (cudaMalloc(&p->err, sizeof(int)) != cudaSuccess || cudaMemset(p->err, 0, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    if (p->err) cudaFree(p->err);
    delete p;
    return GEMM_ERR_OUT_OF_MEMORY;
  }
  *plan = p;
  return GEMM_OK;
}

gemm_status_t gemm_plan_destroy(gemm_plan_t plan) {
  if (!plan) return GEMM_OK;
  DeviceGuard guard(plan->device);
  cudaDeviceSynchronize();
  if (plan->ws) cudaFree(plan->ws);
  if (plan->tws) cudaFree(plan->tws);
  if (plan->counters) cudaFree(plan->counters);
  if (plan->err) cudaFree(plan->err);
  delete plan;
  return GEMM_OK;
}

gemm_status_t gemm_check_args(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                              const void* B, int64_t ldb, const void* C, int64_t ldc, float alpha,
                              gemm_dtype_t dtype, gemm_op_t transA, gemm_op_t transB,
                              gemm_epilogue_t epilogue) {
  return check(M, N, K, A, lda, B, ldb, C, ldc, alpha, dtype, transA, transB, epilogue);
}

namespace {

// GEMM_LOG=1: the decisions of a planned call, one line on stderr.
void log_config(const char* who, int64_t M, int64_t N, int64_t K, int dtype, int ta, int tb,
                const gemm_config_info_t& c) {
  static const char* kPath[] = {"none", "tc", "tc_splitk", "gemv_rowdot", "gemv_colstream", "gemv_generic",
                                "scale", "tc_splitk_cluster", "tc_tail_split"};
  static const char* kType[] = {"bf16->f32", "bf16->bf16", "f16->f32", "f16->f16", "tf32->f32"};
  const char* path = c.path >= 0 && c.path <= 8 ? kPath[c.path] : "?";
  const char* type = dtype >= 0 && dtype <= 4 ? kType[dtype] : "?";
  std::fprintf(stderr,
               "gemm_log %s: %lldx%lldx%lld %s op(A)=%c op(B)=%c -> %s tile %dx%d cta/tile %d split %d tail "
               "tiles %d grid %d sms %d tiles %lld waves %.3f tail fraction %.3f launches %d workspace %lld B\n",
               who, (long long)M, (long long)N, (long long)K, type, ta ? 'T' : 'N', tb ? 'T' : 'N', path, c.tile_m,
               c.tile_n, c.cta_per_tile, c.splitk, c.tail_tiles, c.grid, c.sms, (long long)c.tiles, c.waves,
               c.tail_fraction, c.launches, (long long)c.workspace_bytes);
}

int type_kind(gemm_type_t t) {
  return t == GEMM_TYPE_F32 ? dg::OUT_F32 : (t == GEMM_TYPE_BF16 ? dg::OUT_BF16 : dg::OUT_F16);
}

// Arguments of gemm_run_ex; *dtype receives the (operand, output) pair.
gemm_status_t check_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                       int64_t ldb, const void* C, int64_t ldc, gemm_type_t c_type, const void* D,
                       int64_t ldd, gemm_type_t d_type, float alpha, float beta, gemm_type_t ab_type,
                       gemm_op_t ta, gemm_op_t tb, gemm_epilogue_t epi, gemm_dtype_t* dtype) {
  if (ab_type != GEMM_TYPE_BF16 && ab_type != GEMM_TYPE_F16 && ab_type != GEMM_TYPE_TF32)
    return GEMM_ERR_INVALID_ARG;
  if (d_type != GEMM_TYPE_F32 && (d_type != ab_type || ab_type == GEMM_TYPE_TF32)) return GEMM_ERR_INVALID_ARG;
  if (c_type != GEMM_TYPE_BF16 && c_type != GEMM_TYPE_F16 && c_type != GEMM_TYPE_F32)
    return GEMM_ERR_INVALID_ARG;
  const bool f32 = d_type == GEMM_TYPE_F32;
  *dtype = ab_type == GEMM_TYPE_TF32 ? GEMM_TF32_F32
           : ab_type == GEMM_TYPE_BF16 ? (f32 ? GEMM_BF16_F32 : GEMM_BF16_BF16)
                                       : (f32 ? GEMM_F16_F32 : GEMM_F16_F16);
  // D is held to gemm_run's rules for C
  const gemm_status_t st = check(M, N, K, A, lda, B, ldb, D, ldd, alpha, *dtype, ta, tb, epi);
  if (st != GEMM_OK || M == 0 || N == 0 || beta == 0.f) return st;
  if (C == nullptr || ldc < std::max<int64_t>(1, N)) return GEMM_ERR_INVALID_ARG;
  const size_t c_es = c_type == GEMM_TYPE_F32 ? 4 : 2, d_es = f32 ? 4 : 2;
  if (!aligned(C, c_es)) return GEMM_ERR_ALIGNMENT;
  if (C == D) return ldc == ldd && c_type == d_type ? GEMM_OK : GEMM_ERR_INVALID_ARG;
  // a separate C must not share a byte with D (it may overlap A or B: all three are only read)
  if (overlaps(region(C, M, N, ldc, int64_t(c_es)), region(D, M, N, ldd, int64_t(d_es))))
    return GEMM_ERR_INVALID_ARG;
  return GEMM_OK;
}

// Dispatch of a checked call: D <- act(alpha * op(A) @ op(B) + beta * cin).
gemm_status_t run_all(gemm_plan_t plan, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                      const void* B, int64_t ldb, void* D, int64_t ldd, const CinRef& cin, float alpha,
                      float beta, gemm_dtype_t dtype, gemm_op_t transA, gemm_op_t transB,
                      gemm_epilogue_t epilogue, void* stream) {
  struct NvtxRange {  // pops the range on every return
    bool on;
    ~NvtxRange() {
      if (on) nvtxRangePop();
    }
  } range{plan->nvtx};
  if (plan->nvtx) {
    static const char* kType[] = {"bf16->f32", "bf16->bf16", "f16->f32", "f16->f16", "tf32->f32"};
    char name[96];
    std::snprintf(name, sizeof name, "gemm %lldx%lldx%lld %s %c%c", (long long)M, (long long)N, (long long)K,
                  kType[int(dtype)], transA == GEMM_OP_T ? 'T' : 'N', transB == GEMM_OP_T ? 'T' : 'N');
    nvtxRangePushA(name);
  }
  gemm_config_info_t info{};
  info.sms = plan->sms;
  info.splitk = 1;
  if (M == 0 || N == 0) {
    info.path = GEMM_PATH_NONE;
    plan->last = info;
    return GEMM_OK;
  }
  DeviceGuard guard(plan->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dg::EpiParams e{alpha, beta, epilogue.slope, epilogue.act, out_kind(dtype), cin.kind};
  gemm_status_t r;
  bool copy_a = false, copy_b = false;  // TF32 operands copied K-major first (tf32_copies)
  if (K == 0 || alpha == 0.f) {
    info.path = GEMM_PATH_SCALE;
    info.launches = 1;
    dg::DbgSpans dbg{};
#ifdef DG_DEBUG
    {
      Spans sp(plan->err);
      sp.out_matrix(D, M, N, ldd, e.out_kind == dg::OUT_F32 ? 4 : 2);
      if (beta != 0.f) sp.matrix(cin.ptr, M, N, cin.ld, cin.kind == dg::OUT_F32 ? 4 : 2);
      dbg = sp.s;
    }
#endif
    r = dg::launch_scale(int(M), int(N), D, ldd, cin.ptr, cin.ld, e, s, plan->sms, dbg) == cudaSuccess
            ? GEMM_OK
            : GEMM_ERR_CUDA;
  } else if ((M == 1 || N == 1) && !in_is_tf32(dtype)) {
    r = run_gemv(plan, M, N, K, A, lda, B, ldb, D, ldd, dtype, transA, transB, e, cin, s, &info);
  } else if (in_is_tf32(dtype) && (transA == GEMM_OP_T || transB == GEMM_OP_N) &&
             (tf32_copies(M, N, K, transA, transB, &copy_a, &copy_b), copy_a || copy_b)) {
    // Copy the chosen M/N-major TF32 operands K-major into plan workspace
    // (row stride rounded to 4 elements, 16 bytes); the others stay in place.
    const int64_t lda_t = (K + 3) & ~int64_t(3), ldb_t = lda_t;
    const size_t a_bytes = copy_a ? size_t(M) * size_t(lda_t) * 4 : 0;
    const size_t b_bytes = copy_b ? size_t(N) * size_t(ldb_t) * 4 : 0;
    const size_t a_off = 0, b_off = (a_bytes + 255) & ~size_t(255);
    r = ensure_buffer(&plan->tws, &plan->tws_bytes, b_off + b_bytes, s);
    const void* A2 = A;
    const void* B2 = B;
    int64_t lda2 = lda, ldb2 = ldb;
    if (r == GEMM_OK && a_bytes) {  // A stored K x M -> M x K
      A2 = static_cast<char*>(plan->tws) + a_off;
      lda2 = lda_t;
      dg::DbgSpans dbg{};
#ifdef DG_DEBUG
      dbg = Spans(plan->err).matrix(A, K, M, lda, 4).matrix(A2, M, K, lda2, 4).s;
#endif
      if (dg::launch_transpose32(A, lda, int(K), int(M), const_cast<void*>(A2), lda2, s, dbg) != cudaSuccess)
        r = GEMM_ERR_CUDA;
    }
    if (r == GEMM_OK && b_bytes) {  // B stored K x N -> N x K
      B2 = static_cast<char*>(plan->tws) + b_off;
      ldb2 = ldb_t;
      dg::DbgSpans dbg{};
#ifdef DG_DEBUG
      dbg = Spans(plan->err).matrix(B, K, N, ldb, 4).matrix(B2, N, K, ldb2, 4).s;
#endif
      if (dg::launch_transpose32(B, ldb, int(K), int(N), const_cast<void*>(B2), ldb2, s, dbg) != cudaSuccess)
        r = GEMM_ERR_CUDA;
    }
    if (r == GEMM_OK)
      r = run_tc(plan, M, N, K, A2, lda2, B2, ldb2, D, ldd, cin, alpha, beta, dtype,
                 copy_a ? GEMM_OP_N : transA, copy_b ? GEMM_OP_T : transB, epilogue, s, &info);
    info.launches += int(a_bytes > 0) + int(b_bytes > 0);
  } else {
    r = run_tc(plan, M, N, K, A, lda, B, ldb, D, ldd, cin, alpha, beta, dtype, transA, transB, epilogue,
               s, &info);
  }
  if (r != GEMM_OK) cudaGetLastError();
  plan->last = info;
  if (plan->log && r == GEMM_OK) log_config("gemm_run", M, N, K, dtype, transA, transB, info);
  return r;
}

}  // namespace

gemm_status_t gemm_run(gemm_plan_t plan, int64_t M, int64_t N, int64_t K, const void* A,
                       int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, float alpha,
                       float beta, gemm_dtype_t dtype, gemm_op_t transA, gemm_op_t transB,
                       gemm_epilogue_t epilogue, void* stream) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  const gemm_status_t st =
      check(M, N, K, A, lda, B, ldb, C, ldc, alpha, dtype, transA, transB, epilogue);
  if (st != GEMM_OK) return st;
  const CinRef cin{C, ldc, out_kind(dtype)};
  return run_all(plan, M, N, K, A, lda, B, ldb, C, ldc, cin, alpha, beta, dtype, transA, transB,
                 epilogue, stream);
}

gemm_status_t gemm_run_ex(gemm_plan_t plan, int64_t M, int64_t N, int64_t K, const void* A,
                          int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc,
                          gemm_type_t c_type, void* D, int64_t ldd, gemm_type_t d_type, float alpha,
                          float beta, gemm_type_t ab_type, gemm_op_t transA, gemm_op_t transB,
                          gemm_epilogue_t epilogue, void* stream) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  gemm_dtype_t dtype = GEMM_BF16_F32;
  const gemm_status_t st = check_ex(M, N, K, A, lda, B, ldb, C, ldc, c_type, D, ldd, d_type, alpha, beta,
                                    ab_type, transA, transB, epilogue, &dtype);
  if (st != GEMM_OK) return st;
  // with beta == 0 C is not read: the output stands in for it
  const CinRef cin = beta != 0.f ? CinRef{C, ldc, type_kind(c_type)} : CinRef{D, ldd, out_kind(dtype)};
  return run_all(plan, M, N, K, A, lda, B, ldb, D, ldd, cin, alpha, beta, dtype, transA, transB,
                 epilogue, stream);
}

gemm_status_t gemm_check_args_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                 const void* B, int64_t ldb, const void* C, int64_t ldc,
                                 gemm_type_t c_type, const void* D, int64_t ldd, gemm_type_t d_type,
                                 float alpha, float beta, gemm_type_t ab_type, gemm_op_t transA,
                                 gemm_op_t transB, gemm_epilogue_t epilogue) {
  gemm_dtype_t dtype = GEMM_BF16_F32;
  return check_ex(M, N, K, A, lda, B, ldb, C, ldc, c_type, D, ldd, d_type, alpha, beta, ab_type, transA,
                  transB, epilogue, &dtype);
}

gemm_status_t gemm_plan_last_config(gemm_plan_t plan, gemm_config_info_t* out) {
  if (!plan || !out) return GEMM_ERR_INVALID_ARG;
  *out = plan->last;
  return GEMM_OK;
}

gemm_status_t gemm_plan_poll_error(gemm_plan_t plan, void* stream) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  DeviceGuard guard(plan->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  int h = 0;
  if (cudaMemcpy(&h, plan->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
  plan->last_err_bits = h;
  if (h == 0) return GEMM_OK;
  if (cudaMemset(plan->err, 0, sizeof(int)) != cudaSuccess) return GEMM_ERR_CUDA;
  // A kernel that gave up may have left arrival counters above zero.
  if (plan->counters && cudaMemset(plan->counters, 0, plan->counter_count * sizeof(unsigned)) != cudaSuccess)
    return GEMM_ERR_CUDA;
  return (h & dg::DBG_FLAG) ? GEMM_ERR_DEBUG_CHECK : GEMM_ERR_TIMEOUT;
}

gemm_status_t gemm_plan_last_error_bits(gemm_plan_t plan, int64_t* bits) {
  if (!plan || !bits) return GEMM_ERR_INVALID_ARG;
  *bits = plan->last_err_bits;
  return GEMM_OK;
}

int gemm_debug_build(void) {
#ifdef DG_DEBUG
  return 1;
#else
  return 0;
#endif
}

gemm_status_t gemm_plan_set_watchdog(gemm_plan_t plan, uint64_t timeout_ns) {
  if (!plan || timeout_ns < 1000) return GEMM_ERR_INVALID_ARG;
  plan->watchdog_ns = timeout_ns;
  return GEMM_OK;
}

gemm_status_t gemm_plan_set_autotune(gemm_plan_t plan, int enable) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  plan->autotune = enable != 0;
  return GEMM_OK;
}

gemm_status_t gemm_plan_tuned_count(gemm_plan_t plan, int64_t* count) {
  if (!plan || !count) return GEMM_ERR_INVALID_ARG;
  *count = int64_t(plan->tuned.size());
  return GEMM_OK;
}

gemm_status_t gemm_plan_selftest_watchdog(gemm_plan_t plan, void* stream) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  DeviceGuard guard(plan->device);
  if (dg::launch_watchdog_selftest(plan->err, plan->watchdog_ns, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return gemm_plan_poll_error(plan, stream);
}

namespace {
gemm_status_t choose_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, gemm_op_t transA,
                            gemm_op_t transB, int32_t sms, gemm_config_info_t* out);
}  // namespace

gemm_status_t gemm_choose_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                                 gemm_op_t transA, gemm_op_t transB, int32_t sms,
                                 gemm_config_info_t* out) {
  const gemm_status_t st = choose_config(M, N, K, dtype, transA, transB, sms, out);
  if (st == GEMM_OK && env_int("GEMM_LOG", 0) != 0) log_config("gemm_choose_config", M, N, K, dtype, transA, transB, *out);
  return st;
}

namespace {
gemm_status_t choose_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, gemm_op_t transA,
                            gemm_op_t transB, int32_t sms, gemm_config_info_t* out) {
  if (!out || sms <= 0 || M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (dtype < GEMM_BF16_F32 || dtype > GEMM_TF32_F32) return GEMM_ERR_INVALID_ARG;
  if ((transA != GEMM_OP_N && transA != GEMM_OP_T) || (transB != GEMM_OP_N && transB != GEMM_OP_T))
    return GEMM_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  out->sms = sms;
  out->splitk = 1;
  if (M == 0 || N == 0) {
    out->path = GEMM_PATH_NONE;
    return GEMM_OK;
  }
  if (K == 0) {
    out->path = GEMM_PATH_SCALE;
    out->launches = 1;
    return GEMM_OK;
  }
  if ((M == 1 || N == 1) && !in_is_tf32(dtype)) {
    const bool row_major_w = N == 1 ? transA == GEMM_OP_N : transB == GEMM_OP_T;
    const int64_t R = N == 1 ? M : N;
    out->launches = 1;
    if (row_major_w) {
      out->path = K <= dg::gemv_rowdot_max_k() ? GEMM_PATH_GEMV_ROWDOT : GEMM_PATH_GEMV_GENERIC;
    } else {
      const dg::ColstreamPlan cp = dg::plan_gemv_colstream(int(R), int(K), sms);
      out->path = GEMM_PATH_GEMV_COLSTREAM;
      out->splitk = cp.ksplit;
      out->grid = cp.panels * cp.ksplit;
      out->workspace_bytes = cp.ws_bytes;
    }
    return GEMM_OK;
  }
  choose_tc(M, N, K, sms, out_is_f32(dtype) ? 4 : 2, false, out, in_bytes(dtype));
  return GEMM_OK;
}
}  // namespace

gemm_status_t gemm_quantization(int64_t M, int64_t N, int32_t tile_m, int32_t tile_n,
                                int32_t splitk, int32_t sms, int32_t ctas_per_sm,
                                gemm_config_info_t* out) {
  if (!out || M < 0 || N < 0 || tile_m <= 0 || tile_n <= 0 || splitk <= 0 || sms <= 0 ||
      ctas_per_sm <= 0)
    return GEMM_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  quantization(M, N, tile_m, tile_n, splitk, sms, ctas_per_sm, out);
  return GEMM_OK;
}

}  // extern "C"
