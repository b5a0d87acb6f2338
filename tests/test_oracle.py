"""Pins for the CPU oracle: checks it against what the pages and the
mathematics fix, never against itself.

- The worked example of "Learning Triton One Kernel at a Time: Matrix
  Multiplication", section Tiled GEMM ((4,6)@(6,4) split into 3-element partial
  dot products and (2,2) blocks).
- Identity and permutation matrices; the transpose flags and
  (A@B)^T = B^T@A^T ("Learning Triton ...", section Memory coalescing: a
  transpose changes strides, not memory).
- Linearity in alpha and beta; LeakyReLU special cases ("OpenAI open-sources
  the Triton GPU language (part 2)", section Matrix multiplication).
- Exact rational brute force for every M, N, K in 1..6 ("Matrix
  Multiplication Background User's Guide", section 2: each output is a K-long
  dot product).
- Output rounding and input decoding against exact rationals and numpy.
"""
import json
import os
from fractions import Fraction

import math

import numpy as np
import pytest

from dense_gemm_mma_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# (significand bits incl. hidden bit, minimum normal exponent, largest finite value)
FORMATS = {
    "bf16": (8, -126, (2 - Fraction(1, 2 ** 7)) * Fraction(2) ** 127),
    "f16": (11, -14, Fraction(65504)),
    "f32": (24, -126, (2 - Fraction(1, 2 ** 23)) * Fraction(2) ** 127),
}


def round_fraction(q: Fraction, fmt: str):
    """Exact round-to-nearest-even of a rational to a binary format (inf on overflow)."""
    p, emin, maxval = FORMATS[fmt]
    if q == 0:
        return Fraction(0)
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    quantum = Fraction(2) ** (e - (p - 1))
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * quantum
    if r > maxval:
        return float("inf") if q > 0 else float("-inf")
    return r if q > 0 else -r


def dec(bits, fmt):
    """Independent numpy decode of stored bit patterns to float64."""
    bits = np.asarray(bits)
    if fmt == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if fmt == "f16":
        return bits.astype(np.uint16).view(np.float16).astype(np.float64)
    if fmt == "tf32":  # 10 of the 23 fraction bits: clear the 13 lowest of the fp32 word
        w = np.ascontiguousarray(bits, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFFE000)
        return w.view(np.float32).astype(np.float64)
    return np.asarray(bits, dtype=np.float32).astype(np.float64)


def enc_small(vals, fmt):
    """Encode exactly representable small values."""
    v = np.asarray(vals, dtype=np.float32)
    if fmt == "bf16":
        bits = v.view(np.uint32)
        assert np.all(bits & np.uint32(0xFFFF) == 0)
        return (bits >> np.uint32(16)).astype(np.uint16)
    if fmt == "f16":
        return v.astype(np.float16).view(np.uint16)
    return v


def stored(mat_logical, trans):
    """Stored array for an operand given its logical (op) matrix."""
    return np.ascontiguousarray(mat_logical.T if trans else mat_logical)


# ---------------------------------------------------------------- worked example

def test_worked_example_tiled_decomposition(oracle_lib):
    spec = json.load(open(os.path.join(GOLDEN, "worked_example_4x6x4.json")))
    (m, n), (n2, k) = spec["shape_X"], spec["shape_Y"]
    assert n == n2 and spec["shape_Z"] == [m, k]
    # small integers: every product and sum is exact in fp64 and in the formats
    X = [[(3 * i + 5 * j) % 7 - 3 for j in range(n)] for i in range(m)]
    Y = [[(2 * i + 3 * j) % 5 - 2 for j in range(k)] for i in range(n)]
    Xb = enc_small(X, "bf16")
    Yb = enc_small(Y, "bf16")
    # page convention: X (M,N) @ Y (N,K); library convention: A (M x K) @ B (K x N)
    exact, out = oracle_lib.gemm(m, k, n, Xb, Yb, in_fmt="bf16", out_fmt="f32")
    assert exact.shape == (4, 4)

    def dot(xs, ys):
        return sum(a * b for a, b in zip(xs, ys))

    # Z[0,0] as two 3-element partial dot products
    (a0, a1), (b0, b1) = spec["partial_dot_splits"]
    col0 = [Y[r][0] for r in range(n)]
    z00 = dot(X[0][a0:a1], col0[a0:a1]) + dot(X[0][b0:b1], col0[b0:b1])
    assert exact[0, 0] == z00
    assert out[0, 0] == z00

    # every (2,2) block of Z as a sum of three (2,2)@(2,2) block products
    bs = spec["block"][0]
    for bi in range(0, m, bs):
        for bj in range(0, k, bs):
            acc = [[0] * bs for _ in range(bs)]
            for lo, hi in spec["shared_blocks"]:
                for r in range(bs):
                    for c in range(bs):
                        acc[r][c] += dot(X[bi + r][lo:hi], [Y[t][bj + c] for t in range(lo, hi)])
            assert np.array_equal(exact[bi:bi + bs, bj:bj + bs], np.array(acc, dtype=np.float64))


# ------------------------------------------------------------ identity / permutation

def test_identity_and_permutation(oracle_lib):
    M, K, N = 5, 7, 3
    A = inputs.matrix(M, K, 11, 0, "bf16")
    B = inputs.matrix(K, N, 11, 1, "bf16")
    eye_k = enc_small(np.eye(K), "bf16")
    eye_m = enc_small(np.eye(M), "bf16")
    e1, _ = oracle_lib.gemm(M, K, K, A, eye_k)
    assert np.array_equal(e1, dec(A, "bf16"))          # A @ I = A
    e2, _ = oracle_lib.gemm(M, K, M, eye_m, A)
    assert np.array_equal(e2, dec(A, "bf16"))          # I @ A = A
    ref, _ = oracle_lib.gemm(M, N, K, A, B)
    rng = np.random.default_rng(3)
    p = rng.permutation(M)
    e3, _ = oracle_lib.gemm(M, N, K, np.ascontiguousarray(A[p]), B)
    assert np.array_equal(e3, ref[p])                  # (P A) B = P (A B)
    q = rng.permutation(N)
    e4, _ = oracle_lib.gemm(M, N, K, A, np.ascontiguousarray(B[:, q]))
    assert np.array_equal(e4, ref[:, q])               # A (B Q) = (A B) Q
    # permuting the shared dimension is exact on integer data
    Ai = enc_small(np.arange(M * K).reshape(M, K) % 9 - 4, "bf16")
    Bi = enc_small(np.arange(K * N).reshape(K, N) % 7 - 3, "bf16")
    s = rng.permutation(K)
    r1, _ = oracle_lib.gemm(M, N, K, Ai, Bi)
    r2, _ = oracle_lib.gemm(M, N, K, np.ascontiguousarray(Ai[:, s]), np.ascontiguousarray(Bi[s]))
    assert np.array_equal(r1, r2)
    # a permutation matrix moves rows
    P = enc_small(np.eye(M)[p], "bf16")
    e5, _ = oracle_lib.gemm(M, K, M, P, A)
    assert np.array_equal(e5, dec(A, "bf16")[p])


# ----------------------------------------------------------------- transposes

@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_transpose_flags_and_identity(oracle_lib, fmt):
    M, N, K = 6, 5, 9
    A = inputs.matrix(M, K, 21, 0, fmt)
    B = inputs.matrix(K, N, 21, 1, fmt)
    ref, ref_out = oracle_lib.gemm(M, N, K, A, B, in_fmt=fmt)
    for ta in (False, True):
        for tb in (False, True):
            e, o = oracle_lib.gemm(M, N, K, stored(A, ta), stored(B, tb), in_fmt=fmt,
                                   transA=ta, transB=tb)
            assert np.array_equal(e, ref), (ta, tb)
            assert np.array_equal(o, ref_out)
    # (A@B)^T = B^T @ A^T: op(A') = B^T (N x K) stored as B with transA, op(B') = A^T
    et, _ = oracle_lib.gemm(N, M, K, B, A, in_fmt=fmt, transA=True, transB=True)
    assert np.array_equal(et, ref.T)


def test_leading_dimensions_padding_not_read(oracle_lib):
    M, N, K = 4, 3, 5
    A = inputs.matrix(M, K, 5, 0, "bf16", ld=K + 3)     # NaN sentinels in the padding
    B = inputs.matrix(K, N, 5, 1, "bf16", ld=N + 5)
    Ad = np.ascontiguousarray(A[:, :K])
    Bd = np.ascontiguousarray(B[:, :N])
    e1, _ = oracle_lib.gemm(M, N, K, A, B)
    e2, _ = oracle_lib.gemm(M, N, K, Ad, Bd)
    assert np.all(np.isfinite(e1)) and np.array_equal(e1, e2)


# ------------------------------------------------------------------ epilogue

def test_alpha_beta_linearity(oracle_lib):
    M, N, K = 4, 6, 8
    A = enc_small(np.arange(M * K).reshape(M, K) % 5 - 2, "bf16")
    B = enc_small(np.arange(K * N).reshape(K, N) % 3 - 1, "bf16")
    C = (np.arange(M * N).reshape(M, N) % 7 - 3).astype(np.float32)
    s, _ = oracle_lib.gemm(M, N, K, A, B)
    e2, _ = oracle_lib.gemm(M, N, K, A, B, alpha=2.0)
    assert np.array_equal(e2, 2 * s)                   # power-of-two alpha is exact
    for alpha, beta in [(1.0, 1.0), (0.5, -2.0), (-3.0, 0.25), (0.0, 1.5)]:
        e, _ = oracle_lib.gemm(M, N, K, A, B, C=C, alpha=alpha, beta=beta)
        # d(alpha, beta) = alpha * d(1, 0) + beta * C, exact on these dyadic values
        assert np.array_equal(e, alpha * s + beta * C.astype(np.float64))


def test_separate_c_format(oracle_lib):
    """A separate C is decoded in its own format: the same values given as
    bf16, fp16 or fp32 C give the same result, and D's format only decides
    the final rounding."""
    M, N, K = 5, 6, 9
    A = inputs.matrix(M, K, 15, 0, "bf16")
    B = inputs.matrix(K, N, 15, 1, "bf16")
    Cb = inputs.matrix(M, N, 15, 2, "bf16")
    Cf = (Cb.astype(np.uint32) << np.uint32(16)).view(np.float32)   # the same values, as fp32
    Ch = inputs.f32_to_f16_bits(Cf)
    ref, _ = oracle_lib.gemm(M, N, K, A, B, C=Cb, beta=0.75, out_fmt="bf16")
    for C, fmt in ((Cf, "f32"), (Cb, "bf16")):
        for out in ("f32", "bf16", "f16"):
            e, _ = oracle_lib.gemm(M, N, K, A, B, C=C, beta=0.75, out_fmt=out, c_fmt=fmt)
            assert np.array_equal(e, ref)
    hvals = Ch.view(np.float16).astype(np.float64)
    e, _ = oracle_lib.gemm(M, N, K, A, B, C=Ch, beta=0.75, out_fmt="f32", c_fmt="f16")
    plain, _ = oracle_lib.gemm(M, N, K, A, B)
    assert np.array_equal(e, plain + 0.75 * hvals)


def test_beta_zero_does_not_read_c(oracle_lib):
    M, N, K = 3, 4, 5
    A = inputs.matrix(M, K, 9, 0, "bf16")
    B = inputs.matrix(K, N, 9, 1, "bf16")
    Cnan = np.full((M, N), np.nan, dtype=np.float32)
    e, o = oracle_lib.gemm(M, N, K, A, B, C=Cnan, beta=0.0)
    assert np.all(np.isfinite(e)) and np.all(np.isfinite(o))


def test_leaky_relu_special_cases(oracle_lib):
    M, N, K = 8, 8, 16
    A = inputs.matrix(M, K, 13, 0, "bf16")
    B = inputs.matrix(K, N, 13, 1, "bf16")
    plain, _ = oracle_lib.gemm(M, N, K, A, B)
    assert (plain < 0).any() and (plain > 0).any()
    same, _ = oracle_lib.gemm(M, N, K, A, B, act=1, slope=1.0)
    assert np.array_equal(same, plain)                 # slope 1 is the identity
    relu, _ = oracle_lib.gemm(M, N, K, A, B, act=1, slope=0.0)
    assert np.array_equal(relu, np.where(plain > 0, plain, 0.0) + 0.0 * plain)
    leaky, _ = oracle_lib.gemm(M, N, K, A, B, act=1, slope=0.25)
    pos = plain >= 0
    assert np.array_equal(leaky[pos], plain[pos])      # non-negative values untouched
    assert np.array_equal(leaky[~pos], plain[~pos] * 0.25)  # power-of-two slope: exact
    # the activation comes after alpha and beta: alpha = -1 flips which entries are scaled
    neg, _ = oracle_lib.gemm(M, N, K, A, B, act=1, slope=0.25, alpha=-1.0)
    assert np.array_equal(neg[~pos], -plain[~pos])
    assert np.array_equal(neg[plain > 0], -plain[plain > 0] * 0.25)


def _act_of(oracle_lib, x, act):
    """act(x) through the oracle's epilogue: a 1x1x1 product x * 1 (x exact in bf16)."""
    A = inputs.f32_to_bf16_bits(np.array([[x]], dtype=np.float32))
    B = inputs.f32_to_bf16_bits(np.array([[1.0]], dtype=np.float32))
    e, _ = oracle_lib.gemm(1, 1, 1, A, B, act=act)
    return float(e[0, 0])


# Standard normal distribution function Phi and exp at a few points (printed
# tables of the normal distribution; e^-1, e^-2).
PHI = {0.5: 0.6914624612740131, 1.0: 0.8413447460685429, 2.0: 0.9772498680518208}
EXP_NEG = {1.0: 0.36787944117144233, 2.0: 0.1353352832366127}


def test_relu_gelu_silu_against_tables_and_identities(oracle_lib):
    for x in (-3.0, -1.0, -0.5, 0.0, 0.5, 1.0, 2.0, 3.0):
        assert _act_of(oracle_lib, x, 2) == max(x, 0.0)                      # ReLU
    for x, phi in PHI.items():
        assert abs(_act_of(oracle_lib, x, 3) - x * phi) <= 4e-16            # GELU(x) = x Phi(x)
        assert abs(_act_of(oracle_lib, -x, 3) + x * (1.0 - phi)) <= 4e-16   # Phi(-x) = 1 - Phi(x)
    for x, en in EXP_NEG.items():
        assert abs(_act_of(oracle_lib, x, 4) - x / (1.0 + en)) <= 4e-16     # SiLU(x) = x / (1 + e^-x)
    for act in (3, 4):                                                      # f(x) - f(-x) = x
        for x in (0.25, 0.5, 1.0, 1.5, 2.0, 3.0, 6.0):
            assert abs(_act_of(oracle_lib, x, act) - _act_of(oracle_lib, -x, act) - x) <= 1e-15
        assert _act_of(oracle_lib, 0.0, act) == 0.0


def test_activation_follows_alpha_and_beta(oracle_lib):
    M, N, K = 6, 5, 7
    A = inputs.matrix(M, K, 14, 0, "bf16")
    B = inputs.matrix(K, N, 14, 1, "bf16")
    C = inputs.matrix(M, N, 14, 2, "f32")
    pre, _ = oracle_lib.gemm(M, N, K, A, B, C=C, alpha=-1.5, beta=0.5)
    phi = lambda v: 0.5 * np.vectorize(math.erfc)(-v / math.sqrt(2.0))
    for act, f in ((2, lambda v: np.where(v < 0, 0.0, v)), (3, lambda v: v * phi(v)),
                   (4, lambda v: v / (1.0 + np.exp(-v)))):
        got, _ = oracle_lib.gemm(M, N, K, A, B, C=C, alpha=-1.5, beta=0.5, act=act)
        assert np.allclose(got, f(pre), rtol=1e-15, atol=1e-16)


# ------------------------------------------------------------- brute force

def _exact_product(Ad, Bd, M, N, K):
    Af = [[Fraction(float(Ad[i, k])) for k in range(K)] for i in range(M)]
    Bf = [[Fraction(float(Bd[k, j])) for j in range(N)] for k in range(K)]
    return [[sum((Af[i][k] * Bf[k][j] for k in range(K)), Fraction(0)) for j in range(N)]
            for i in range(M)], Af, Bf


@pytest.mark.parametrize("in_fmt,out_fmt", [("bf16", "f32"), ("bf16", "bf16"), ("f16", "f32"),
                                            ("f16", "f16"), ("tf32", "f32")])
def test_brute_force_exact_rationals(oracle_lib, in_fmt, out_fmt):
    """Every M, N, K in 1..6: oracle vs exact rational arithmetic."""
    u = Fraction(1, 2 ** 53)
    seed = 100
    for M in range(1, 7):
        for N in range(1, 7):
            for K in range(1, 7):
                seed += 1
                ta, tb = bool(seed & 1), bool(seed & 2)
                A = inputs.matrix(M, K, seed, 0, in_fmt)
                B = inputs.matrix(K, N, seed, 1, in_fmt)
                C = inputs.matrix(M, N, seed, 2, out_fmt)
                alpha, beta = [(1.0, 0.0), (0.75, -1.5), (-2.0, 0.5), (1.25, 1.0)][seed % 4]
                Ad, Bd, Cd = dec(A, in_fmt), dec(B, in_fmt), dec(C, out_fmt)
                exact, out = oracle_lib.gemm(M, N, K, stored(A, ta), stored(B, tb), C=C,
                                             alpha=alpha, beta=beta, in_fmt=in_fmt,
                                             out_fmt=out_fmt, transA=ta, transB=tb)
                S, Af, Bf = _exact_product(Ad, Bd, M, N, K)
                for i in range(M):
                    for j in range(N):
                        absum = sum(abs(Af[i][k] * Bf[k][j]) for k in range(K))
                        cterm = Fraction(beta) * Fraction(float(Cd[i, j])) if beta else 0
                        d = Fraction(alpha) * S[i][j] + cterm
                        bound = (K + 3) * u * (abs(Fraction(alpha)) * absum + abs(cterm)) * 2
                        assert abs(Fraction(float(exact[i, j])) - d) <= bound, (M, N, K, i, j)
                        r = round_fraction(d, out_fmt)
                        got = dec(out[i, j], out_fmt)
                        if float(r) != float(got):
                            # only allowed when d sits within the fp64 error of a rounding tie
                            r2 = round_fraction(Fraction(float(exact[i, j])), out_fmt)
                            assert float(r2) == float(got) and bound > 0, (M, N, K, i, j)


# ------------------------------------------------------------ rounding / decoding

def test_tf32_operand_decode(oracle_lib):
    """TF32 (section 2.2, Table 1): sign, 8-bit exponent, 10 fraction bits of
    an fp32 word.  Words with low bits set lose them toward zero: 1 + 2^-11 +
    2^-12 gives 1.0 (nearest rounding would give 1 + 2^-10)."""
    cases = {0x3F802000: 1.0 + 2.0 ** -10, 0x3F801000: 1.0, 0x3F801800: 1.0, 0x3F803000: 1.0 + 2.0 ** -10,
             0xBF803000: -(1.0 + 2.0 ** -10), 0x3FFFE000: 2.0 - 2.0 ** -10, 0x3FFFFFFF: 2.0 - 2.0 ** -10,
             0x40490FDB: 3.140625, 0x00800000: 2.0 ** -126, 0x00000000: 0.0, 0x80000000: -0.0}
    for bits, v in cases.items():
        got = oracle_lib.decode(bits, "tf32")
        assert got == v and math.copysign(1.0, got) == math.copysign(1.0, v), hex(bits)
    # products of two TF32 values (11 significant bits each) are exact in fp32
    rng = np.random.default_rng(5)
    a = dec(rng.uniform(-4, 4, 10000).astype(np.float32), "tf32")
    b = dec(rng.uniform(-4, 4, 10000).astype(np.float32), "tf32")
    assert np.array_equal((a.astype(np.float32) * b.astype(np.float32)).astype(np.float64), a * b)


def test_decode_all_patterns(oracle_lib):
    for fmt in ("bf16", "f16"):
        bits = np.arange(65536, dtype=np.uint32)
        ref = dec(bits.astype(np.uint16), fmt)
        step = 1 if fmt == "f16" else 7   # bf16: a stride keeps the ctypes loop short
        for b in range(0, 65536, step):
            got = oracle_lib.decode(b, fmt)
            r = ref[b]
            assert (np.isnan(got) and np.isnan(r)) or got == r, (fmt, hex(b))


def test_round_bf16_ties_and_neighbours(oracle_lib):
    """Midpoints between adjacent bf16 values go to the even one; anything
    strictly nearer one side goes there (exhaustive over positive finite bf16)."""
    vals = dec(np.arange(0, 0x7F80, dtype=np.uint16), "bf16")   # 0 .. largest finite
    for b in range(0, 0x7F7F, 5):
        lo, hi = vals[b], vals[b + 1]
        mid = (lo + hi) / 2                                     # exact in fp64
        want = b if b % 2 == 0 else b + 1
        assert oracle_lib.round_bf16(mid) == want
        assert oracle_lib.round_bf16(np.nextafter(mid, np.inf)) == b + 1
        assert oracle_lib.round_bf16(np.nextafter(mid, -np.inf)) == b
        assert oracle_lib.round_bf16(-mid) == (want | 0x8000)
    top = float(vals[0x7F7F])
    half_ulp = 2.0 ** (127 - 8)
    assert oracle_lib.round_bf16(top + half_ulp) == 0x7F80      # tie to even overflows
    assert oracle_lib.round_bf16(top + half_ulp * 0.99) == 0x7F7F
    assert oracle_lib.round_bf16(-0.0) == 0x8000
    assert oracle_lib.round_bf16(float("nan")) & 0x7F80 == 0x7F80


def test_round_against_exact_rationals_and_numpy(oracle_lib):
    rng = np.random.default_rng(7)
    xs = rng.standard_normal(3000) * np.exp2(rng.integers(-140, 130, 3000))
    xs = np.concatenate([xs, [65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                              2.0 ** -133, 2.0 ** -134, 1.5 * 2.0 ** -134, 1 + 2.0 ** -8,
                              1 + 3 * 2.0 ** -9, 1 + 2.0 ** -11, 1 + 2.0 ** -24]])
    for x in xs:
        x = float(x)
        rb = round_fraction(Fraction(x), "bf16")
        assert dec(np.uint16(oracle_lib.round_bf16(x)), "bf16") == float(rb), x
        rh = oracle_lib.round_f16(x)
        assert rh == int(np.float16(x).view(np.uint16)), x        # numpy: correctly rounded
        assert dec(np.uint16(rh), "f16") == float(round_fraction(Fraction(x), "f16")), x
        assert oracle_lib.round_f32(x) == float(np.float32(x)), x


def test_sample_matches_full(oracle_lib):
    M, N, K = 9, 7, 33
    A = inputs.matrix(M, K, 77, 0, "bf16")
    B = inputs.matrix(N, K, 77, 1, "bf16")
    C = inputs.matrix(M, N, 77, 2, "f32")
    e, o = oracle_lib.gemm(M, N, K, A, B, C=C, beta=0.5, transB=True, act=1, slope=0.01,
                           out_fmt="bf16")
    rows = np.array([0, 8, 3, 8, 0])
    cols = np.array([0, 6, 2, 0, 6])
    es, os_ = oracle_lib.sample(rows, cols, K, A, B, C=C, beta=0.5, transB=True, act=1,
                                slope=0.01, out_fmt="bf16")
    assert np.array_equal(es, e[rows, cols]) and np.array_equal(os_, o[rows, cols])


def test_k_zero_is_beta_c(oracle_lib):
    M, N = 3, 4
    A = np.zeros((M, 1), dtype=np.uint16)
    B = np.zeros((1, N), dtype=np.uint16)
    C = inputs.matrix(M, N, 3, 2, "f32")
    e, _ = oracle_lib.gemm(M, N, 0, A, B, C=C, alpha=1.0, beta=0.5)
    assert np.array_equal(e, 0.5 * C.astype(np.float64))
