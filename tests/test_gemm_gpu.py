"""GPU parity tests: the CUDA path through the C ABI against the CPU oracle.

Small and medium shapes are compared in full; the full-size workloads of the
benchmark configurations are compared on 4096 sampled outputs (corners, last
row and column, tile boundaries and random entries) recomputed one by one by
the oracle.  Tolerance: see tests/gemm_case.py.
"""
import os

import numpy as np
import pytest

from tests.gemm_case import run_case, run_case_ex

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def plan():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from dense_gemm_mma_gb300 import gemm
    p = gemm.Plan(0)
    yield p
    p.close()


# ------------------------------------------------------------------ basics

def test_watchdog_selftest_returns_and_context_survives(plan):
    from dense_gemm_mma_gb300 import gemm
    assert gemm.gemm_plan_set_watchdog(plan.handle, 50_000_000) == gemm.GEMM_OK
    assert gemm.gemm_plan_selftest_watchdog(plan.handle, None) == gemm.GEMM_ERR_TIMEOUT
    assert gemm.gemm_plan_set_watchdog(plan.handle, 2_000_000_000) == gemm.GEMM_OK
    assert plan.poll_error() == gemm.GEMM_OK        # cleared by the self-test's poll
    run_case(plan, 128, 64, 64, env={"GEMM_FORCE_TILE": "128x64"})


@pytest.mark.parametrize("bn", [64, 128, 256])
def test_single_tile_single_kblock(plan, bn):
    r = run_case(plan, 128, bn, 64, env={"GEMM_FORCE_TILE": f"128x{bn}"})
    assert r.info["path"] == "tc" and r.info["tile_n"] == bn and r.info["tiles"] == 1


def test_config1_512_cubed(plan):
    r = run_case(plan, 512, 512, 512, seed=1234)
    assert r.info["path"] in ("tc", "tc_splitk")


@pytest.mark.parametrize("bn", [64, 128, 256])
@pytest.mark.parametrize("shape", [(300, 520, 200), (129, 257, 1000), (640, 384, 77)])
def test_tile_widths_ragged(plan, bn, shape):
    r = run_case(plan, *shape, env={"GEMM_FORCE_TILE": f"128x{bn}"}, seed=sum(shape) + bn)
    assert r.info["tile_n"] == bn


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
@pytest.mark.parametrize("ta", [False, True])
@pytest.mark.parametrize("tb", [False, True])
def test_transpose_flags(plan, fmt, ta, tb):
    run_case(plan, 200, 300, 136, in_fmt=fmt, ta=ta, tb=tb, seed=5 + 2 * ta + tb)


@pytest.mark.parametrize("in_fmt,out_fmt", [("bf16", "bf16"), ("f16", "f16"), ("f16", "f32"),
                                            ("bf16", "f32")])
def test_dtypes(plan, in_fmt, out_fmt):
    run_case(plan, 257, 200, 513, in_fmt=in_fmt, out_fmt=out_fmt, seed=17)


@pytest.mark.parametrize("out_fmt", ["f32", "bf16", "f16"])
def test_beta_alpha_leaky_relu(plan, out_fmt):
    in_fmt = "f16" if out_fmt == "f16" else "bf16"
    run_case(plan, 260, 390, 300, in_fmt=in_fmt, out_fmt=out_fmt, alpha=1.0, beta=0.5, act=1,
             slope=0.01, seed=31)
    run_case(plan, 130, 200, 96, in_fmt=in_fmt, out_fmt=out_fmt, alpha=-2.5, beta=-1.0, seed=32)
    run_case(plan, 130, 200, 96, in_fmt=in_fmt, out_fmt=out_fmt, alpha=0.75, act=1, slope=0.2,
             seed=33, ta=True)


def test_alpha_zero_and_k_zero_scale_c(plan):
    r = run_case(plan, 100, 70, 50, alpha=0.0, beta=0.5, act=1, slope=0.25, seed=41)
    assert r.info["path"] == "scale"
    r = run_case(plan, 100, 70, 0, beta=2.0, seed=42)
    assert r.info["path"] == "scale"
    r = run_case(plan, 100, 70, 0, beta=0.0, seed=43)            # C <- 0 without reading C
    assert r.info["path"] == "scale"


@pytest.mark.parametrize("ta,tb", [(False, False), (True, True)])
def test_leading_dimension_padding(plan, ta, tb):
    run_case(plan, 200, 136, 264, ta=ta, tb=tb, pad=(8, 24, 4), seed=51)
    run_case(plan, 200, 136, 264, out_fmt="bf16", ta=ta, tb=tb, pad=(16, 8, 8), seed=52)


EDGE = [1, 7, 8, 15, 16, 17, 127, 128, 129, 255, 257]


@pytest.mark.parametrize("M", EDGE)
def test_edge_shapes_m_by_n(plan, M):
    for N in EDGE:
        run_case(plan, M, N, 129, seed=1000 + M * 7 + N)


def test_edge_shapes_k(plan):
    for K in [1, 2, 7, 8, 15, 16, 17, 63, 64, 65, 127, 128, 129, 255, 257]:
        run_case(plan, 129, 257, K, seed=2000 + K)
        run_case(plan, 129, 257, K, ta=True, tb=True, seed=3000 + K)


@pytest.mark.parametrize("out_fmt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", [2, 3, 9, 257, 258, 263])
def test_unaligned_row_tail_of_c(plan, out_fmt, N):
    """Rows of C whose byte length is not a multiple of 16: the last partial
    16-byte piece is written by the kernel's threads, never by a TMA store, so
    the ld padding next to it keeps its sentinel."""
    in_fmt = "f16" if out_fmt == "f16" else "bf16"
    run_case(plan, 130, N, 200, in_fmt=in_fmt, out_fmt=out_fmt, seed=N, pad=(0, 0, 8))
    run_case(plan, 130, N, 200, in_fmt=in_fmt, out_fmt=out_fmt, beta=0.5, act=1, slope=0.1,
             seed=N + 1, pad=(0, 0, 8))


# ------------------------------------------------------------------- CTA pair

@pytest.mark.parametrize("shape", [(256, 256, 64), (300, 520, 200), (129, 257, 1000), (640, 384, 77),
                                   (513, 129, 300), (2, 3, 5)])
def test_cta_pair_ragged(plan, shape):
    r = run_case(plan, *shape, env={"GEMM_FORCE_TILE": "256x256"}, seed=sum(shape) + 1)
    assert r.info["tile_m"] == 256 and r.info["cta_per_tile"] == 2 and r.info["grid"] % 2 == 0


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
@pytest.mark.parametrize("ta,tb", [(False, False), (False, True), (True, False), (True, True)])
def test_cta_pair_transposes(plan, fmt, ta, tb):
    run_case(plan, 300, 384, 200, in_fmt=fmt, ta=ta, tb=tb, env={"GEMM_FORCE_TILE": "256x256"}, seed=11)


@pytest.mark.parametrize("out_fmt", ["f32", "bf16", "f16"])
def test_cta_pair_epilogues_and_tails(plan, out_fmt):
    in_fmt = "f16" if out_fmt == "f16" else "bf16"
    env = {"GEMM_FORCE_TILE": "256x256"}
    run_case(plan, 257, 300, 513, in_fmt=in_fmt, out_fmt=out_fmt, beta=0.5, act=1, slope=0.1, env=env, seed=12)
    run_case(plan, 260, 257, 129, in_fmt=in_fmt, out_fmt=out_fmt, alpha=-2.0, env=env, seed=13, pad=(0, 0, 8))


def test_cta_pair_splitk_deterministic(plan):
    r = run_case(plan, 512, 512, 4096, env={"GEMM_FORCE_TILE": "256x256", "GEMM_FORCE_SPLITK": "3"},
                 repeat=2, seed=14)
    assert r.info["splitk"] == 3 and r.info["cta_per_tile"] == 2
    assert np.array_equal(r.outputs[0].view(np.uint8), r.outputs[1].view(np.uint8))


# -------------------------------------------------------------------- split-K

@pytest.mark.parametrize("splits", [2, 3, 7])
def test_splitk_forced_and_deterministic(plan, splits):
    r = run_case(plan, 256, 256, 4096, env={"GEMM_FORCE_SPLITK": str(splits), "GEMM_SPLITK_CLUSTER": "0"},
                 repeat=2, seed=60)
    assert r.info["path"] == "tc_splitk" and r.info["splitk"] == splits
    assert np.array_equal(r.outputs[0].view(np.uint8), r.outputs[1].view(np.uint8))


FUSED_CASES = [
    ("128x128", (256, 256, 4096), {"GEMM_FORCE_SPLITK": "7", "GEMM_SPLITK_CLUSTER": "0"}, "f32"),
    ("128x64", (300, 200, 3000), {"GEMM_FORCE_SPLITK": "5", "GEMM_SPLITK_CLUSTER": "0"}, "bf16"),
    ("256x256", (512, 520, 4096), {"GEMM_FORCE_SPLITK": "3"}, "f32"),
    ("128x256", (2600, 2000, 330), {"GEMM_TAIL_SPLIT": "3"}, "bf16"),
    ("256x256", (2600, 2000, 260), {"GEMM_TAIL_SPLIT": "3"}, "f32"),
]


@pytest.mark.parametrize("tile,shape,env,out_fmt", FUSED_CASES,
                         ids=[f"{c[0]}_{'x'.join(map(str, c[1]))}" for c in FUSED_CASES])
def test_fused_reduction_bitwise_equals_reduction_kernel(plan, tile, shape, env, out_fmt):
    """With GEMM_FUSED_REDUCE=1, K slices that all run at once are summed
    inside the GEMM kernel: each CTA publishes its slice's partials, waits for
    the tile's other slices and sums its share of the tile over the slices in
    order.  The tile reduction kernel (the default) sums the same partials in
    the same order with the same epilogue, so the two agree bit for bit; both
    match the oracle and repeat bit for bit (the arrival counters are back at
    zero after a call)."""
    env = {**env, "GEMM_FORCE_TILE": tile}
    kw = dict(beta=0.5, act=1, slope=0.2, out_fmt=out_fmt, seed=90 + shape[2] % 7, pad=(0, 0, 8))
    a = run_case(plan, *shape, env={**env, "GEMM_FUSED_REDUCE": "1"}, repeat=3, **kw)
    b = run_case(plan, *shape, env=env, **kw)
    assert a.info["launches"] == 1 and b.info["launches"] == 2
    assert a.info["path"] == b.info["path"] and a.info["path"] in ("tc_splitk", "tc_tail_split")
    for out in a.outputs[1:] + b.outputs:
        assert np.array_equal(a.outputs[0].view(np.uint8), out.view(np.uint8))


# ------------------------------------------------------ further activations

ACTS = {"relu": 2, "gelu": 3, "silu": 4}


@pytest.mark.parametrize("act", sorted(ACTS))
@pytest.mark.parametrize("out_fmt", ["f32", "bf16"])
def test_activations_every_path(plan, act, out_fmt):
    """Each activation on every kernel that applies an epilogue: one-CTA tiles,
    the CTA pair, the K pair, tail and full split-K (reduction kernel), the
    GEMV kernels and the scale path."""
    a = ACTS[act]
    kw = dict(out_fmt=out_fmt, act=a, alpha=1.5, beta=-0.5, seed=100 + a)
    run_case(plan, 300, 520, 200, env={"GEMM_FORCE_TILE": "128x128", "GEMM_FORCE_SPLITK": "1"}, **kw)
    run_case(plan, 257, 300, 513, env={"GEMM_FORCE_TILE": "256x256"}, **kw)
    run_case(plan, 384, 260, 1000, env={"GEMM_SPLITK_CLUSTER": "1", "GEMM_FORCE_SPLITK": "2"}, **kw)
    run_case(plan, 1300, 2000, 333, env={"GEMM_TAIL_SPLIT": "3", "GEMM_FORCE_TILE": "128x128"}, **kw)
    run_case(plan, 200, 150, 3000, env={"GEMM_FORCE_SPLITK": "5", "GEMM_SPLITK_CLUSTER": "0"}, **kw)
    run_case(plan, 1, 4100, 2000, **kw)               # column-stream GEMV
    run_case(plan, 3000, 1, 2000, **kw)               # row-dot GEMV
    run_case(plan, 64, 80, 0, **kw)                   # K = 0: act(beta * C)


# ------------------------------------------------ separate C and D (run_ex)

@pytest.mark.parametrize("c_fmt,d_fmt", [("f32", "bf16"), ("bf16", "f32"), ("f16", "bf16"), ("f32", "f32")])
def test_separate_c_d_every_path(plan, c_fmt, d_fmt):
    """D <- act(alpha AB + beta C) with C kept apart, on every path that reads
    C: one-CTA tiles, the CTA pair, the K pair, the tail split and split-K
    (tile reduction), both GEMV kernels and the K = 0 scale path.  Odd ldc
    (a separate C needs no 16-byte rows), ragged shapes."""
    kw = dict(c_fmt=c_fmt, d_fmt=d_fmt, alpha=1.25, beta=-0.75, act=1, slope=0.2, seed=120, pad=(0, 0, 3, 8))
    run_case_ex(plan, 300, 520, 200, env={"GEMM_FORCE_TILE": "128x128", "GEMM_FORCE_SPLITK": "1"}, **kw)
    run_case_ex(plan, 257, 300, 513, env={"GEMM_FORCE_TILE": "256x256"}, **kw)
    run_case_ex(plan, 384, 260, 1000, env={"GEMM_SPLITK_CLUSTER": "1", "GEMM_FORCE_SPLITK": "2"}, **kw)
    run_case_ex(plan, 1300, 2000, 333, env={"GEMM_TAIL_SPLIT": "3", "GEMM_FORCE_TILE": "128x128"}, **kw)
    run_case_ex(plan, 200, 150, 3000, env={"GEMM_FORCE_SPLITK": "5", "GEMM_SPLITK_CLUSTER": "0"}, **kw)
    run_case_ex(plan, 1, 4100, 2000, **kw)
    run_case_ex(plan, 3000, 1, 2000, **kw)
    run_case_ex(plan, 64, 80, 0, **kw)


def test_separate_c_d_config3_alternative_reading(plan):
    """Config 3's second run read the other way: fp32 C (beta 0.5) in, bf16 D
    out, LeakyReLU 0.01, at the full 8192^3 size on 4096 sampled outputs."""
    r = run_case_ex(plan, 8192, 8192, 8192, c_fmt="f32", d_fmt="bf16", beta=0.5, act=1, slope=0.01,
                    seed=1236, sample=4096)
    assert r.info["cta_per_tile"] == 2


def test_separate_c_d_beta_zero_without_c(plan):
    run_case_ex(plan, 260, 300, 400, c_fmt="f32", d_fmt="bf16", beta=0.0, c_none=True, seed=121)


# ------------------------------------------------------------ input slices

def test_input_slices_through_strides(plan):
    """Slicing fused into the product: A, B and C are row/column slices of
    larger tensors, passed as a pointer into the parent plus its row stride
    (torch views through Plan.run), on the tensor-core, K-pair and GEMV paths;
    the parents' elements outside the slices hold NaN and are neither read
    nor written."""
    import torch
    import oracle
    from dense_gemm_mma_gb300 import inputs
    from tests.gemm_case import decode, from_device, to_device

    def parent(rows, cols, tid, fmt, seed):
        cols = -(-cols // 8) * 8                      # rows of 16-byte multiples (the ld rule)
        X = inputs.matrix(rows, cols, seed, tid, fmt)
        return X, to_device(X, fmt)

    for (M, N, K, r0, c0, env) in [(300, 200, 500, 7, 24, {}),
                                   (1024, 128, 2048, 3, 16, {"GEMM_SPLITK_CLUSTER": "1", "GEMM_FORCE_SPLITK": "2"}),
                                   (1, 3000, 1000, 5, 8, {})]:
        seed = 130 + M
        Ap, Apd = parent(M + r0 + 9, K + c0 + 40, 0, "bf16", seed)
        Bp, Bpd = parent(K + r0 + 5, N + c0 + 24, 1, "bf16", seed)
        Cp = np.full((M + r0 + 3, -(-(N + c0 + 12) // 4) * 4), np.nan, dtype=np.float32)
        Cpd = to_device(Cp, "f32")
        A = Ap[r0:r0 + M, c0:c0 + K]
        B = Bp[r0:r0 + K, c0:c0 + N]
        # NaN around the slices of A and B: any read outside them would poison a result
        Apd[:r0] = float("nan"); Apd[r0 + M:] = float("nan"); Apd[:, :c0] = float("nan"); Apd[:, c0 + K:] = float("nan")
        Bpd[:r0] = float("nan"); Bpd[r0 + K:] = float("nan"); Bpd[:, :c0] = float("nan"); Bpd[:, c0 + N:] = float("nan")
        old = {k: os.environ.get(k) for k in env}
        os.environ.update(env)
        try:
            st = plan.run(Apd[r0:r0 + M, c0:c0 + K], Bpd[r0:r0 + K, c0:c0 + N], Cpd[r0:r0 + M, c0:c0 + N])
        finally:
            for k, v in old.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        assert st == 0
        torch.cuda.synchronize()
        out = from_device(Cpd, "f32")
        inside = np.zeros(out.shape, dtype=bool)
        inside[r0:r0 + M, c0:c0 + N] = True
        assert np.isnan(out[~inside]).all()                   # nothing written outside the slice of C
        exact, _ = oracle.gemm(M, N, K, np.ascontiguousarray(A), np.ascontiguousarray(B))
        amax = np.abs(decode(A, "bf16")).max()
        bmax = np.abs(decode(B, "bf16")).max()
        got = out[r0:r0 + M, c0:c0 + N].astype(np.float64)
        assert np.all(np.abs(got - exact) <= 1e-5 * K * amax * bmax + 2.0 ** -21 * np.abs(exact)), (M, N, K)


# --------------------------------------------------------------------- TF32

@pytest.mark.parametrize("ta,tb", [(False, True), (False, False), (True, True), (True, False)])
def test_tf32_layouts_ragged(plan, ta, tb):
    """TF32 operands (fp32 words, low 13 fraction bits dropped) in every
    layout; M/N-major operands are read by the MMAs where they are stored
    (tiles swizzled in 32-byte units), so one launch unless K is split; with
    GEMM_TF32_TRANSPOSE=1 they are first copied K-major into workspace."""
    r = run_case(plan, 300, 520, 333, in_fmt="tf32", ta=ta, tb=tb, seed=140 + 2 * ta + tb)
    assert r.info["tile_k"] == 32
    assert r.info["launches"] == (2 if r.info["path"] in ("tc_splitk", "tc_tail_split") else 1)
    if ta or not tb:
        r2 = run_case(plan, 300, 520, 333, in_fmt="tf32", ta=ta, tb=tb, seed=140 + 2 * ta + tb,
                      env={"GEMM_TF32_TRANSPOSE": "1"})
        assert r2.info["launches"] == r.info["launches"] + int(ta) + int(not tb)


@pytest.mark.parametrize("M,N,K,copies", [(4096, 4096, 4096, 1), (8192, 128, 8192, 1), (600, 520, 700, 0)])
def test_tf32_mn_major_operands_copied_only_where_it_pays(plan, M, N, K, copies):
    """Both operands M/N-major (A stored K x M, B stored K x N): the MMAs read
    them in place unless the estimated slowdown exceeds a copy; on 4096^3 the
    estimate copies one operand, on 8192 x 128 x 8192 the small B (4 MB) and
    reads the 268 MB A in place, and a small call copies nothing."""
    r = run_case(plan, M, N, K, in_fmt="tf32", ta=True, tb=False, seed=155, sample=None if M * N < 10 ** 6 else 2048)
    base = 2 if r.info["path"] in ("tc_splitk", "tc_tail_split") else 1
    assert r.info["launches"] - base == copies, r.info


@pytest.mark.parametrize("ta,tb", [(False, True), (True, False)])
def test_tf32_tile_widths_pair_kpair_splits(plan, ta, tb):
    """Every tile mode with K-major TF32 operands and with both operands
    M/N-major (A stored K x M, B stored K x N: four 32-element boxes per
    128-row panel, swizzled in 32-byte units)."""
    envs = [{"GEMM_FORCE_TILE": "128x64"}, {"GEMM_FORCE_TILE": "128x128"}, {"GEMM_FORCE_TILE": "128x256"},
            {"GEMM_FORCE_TILE": "256x256"}, {"GEMM_SPLITK_CLUSTER": "1", "GEMM_FORCE_SPLITK": "2"},
            {"GEMM_FORCE_SPLITK": "5", "GEMM_SPLITK_CLUSTER": "0"},
            {"GEMM_TAIL_SPLIT": "3", "GEMM_FORCE_TILE": "128x128"}]
    for env in envs:
        M, N = (1300, 2000) if "GEMM_TAIL_SPLIT" in env else (257, 300)
        run_case(plan, M, N, 515, in_fmt="tf32", ta=ta, tb=tb, beta=0.5, act=1, slope=0.1, env=env,
                 seed=150 + ta)


def test_tf32_gemv_shapes_and_edges(plan):
    run_case(plan, 1, 3000, 1000, in_fmt="tf32", seed=160)            # M = 1 on the tensor cores
    run_case(plan, 3000, 1, 1000, in_fmt="tf32", tb=True, seed=161)   # N = 1
    run_case(plan, 200, 3, 300, in_fmt="tf32", tb=True, beta=1.0, seed=162, pad=(0, 0, 1))  # N < 4, odd ldc
    run_case(plan, 129, 257, 7, in_fmt="tf32", seed=163)              # K < 32: one partial k-block


def test_tf32_drops_the_low_fraction_bits(plan):
    """Every A entry is the fp32 word 1 + 2^-11 + 2^-12, every B entry 1: with
    the 13 low fraction bits dropped each product is 1 and every output is
    exactly K; rounding to 10 bits would give K * (1 + 2^-10)."""
    torch = pytest.importorskip("torch")
    from dense_gemm_mma_gb300 import gemm
    M, N, K = 256, 256, 1024
    A = torch.full((M, K), 1.0 + 2.0 ** -11 + 2.0 ** -12, device="cuda", dtype=torch.float32)
    B = torch.ones(N, K, device="cuda", dtype=torch.float32)
    C = torch.zeros(M, N, device="cuda", dtype=torch.float32)
    assert plan.run(A, B, C, transB=True) == gemm.GEMM_OK
    torch.cuda.synchronize()
    assert torch.all(C == float(K)).item()


def test_tf32_with_separate_c_and_benchmark_mode():
    """TF32 operands through gemm_run_ex (bf16 C in, fp32 D out, A stored
    K x M and B stored K x N) and under benchmark mode."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_mma_gb300 import gemm
    p = gemm.Plan(0)
    try:
        run_case_ex(p, 300, 260, 515, in_fmt="tf32", c_fmt="bf16", d_fmt="f32", beta=0.5, act=3, seed=170,
                    ta=True, pad=(0, 0, 1, 4))
        assert gemm.gemm_plan_set_autotune(p.handle, True) == gemm.GEMM_OK
        r = run_case(p, 1300, 1000, 700, in_fmt="tf32", beta=-1.0, seed=171)
        assert gemm.gemm_plan_tuned_count(p.handle) == 1 and r.info["tile_k"] == 32
    finally:
        p.close()


def test_tf32_full_size_sampled(plan):
    r = run_case(plan, 8192, 8192, 8192, in_fmt="tf32", tb=True, sample=4096, seed=1236)
    assert r.info["tile_k"] == 32


# ------------------------------------------- split-K reduced on chip (K pair)

KPAIR = {"GEMM_SPLITK_CLUSTER": "1", "GEMM_FORCE_SPLITK": "2"}


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("shape", [(300, 520, 1000), (129, 257, 130), (640, 384, 65), (128, 128, 128)])
def test_kpair_ragged(plan, bn, shape):
    r = run_case(plan, *shape, env={**KPAIR, "GEMM_FORCE_TILE": f"128x{bn}"}, seed=sum(shape) + bn + 1)
    assert r.info["path"] == "tc_splitk_cluster" and r.info["tile_n"] == bn
    assert r.info["splitk"] == 2 and r.info["cta_per_tile"] == 2 and r.info["launches"] == 1
    assert r.info["workspace_bytes"] == 0


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("out_fmt", ["f32", "bf16", "f16"])
def test_kpair_epilogues_transposes_and_tails(plan, bn, out_fmt):
    in_fmt = "f16" if out_fmt == "f16" else "bf16"
    env = {**KPAIR, "GEMM_FORCE_TILE": f"128x{bn}"}
    # beta and LeakyReLU; N not a multiple of 16 bytes of C (thread-written tail)
    run_case(plan, 257, 300, 513, in_fmt=in_fmt, out_fmt=out_fmt, beta=0.5, act=1, slope=0.1, env=env,
             seed=70 + bn)
    run_case(plan, 260, 203, 777, in_fmt=in_fmt, out_fmt=out_fmt, alpha=-2.0, beta=-1.0, ta=True, tb=True,
             env=env, seed=71 + bn, pad=(8, 16, 8))
    run_case(plan, 130, 129, 200, in_fmt=in_fmt, out_fmt=out_fmt, ta=True, env=env, seed=72 + bn)
    run_case(plan, 200, 136, 300, in_fmt=in_fmt, out_fmt=out_fmt, tb=True, env=env, seed=73 + bn)


@pytest.mark.parametrize("bn", [128, 256])
def test_kpair_many_tiles_per_cluster(plan, bn):
    """More tiles than resident clusters: each cluster walks several tiles, so
    both tensor-memory accumulators and every exchange-barrier phase turn over."""
    r = run_case(plan, 4100, 1030, 700, env={**KPAIR, "GEMM_FORCE_TILE": f"128x{bn}"}, seed=74 + bn,
                 sample=4096, out_fmt="bf16", beta=0.25)
    assert r.info["tiles"] > r.info["grid"]


@pytest.mark.parametrize("bn", [128, 256])
def test_kpair_bitwise_equals_two_slice_reduction(plan, bn):
    """Both forms add the same two fp32 slices once and apply the same
    epilogue, so their outputs agree bit for bit, and repeat bit for bit."""
    env = {"GEMM_FORCE_SPLITK": "2", "GEMM_FORCE_TILE": f"128x{bn}"}
    a = run_case(plan, 384, 520, 3000, env={**env, "GEMM_SPLITK_CLUSTER": "1"}, beta=0.5, act=1, slope=0.2,
                 repeat=2, seed=75)
    b = run_case(plan, 384, 520, 3000, env={**env, "GEMM_SPLITK_CLUSTER": "0"}, beta=0.5, act=1, slope=0.2,
                 seed=75)
    assert a.info["path"] == "tc_splitk_cluster" and b.info["path"] == "tc_splitk"
    assert np.array_equal(a.outputs[0].view(np.uint8), a.outputs[1].view(np.uint8))
    assert np.array_equal(a.outputs[0].view(np.uint8), b.outputs[0].view(np.uint8))


def test_kpair_plan_cache_and_watchdog_clear(plan):
    r = run_case(plan, 1024, 128, 8192, env=KPAIR, repeat=3, seed=76)
    assert r.info["path"] == "tc_splitk_cluster"
    assert plan.poll_error() == 0


# ------------------------------------------------ tail-wave split (hybrid)

@pytest.mark.parametrize("tile,shape", [("128x64", (1300, 1000, 300)), ("128x128", (1300, 2000, 333)),
                                        ("128x256", (2600, 2000, 330)), ("256x256", (2600, 2000, 260))])
def test_tail_split_ragged(plan, tile, shape):
    """More tiles than one wave, the last wave partly filled: whole tiles for
    the first wave, K slices for the rest, reduced by the tile reduction."""
    r = run_case(plan, *shape, env={"GEMM_TAIL_SPLIT": "3", "GEMM_FORCE_TILE": tile}, seed=80 + len(tile))
    i = r.info
    assert i["path"] == "tc_tail_split" and i["splitk"] == 3 and 0 < i["tail_tiles"] < i["tiles"]
    assert i["units"] == i["tiles"] - i["tail_tiles"] + 3 * i["tail_tiles"] and i["launches"] == 2


@pytest.mark.parametrize("out_fmt", ["f32", "bf16", "f16"])
def test_tail_split_epilogues_and_transposes(plan, out_fmt):
    in_fmt = "f16" if out_fmt == "f16" else "bf16"
    env = {"GEMM_TAIL_SPLIT": "2", "GEMM_FORCE_TILE": "128x128"}
    run_case(plan, 1290, 2003, 515, in_fmt=in_fmt, out_fmt=out_fmt, beta=0.5, act=1, slope=0.1,
             ta=True, env=env, seed=82, pad=(8, 0, 8))
    run_case(plan, 1301, 1930, 200, in_fmt=in_fmt, out_fmt=out_fmt, alpha=-1.5, tb=True, env=env, seed=83)


def test_tail_split_deterministic_and_pair(plan):
    r = run_case(plan, 2600, 2000, 640, env={"GEMM_TAIL_SPLIT": "5", "GEMM_FORCE_TILE": "256x256"},
                 repeat=2, seed=84, beta=1.0, out_fmt="bf16")
    assert r.info["path"] == "tc_tail_split" and r.info["cta_per_tile"] == 2
    assert np.array_equal(r.outputs[0].view(np.uint8), r.outputs[1].view(np.uint8))


def test_tail_split_planner_choice_wave_shape(plan):
    """2304 x 2176 x 4096 fp16: 81 pair tiles on 76 pairs; the planner splits the 5 tail tiles."""
    r = run_case(plan, 2304, 2176, 4096, in_fmt="f16", sample=4096, seed=1238)
    assert r.info["path"] == "tc_tail_split" and r.info["tail_tiles"] == 5


# ------------------------------------------------------------ CUDA graphs

def test_cuda_graph_capture_and_replay(plan):
    """A sequence of calls (K pair, tail split, pair tile, GEMV, TF32 with a
    transpose) captured into one CUDA graph after a warm-up call of each, then
    replayed on new input values: results match eager calls bit for bit."""
    torch = pytest.importorskip("torch")
    from dense_gemm_mma_gb300 import gemm
    g = torch.Generator(device="cuda").manual_seed(5)
    shapes = [(8192, 128, 2048, torch.bfloat16, True), (1300, 2000, 512, torch.bfloat16, False),
              (1024, 1024, 1024, torch.float16, False), (1, 4096, 2048, torch.bfloat16, False),
              (300, 264, 320, torch.float32, False)]
    bufs = []
    for M, N, K, dt, tb in shapes:
        A = torch.empty(M, K, device="cuda", dtype=dt)
        B = torch.empty((N, K) if tb else (K, N), device="cuda", dtype=dt)
        bufs.append((A, B, torch.zeros(M, N, device="cuda"), tb))

    def fill():
        for A, B, C, _ in bufs:
            A.copy_(torch.randn(A.shape, device="cuda", generator=g))
            B.copy_(torch.randn(B.shape, device="cuda", generator=g))

    def run_all():
        for A, B, C, tb in bufs:
            assert plan.run(A, B, C, transB=tb) == gemm.GEMM_OK

    fill()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        run_all()                      # warm-up: plans, descriptors and workspace exist
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        run_all()
    fill()                             # new values in the same buffers
    graph.replay()
    torch.cuda.synchronize()
    replayed = [C.clone() for _, _, C, _ in bufs]
    with torch.cuda.stream(stream):
        run_all()
    torch.cuda.synchronize()
    for (_, _, C, _), R in zip(bufs, replayed):
        assert torch.equal(C, R)
    assert plan.poll_error() == gemm.GEMM_OK


def test_plain_launches_without_programmatic_dependence(monkeypatch):
    """A plan created with GEMM_PDL=0 launches every kernel plainly (no
    programmatic stream serialization); each path still matches the oracle."""
    torch = pytest.importorskip("torch")
    from dense_gemm_mma_gb300 import gemm
    monkeypatch.setenv("GEMM_PDL", "0")
    p = gemm.Plan(0)
    try:
        cases = [((1024, 1024, 1024), {}, "tc_splitk_cluster"),
                 ((2304, 2176, 4096), {}, "tc_tail_split"),
                 ((256, 256, 8192), {"GEMM_FORCE_SPLITK": "8", "GEMM_SPLITK_CLUSTER": "0"}, "tc_splitk"),
                 ((300, 520, 200), {}, None),
                 ((1, 4096, 2048), {}, "gemv_colstream")]
        for (M, N, K), env, path in cases:
            r = run_case(p, M, N, K, env=env, sample=2048 if M * N > 2_000_000 else None,
                         in_fmt="f16" if M == 2304 else "bf16")
            if path:
                assert r.info["path"] == path, (M, N, K, r.info["path"])
        r = run_case(p, 1, 4096, 2048, tb=True)
        assert r.info["path"] == "gemv_rowdot"
    finally:
        p.close()


@pytest.mark.parametrize("first,second", [((8192, 128, 2048), (8192, 128, 64)),     # K pair -> tile
                                          ((1, 4096, 2048), (1, 4096, 512)),        # GEMV -> GEMV
                                          ((2304, 2176, 512), (2304, 2176, 4096))])  # pair tile -> tail split
def test_back_to_back_beta_reads_the_previous_output(plan, first, second):
    """A call that reads C (beta = 1) right after the call that wrote it, with
    no synchronisation between them: its result matches the oracle applied to
    the first call's output (the first call is deterministic, so running it
    again alone gives the bits the second call must have read)."""
    torch = pytest.importorskip("torch")
    from dense_gemm_mma_gb300 import gemm, inputs
    from tests.gemm_case import decode, from_device, sample_positions, to_device, ulp
    import oracle
    s = torch.cuda.current_stream().cuda_stream
    BF32 = gemm.DTYPES[("bf16", "f32")]
    (M, N, K1), (_, _, K2) = first, second
    A1 = inputs.matrix(M, K1, 131, inputs.TENSOR_A, "bf16")
    B1 = inputs.matrix(K1, N, 132, inputs.TENSOR_B, "bf16")
    A2 = inputs.matrix(M, K2, 133, inputs.TENSOR_A, "bf16")
    B2 = inputs.matrix(K2, N, 134, inputs.TENSOR_B, "bf16")
    A1d, B1d, A2d, B2d = (to_device(X, "bf16") for X in (A1, B1, A2, B2))
    C = torch.full((M, N), float("nan"), device="cuda")

    def run(A, B, K, Cd, beta):
        assert gemm.gemm_run(plan.handle, M, N, K, A.data_ptr(), K, B.data_ptr(), N, Cd.data_ptr(), N,
                             1.0, beta, BF32, 0, 0, 0, 0.0, s) == gemm.GEMM_OK
        return plan.last_config()["path"]

    torch.cuda.synchronize()
    p1 = run(A1d, B1d, K1, C, 0.0)
    p2 = run(A2d, B2d, K2, C, 1.0)
    torch.cuda.synchronize()
    second_out = from_device(C, "f32")
    X = torch.full((M, N), float("nan"), device="cuda")
    run(A1d, B1d, K1, X, 0.0)
    torch.cuda.synchronize()
    assert plan.poll_error() == gemm.GEMM_OK
    first_out = from_device(X, "f32")
    if M * N > 2_000_000:  # sampled outputs, recomputed one by one
        rows, cols = sample_positions(M, N, 4096, seed=9)
        exact, rounded = oracle.sample(rows, cols, K2, A2, B2, C=first_out, alpha=1.0, beta=1.0,
                                       in_fmt="bf16", out_fmt="f32")
        got, cin = second_out[rows, cols], first_out[rows, cols]
    else:
        exact, rounded = oracle.gemm(M, N, K2, A2, B2, C=first_out.copy(), alpha=1.0, beta=1.0,
                                     in_fmt="bf16", out_fmt="f32")
        got, cin = second_out, first_out
    amax, bmax = float(np.abs(decode(A2, "bf16")).max()), float(np.abs(decode(B2, "bf16")).max())
    tol = 1e-5 * K2 * amax * bmax + 2.0 ** -21 * (np.abs(exact) + np.abs(cin)) + ulp(exact, "f32")
    err = np.abs(got.astype(np.float64) - decode(rounded, "f32"))
    assert (err <= tol).all(), (p1, p2, int((~(err <= tol)).sum()))


def _check_link(got_bits, A, B, M, N, K, lda, ldb, out_fmt, tb=False, what=""):
    """One call's output against the oracle on the inputs it should have seen."""
    import oracle
    from tests.gemm_case import decode, ulp
    exact, rounded = oracle.gemm(M, N, K, A, B, lda=lda, ldb=ldb, in_fmt="bf16", out_fmt=out_fmt,
                                 transB=tb)
    amax = float(np.abs(decode(A, "bf16")).max())
    bmax = float(np.abs(decode(B, "bf16")).max())
    tol = 1e-5 * K * amax * bmax + 2.0 ** -21 * np.abs(exact) + ulp(exact, out_fmt)
    err = np.abs(decode(got_bits, out_fmt) - decode(rounded, out_fmt))
    assert (err <= tol).all(), f"{what}: {int((~(err <= tol)).sum())} outputs off"


def test_back_to_back_calls_keep_stream_order(plan):
    """Calls enqueued back to back with no synchronisation between them (the
    kernels launch as programmatic dependents of their predecessor): a chain
    in which every call reads the previous call's output, across the K-pair,
    one-CTA tile, split-K and both GEMV kernels, sees finished inputs; and a
    call that overwrites a matrix the previous call is still streaming does
    not disturb that call.  Each output is checked against the oracle on the
    inputs it should have read."""
    torch = pytest.importorskip("torch")
    from dense_gemm_mma_gb300 import gemm, inputs
    from tests.gemm_case import from_device, to_device
    s = torch.cuda.current_stream().cuda_stream
    BF32 = gemm.DTYPES[("bf16", "f32")]
    BB = gemm.DTYPES[("bf16", "bf16")]
    torch.cuda.synchronize()
    # read after write: X0 -> X1 -> X2 -> X3 -> y -> z
    links = [  # (M, N, K, out) of each link; the input is the previous output
        (1024, 256, 2048, "bf16"), (1024, 1024, 256, "bf16"), (1024, 128, 1024, "bf16"),
        (1, 4096, 128, "bf16"), (1, 2048, 4096, "f32")]
    X0 = inputs.matrix(1024, 2048, 61, inputs.TENSOR_A, "bf16")
    Ws = [inputs.matrix(K, N, 62 + i, inputs.TENSOR_B, "bf16") if i < 4 else
          inputs.matrix(N, K, 62 + i, inputs.TENSOR_B, "bf16")  # the last B is given transposed
          for i, (M, N, K, _) in enumerate(links)]
    dev_in = to_device(X0, "bf16")
    dev_w = [to_device(W, "bf16") for W in Ws]
    outs, paths = [], []
    for i, (M, N, K, fmt) in enumerate(links):
        out = torch.empty((M, N), device="cuda", dtype=torch.float32 if fmt == "f32" else torch.bfloat16)
        tb = i == 4
        st = gemm.gemm_run(plan.handle, M, N, K, dev_in.data_ptr(), dev_in.shape[1] if dev_in.dim() == 2 else K,
                           dev_w[i].data_ptr(), K if tb else N, out.data_ptr(), N, 1.0, 0.0,
                           BF32 if fmt == "f32" else BB, 0, int(tb), 0, 0.0, s)
        assert st == gemm.GEMM_OK
        paths.append(plan.last_config()["path"])
        outs.append(out)
        # the next link reads this output (its first row only, for the GEMVs)
        dev_in = out[:1] if i == 2 else out
    # write after read: P @ Q streams P while the next call writes its result into P
    P = inputs.matrix(8192, 1024, 71, inputs.TENSOR_A, "bf16")
    Q = inputs.matrix(1024, 128, 72, inputs.TENSOR_B, "bf16")
    R = inputs.matrix(8192, 64, 73, inputs.TENSOR_A, "bf16")
    T = inputs.matrix(64, 1024, 74, inputs.TENSOR_B, "bf16")
    Pd, Qd, Rd, Td = (to_device(X, "bf16") for X in (P, Q, R, T))
    Y = torch.empty((8192, 128), device="cuda", dtype=torch.float32)
    assert gemm.gemm_run(plan.handle, 8192, 128, 1024, Pd.data_ptr(), 1024, Qd.data_ptr(), 128,
                         Y.data_ptr(), 128, 1.0, 0.0, BF32, 0, 0, 0, 0.0, s) == gemm.GEMM_OK
    paths.append(plan.last_config()["path"])
    assert gemm.gemm_run(plan.handle, 8192, 1024, 64, Rd.data_ptr(), 64, Td.data_ptr(), 1024,
                         Pd.data_ptr(), 1024, 1.0, 0.0, BB, 0, 0, 0, 0.0, s) == gemm.GEMM_OK
    paths.append(plan.last_config()["path"])
    torch.cuda.synchronize()
    assert plan.poll_error() == gemm.GEMM_OK
    assert "tc_splitk_cluster" in paths and "gemv_colstream" in paths and "gemv_rowdot" in paths, paths

    host_in = X0
    for i, (M, N, K, fmt) in enumerate(links):
        got = from_device(outs[i], fmt)
        A = host_in if i != 3 else host_in[:1]
        _check_link(got, A, Ws[i], M, N, K, A.shape[1], Ws[i].shape[1], fmt, tb=(i == 4),
                    what=f"link {i} ({paths[i]})")
        host_in = got
    _check_link(from_device(Y, "f32"), P, Q, 8192, 128, 1024, 1024, 128, "f32", what=f"P @ Q ({paths[5]})")
    _check_link(from_device(Pd, "bf16"), R, T, 8192, 1024, 64, 64, 1024, "bf16", what=f"R @ T into P ({paths[6]})")


# ----------------------------------------------------------- benchmark mode

def test_autotune_benchmark_mode():
    """Benchmark mode times the planner's leading candidates once per shape on
    a scratch copy of C: with beta != 0 the result still matches the oracle
    (the trials did not touch C), a second call of the same shape on new
    buffers reuses the decision, and a new shape is timed once more."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_mma_gb300 import gemm
    p = gemm.Plan(0)
    try:
        assert gemm.gemm_plan_set_autotune(p.handle, True) == gemm.GEMM_OK
        assert gemm.gemm_plan_tuned_count(p.handle) == 0
        r1 = run_case(p, 1300, 2000, 700, beta=0.5, act=1, slope=0.1, out_fmt="bf16", seed=90)
        assert gemm.gemm_plan_tuned_count(p.handle) == 1
        r2 = run_case(p, 1300, 2000, 700, beta=0.5, act=1, slope=0.1, out_fmt="bf16", seed=91)
        assert gemm.gemm_plan_tuned_count(p.handle) == 1 and r2.info == r1.info
        run_case(p, 2304, 2176, 1024, in_fmt="f16", seed=92, sample=2048)
        assert gemm.gemm_plan_tuned_count(p.handle) == 2
        assert p.poll_error() == gemm.GEMM_OK
    finally:
        p.close()


def test_splitk_ragged_with_beta(plan):
    r = run_case(plan, 200, 150, 3000, out_fmt="bf16", beta=0.5, act=1, slope=0.1,
                 env={"GEMM_FORCE_SPLITK": "5", "GEMM_FORCE_TILE": "128x64"}, seed=61)
    assert r.info["splitk"] == 5


def test_plan_cache_survives_workspace_growth(plan):
    """A repeated call reuses its cached plan and descriptors; when another
    call grows (reallocates) the plan's workspace in between, the cached
    split-K call re-targets the new workspace and gives the same bits."""
    import torch
    from dense_gemm_mma_gb300 import gemm, inputs
    from tests.gemm_case import decode, to_device
    import oracle
    M, N, K = 256, 256, 16384
    A = inputs.matrix(M, K, 301, inputs.TENSOR_A, "bf16")
    B = inputs.matrix(K, N, 301, inputs.TENSOR_B, "bf16")
    Ad, Bd = to_device(A, "bf16"), to_device(B, "bf16")
    C1 = torch.zeros(M, N, device="cuda")
    st = torch.cuda.current_stream().cuda_stream

    def call(c):
        assert gemm.gemm_run(plan.handle, M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, c.data_ptr(), N,
                             1.0, 0.0, gemm.GEMM_BF16_F32, 0, 0, 0, 0.0, st) == gemm.GEMM_OK
        torch.cuda.synchronize()
        return plan.last_config()

    info1 = call(C1)
    assert info1["path"] == "tc_splitk"
    first = C1.cpu().numpy().copy()
    # a larger split-K problem grows the workspace
    M2, N2, K2 = 1024, 1024, 65536
    A2 = torch.zeros(M2, K2, device="cuda", dtype=torch.bfloat16)
    B2 = torch.zeros(K2, N2, device="cuda", dtype=torch.bfloat16)
    C2 = torch.zeros(M2, N2, device="cuda")
    assert gemm.gemm_run(plan.handle, M2, N2, K2, A2.data_ptr(), K2, B2.data_ptr(), N2, C2.data_ptr(), N2,
                         1.0, 0.0, gemm.GEMM_BF16_F32, 0, 0, 0, 0.0, st) == gemm.GEMM_OK
    torch.cuda.synchronize()
    info2 = plan.last_config()
    assert info2["workspace_bytes"] > info1["workspace_bytes"]
    C1.zero_()
    info3 = call(C1)
    assert info3["splitk"] == info1["splitk"]
    assert np.array_equal(C1.cpu().numpy().view(np.uint32), first.view(np.uint32))
    # and it is right: sampled against the oracle
    rows = np.arange(0, M, 17)
    cols = (rows * 7) % N
    exact, _ = oracle.sample(rows, cols, K, A, B)
    assert np.all(np.abs(first[rows, cols] - exact) <= 1e-5 * K + 2.0 ** -21 * np.abs(exact))
    # a different output pointer with the same shape is a different entry
    C3 = torch.zeros(M, N, device="cuda")
    call(C3)
    assert np.array_equal(C3.cpu().numpy().view(np.uint32), first.view(np.uint32))


# ----------------------------------------------------------------------- GEMV

@pytest.mark.parametrize("tb", [False, True])
def test_gemv_m1_config(plan, tb):
    r = run_case(plan, 1, 8192, 8192, tb=tb, seed=1235)
    assert r.info["path"] == ("gemv_rowdot" if tb else "gemv_colstream")
    # one wave: at most the CTAs that fit at once (row dot: eight per SM, one row per warp)
    sms = r.info["sms"]
    assert 0 < r.info["grid"] <= (8 if tb else 4) * sms
    if tb:
        assert r.info["grid"] == 8192 // 8


@pytest.mark.parametrize("ta", [False, True])
def test_gemv_n1(plan, ta):
    r = run_case(plan, 8192, 1, 4096, ta=ta, seed=71)
    assert r.info["path"] == ("gemv_colstream" if ta else "gemv_rowdot")


@pytest.mark.parametrize("shape", [(1, 1000, 777), (1000, 1, 777), (1, 1, 333), (1, 13, 5),
                                   (9, 1, 70000)])
@pytest.mark.parametrize("ta,tb", [(False, False), (True, True), (False, True)])
def test_gemv_odd_shapes(plan, shape, ta, tb):
    run_case(plan, *shape, ta=ta, tb=tb, seed=sum(shape) + ta)


def test_gemv_epilogue_and_dtypes(plan):
    run_case(plan, 1, 3000, 1000, in_fmt="f16", out_fmt="f16", beta=0.5, act=1, slope=0.01, seed=81)
    run_case(plan, 3000, 1, 1000, out_fmt="bf16", alpha=2.0, beta=-1.0, seed=82)
    run_case(plan, 1, 3000, 1000, tb=True, out_fmt="f32", alpha=0.5, beta=1.0, act=1, slope=0.3,
             seed=83)


def test_gemv_misaligned_pointers_take_generic_path(plan):
    r = run_case(plan, 1, 500, 300, tb=True, offsets=(1, 1, 1), seed=91)
    assert r.info["path"] == "gemv_generic"
    r = run_case(plan, 500, 1, 300, offsets=(1, 3, 1), seed=92)
    assert r.info["path"] == "gemv_generic"


@pytest.mark.parametrize("splits", [1, 2, 3])
def test_gemv_colstream_long_slices(plan, splits):
    """Slices longer than the shared-memory x chunk (2048 rows) are walked in chunks."""
    r = run_case(plan, 1, 1500, 5000, env={"GEMM_FORCE_GEMV_SPLITK": str(splits)}, seed=95 + splits)
    assert r.info["path"] == "gemv_colstream" and r.info["splitk"] == splits


def test_gemv_deterministic(plan):
    r = run_case(plan, 1, 8192, 8192, repeat=3, seed=93, check=False)
    assert all(np.array_equal(r.outputs[0], o) for o in r.outputs[1:])


# ------------------------------------------------ offsets past 2^31 and 2^32

@pytest.mark.parametrize("case", ["tc_a", "tc_c", "kpair_a", "pair_a", "gemv_colstream", "gemv_rowdot"])
def test_operands_spanning_8_gib(plan, case):
    """Leading dimensions of 65536 (or 32768 for fp32 C; 262144 for the K
    pair's A, 4 GiB) put the last rows of an operand 8 GiB past its base, so
    every address of the path needs more than 32 bits, while the matrices
    hold little data: sampled
    outputs against the oracle on compact host copies, and sentinels in the
    padding that the call must not touch."""
    torch = pytest.importorskip("torch")
    from dense_gemm_mma_gb300 import gemm, inputs
    from tests.gemm_case import decode, sample_positions, ulp
    import oracle
    BIG = 65536
    # (M, N, K, transB, which operand is padded, its leading dimension, planner switches, path)
    M, N, K, tb, padded, ld, env, want = {
        "tc_a": (BIG, 128, 64, False, "A", BIG, {}, "tc"),
        "tc_c": (BIG, 64, 64, False, "C", BIG // 2, {}, "tc"),
        "kpair_a": (8192, 128, 8192, False, "A", 4 * BIG, {}, "tc_splitk_cluster"),   # 4 GiB
        "pair_a": (BIG, 256, 64, False, "A", BIG, {"GEMM_FORCE_TILE": "256x256"}, "tc"),
        "gemv_colstream": (1, 64, BIG, False, "B", BIG, {}, "gemv_colstream"),
        "gemv_rowdot": (1, BIG, 64, True, "B", BIG, {}, "gemv_rowdot")}[case]
    for k, v in env.items():
        os.environ[k] = v
    A = inputs.matrix(M, K, 101, inputs.TENSOR_A, "bf16")
    B = inputs.matrix(N, K, 102, inputs.TENSOR_B, "bf16") if tb else inputs.matrix(K, N, 102, inputs.TENSOR_B, "bf16")

    def place(host, ld_big, dtype, fill):
        rows, cols = host.shape
        full = torch.full((rows * ld_big,), fill, dtype=dtype, device="cuda")
        view = full.view(rows, ld_big)[:, :cols]
        src = torch.from_numpy(host.view(np.int16) if host.dtype == np.uint16 else host)
        view.copy_(src.view(dtype).cuda() if host.dtype == np.uint16 else src.cuda())
        return full, view

    bf = torch.bfloat16
    nan = float("nan")
    big = {}  # the 8 GiB buffers, freed at the end
    if padded == "A":
        big["A"], Ad = place(A, ld, bf, nan)
        Bd = torch.from_numpy(B.view(np.int16)).view(bf).cuda()
        lda, ldb = ld, B.shape[1]
    else:
        Ad = torch.from_numpy(A.view(np.int16)).view(bf).cuda()
        lda = K
        if padded == "B":
            big["B"], Bd = place(B, ld, bf, nan)
            ldb = ld
        else:
            Bd = torch.from_numpy(B.view(np.int16)).view(bf).cuda()
            ldb = B.shape[1]
    if padded == "C":
        big["C"], Cd = place(np.zeros((M, N), np.float32), ld, torch.float32, nan)
        ldc = ld
    else:
        Cd = torch.full((M, N), nan, dtype=torch.float32, device="cuda")
        ldc = N
    try:
        st = gemm.gemm_run(plan.handle, M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb, Cd.data_ptr(), ldc,
                           1.0, 0.0, gemm.DTYPES[("bf16", "f32")], 0, int(tb), 0, 0.0,
                           torch.cuda.current_stream().cuda_stream)
    finally:
        for k in env:
            os.environ.pop(k, None)
    assert st == gemm.GEMM_OK
    torch.cuda.synchronize()
    assert plan.poll_error() == gemm.GEMM_OK
    info = plan.last_config()
    assert info["path"] == want, info["path"]
    if case == "pair_a":
        assert info["cta_per_tile"] == 2
    rows, cols = sample_positions(M, N, 4096, seed=7)
    got = Cd.cpu().numpy()[rows, cols].astype(np.float64)
    exact, rounded = oracle.sample(rows, cols, K, A, B, lda=K, ldb=B.shape[1], in_fmt="bf16", out_fmt="f32",
                                   transB=tb)
    amax = float(np.abs(decode(A, "bf16")).max())
    bmax = float(np.abs(decode(B, "bf16")).max())
    tol = 1e-5 * K * amax * bmax + 2.0 ** -21 * np.abs(exact) + ulp(exact, "f32")
    assert (np.abs(got - decode(rounded, "f32")) <= tol).all(), case
    if padded == "C":  # padding of C's rows, including the far end, still holds its sentinel
        pad = big["C"].view(M, ld)[[0, M // 2, M - 1], N:N + 64].cpu().numpy()
        assert np.isnan(pad).all()
    del Ad, Bd, Cd
    big.clear()
    torch.cuda.empty_cache()


# ------------------------------------------------------- full-size workloads

SAMPLE = 4096


def test_full_config2_skinny_both_b_layouts(plan):
    for tb in (False, True):
        run_case(plan, 8192, 128, 8192, tb=tb, seed=1235, sample=SAMPLE)


def test_full_config3_square_bf16_out(plan):
    r = run_case(plan, 8192, 8192, 8192, out_fmt="bf16", seed=1236, sample=SAMPLE)
    assert r.info["path"] in ("tc", "tc_tail_split") and r.info["cta_per_tile"] == 2


def test_full_config3_beta_leaky_relu(plan):
    run_case(plan, 8192, 8192, 8192, out_fmt="f32", beta=0.5, act=1, slope=0.01, seed=1236,
             sample=SAMPLE)


def test_full_config4_tile_sweep_points(plan):
    run_case(plan, 6912, 2048, 4096, seed=1237, sample=SAMPLE)
    for n in (128, 136, 200, 256):
        run_case(plan, 27648, n, 4096, seed=1237, sample=SAMPLE)


def test_full_config5_wave_sweep_points_and_splitk(plan):
    for n in (1024, 1536, 1544, 3080, 6400):
        run_case(plan, 2304, n, 4096, in_fmt="f16", seed=1238, sample=SAMPLE)
    r = run_case(plan, 256, 256, 65536, in_fmt="f16", seed=1238, sample=SAMPLE, repeat=2)
    assert r.info["path"] == "tc_splitk"
    assert np.array_equal(r.outputs[0].view(np.uint8), r.outputs[1].view(np.uint8))


def test_nvtx_ranges_do_not_change_results(monkeypatch):
    """GEMM_NVTX=1 at plan creation wraps every call in an NVTX range; without
    a profiler attached the ranges are inert and the results are the oracle's."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_mma_gb300 import gemm
    monkeypatch.setenv("GEMM_NVTX", "1")
    p = gemm.Plan(0)
    try:
        run_case(p, 300, 260, 333, seed=501)
        run_case(p, 1, 3000, 1000, seed=502)
    finally:
        p.close()
