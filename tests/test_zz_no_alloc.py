"""gemm_gemv_noalloc: the GEMV entry point for callers that may not call
cudaMalloc where they run (a plugin inside a framework that owns all device
memory through its own pool allocator, or a latency-critical loop that cannot
take cudaMalloc's implicit synchronisation).  Its scratch is a fixed device
array of the library, so it needs no plan and allocates nothing.

Every call is checked through the C ABI against the CPU oracle, element by
element, within the tolerance the parity tests use, on two calls in a row:
the second call runs on the scratch as the first call left it (partial sums
of the first call's K slices), and device memory must not move during it.
Two cases force a K split larger than the fixed scratch holds, so that the
entry point's shrinking of the split runs: once down to fewer slices, once
down to a single slice.  This file is collected last so that a run stopping
at the first failure has run every other test.
"""
import os

import numpy as np
import pytest

from tests.gemm_case import decode, from_device, round_up, to_device, ulp

pytestmark = pytest.mark.gpu

CASES = [
    # M, N, K, in, out, transA, transB, alpha, beta, act, slope, forced GEMV K split
    (1, 8192, 8192, "bf16", "f32", False, False, 1.0, 0.0, 0, 0.0, None),
    (1, 1000, 777, "bf16", "bf16", True, False, 0.5, -1.0, 1, 0.01, None),
    (3000, 1, 2500, "f16", "f16", True, True, 1.0, 0.5, 1, 0.2, None),
    (1, 70000, 1024, "f16", "f32", False, False, 2.0, 0.0, 0, 0.0, None),
    # 137 panels x 512 columns: 64 slices asked for, the partials hold 14
    (1, 70000, 1024, "bf16", "f32", False, False, 1.0, 0.5, 0, 0.0, "64"),
    # 1172 panels: not even two slices fit, so one slice and no partials
    (1, 600000, 128, "bf16", "f32", False, False, 1.0, 0.0, 0, 0.0, "4"),
]


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from dense_gemm_mma_gb300 import gemm
    return gemm


def _operands(M, N, K, in_fmt, out_fmt, ta, tb, seed):
    from dense_gemm_mma_gb300 import inputs
    a_rows, a_cols = (K, M) if ta else (M, K)
    b_rows, b_cols = (N, K) if tb else (K, N)
    lda = round_up(a_cols, 8)
    ldb = round_up(b_cols, 8)
    ldc = round_up(N, 16 // (4 if out_fmt == "f32" else 2))
    A = inputs.matrix(a_rows, a_cols, seed, inputs.TENSOR_A, in_fmt, ld=lda)
    B = inputs.matrix(b_rows, b_cols, seed, inputs.TENSOR_B, in_fmt, ld=ldb)
    C = inputs.matrix(M, N, seed, inputs.TENSOR_C, out_fmt, ld=ldc)
    return A, B, C, lda, ldb, ldc


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:3])) + f"_{c[3]}_{c[4]}"
                         + (f"_split{c[11]}" if c[11] else ""))
def test_noalloc_matches_oracle_on_two_calls(lib, case):
    import torch

    import oracle
    gemm = lib
    M, N, K, in_fmt, out_fmt, ta, tb, alpha, beta, act, slope, force = case
    A, B, C, lda, ldb, ldc = _operands(M, N, K, in_fmt, out_fmt, ta, tb, seed=M + N + K)
    Ad, Bd, C0 = to_device(A, in_fmt), to_device(B, in_fmt), to_device(C, out_fmt)
    dtype = gemm.DTYPES[(in_fmt, out_fmt)]
    stream = torch.cuda.current_stream().cuda_stream

    exact, rounded = oracle.gemm(M, N, K, A, B, lda=lda, ldb=ldb, C=C, ldc=ldc, alpha=alpha, beta=beta,
                                 in_fmt=in_fmt, out_fmt=out_fmt, transA=ta, transB=tb, act=act, slope=slope)
    ref = decode(rounded, out_fmt)
    a_dec, b_dec = decode(A, in_fmt), decode(B, in_fmt)
    a_max = float(np.abs(a_dec[np.isfinite(a_dec)]).max())
    b_max = float(np.abs(b_dec[np.isfinite(b_dec)]).max())
    c_in = np.abs(decode(C[:, :N], out_fmt)) if beta != 0.0 else 0.0
    tol = (1e-5 * K * a_max * b_max * max(1.0, abs(alpha))
           + 2.0 ** -21 * (np.abs(exact) + abs(beta) * c_in) + ulp(exact, out_fmt))

    old = os.environ.get("GEMM_FORCE_GEMV_SPLITK")
    if force:
        os.environ["GEMM_FORCE_GEMV_SPLITK"] = force
    try:
        for call in range(2):
            Cn = C0.clone()
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
            st = gemm.gemm_gemv_noalloc(M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb, Cn.data_ptr(),
                                        ldc, alpha, beta, dtype, int(ta), int(tb), act, slope, stream)
            assert st == gemm.GEMM_OK, gemm.gemm_status_string(st)
            torch.cuda.synchronize()
            if call == 1:  # after the first call's one-time set-up, device memory does not move
                assert torch.cuda.mem_get_info()[0] == free_before
            out = from_device(Cn, out_fmt).reshape(M, ldc)
            got = decode(out[:, :N], out_fmt)
            err = np.abs(got - ref)
            bad = ~(err <= tol)
            assert not bad.any(), (f"call {call}: {int(bad.sum())} outputs off, max err {err.max()}, "
                                   f"first at {tuple(np.argwhere(bad)[0])}")
            # the ld padding of C is untouched
            assert np.array_equal(out[:, N:].view(np.uint8), C[:, N:].view(np.uint8))
    finally:
        if old is None:
            os.environ.pop("GEMM_FORCE_GEMV_SPLITK", None)
        else:
            os.environ["GEMM_FORCE_GEMV_SPLITK"] = old


def test_noalloc_rejects_what_it_cannot_hold(lib):
    gemm = lib
    fake = 0x100000  # never dereferenced: rejected before any launch
    # output longer than the fixed scratch holds
    assert gemm.gemm_gemv_noalloc(1, 3_000_000, 64, fake, 64, fake, 3_000_000, fake + (1 << 32),
                                  3_000_000, 1.0, 0.0, gemm.GEMM_BF16_F32, 0, 0) == gemm.GEMM_ERR_UNSUPPORTED
    # not a column-stream GEMV shape
    assert gemm.gemm_gemv_noalloc(64, 64, 64, fake, 64, fake + (1 << 32), 64, fake + (2 << 32), 64, 1.0,
                                  0.0, gemm.GEMM_BF16_F32, 0, 0) == gemm.GEMM_ERR_UNSUPPORTED
    assert gemm.gemm_gemv_noalloc(1, 64, 64, fake, 64, fake + (1 << 32), 64, fake + (2 << 32), 64, 1.0,
                                  0.0, gemm.GEMM_BF16_F32, 0, 1) == gemm.GEMM_ERR_UNSUPPORTED
    # argument errors are gemm_run's
    assert gemm.gemm_gemv_noalloc(1, 64, 64, fake, 64, fake, 32, fake, 64, 1.0, 0.0,
                                  gemm.GEMM_BF16_F32, 0, 0) == gemm.GEMM_ERR_INVALID_ARG
    # ... the output sharing bytes with an operand included
    assert gemm.gemm_gemv_noalloc(1, 64, 64, fake, 64, fake + (1 << 32), 64, fake + (1 << 32) + 64, 64,
                                  1.0, 0.0, gemm.GEMM_BF16_F32, 0, 0) == gemm.GEMM_ERR_INVALID_ARG
