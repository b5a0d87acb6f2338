"""GEMM cases run through the debug build of the library (device-side bounds
and copy-rule checks, include/gemm.h: gemm_debug_build).  test_debug_build.py
runs this module in a child process with GEMM_DEBUG=1, which makes the
binding load libdgemm_gb300_debug.so at its first load:

    python -m tests.debug_cases parity   every kernel path, compared with the
                                         oracle element by element; no check fails
    python -m tests.debug_cases shrink   run with GEMM_DEBUG_SHRINK=4: the output's
                                         range is taken 4 bytes short, so on each path
                                         that writes the last output element with a
                                         plain store its check fails and the store is
                                         skipped; every other element is right

Prints one line starting with "ok" on success.
"""
from __future__ import annotations

import os
import sys

import numpy as np

import oracle
from dense_gemm_mma_gb300 import gemm, inputs
from tests.gemm_case import decode, from_device, round_up, run_case, run_case_ex, to_device

PATH_CASES = [
    # M, N, K and run_case keyword arguments
    (300, 260, 333, {}),                                                   # one-CTA tiles, fp32 tail columns
    (300, 262, 333, {"out_fmt": "bf16", "beta": 0.5, "act": 1, "slope": 0.1}),
    (700, 600, 300, {"env": {"GEMM_FORCE_TILE": "256x256"}}),               # CTA pair
    (257, 300, 515, {"beta": 0.5, "env": {"GEMM_SPLITK_CLUSTER": "1", "GEMM_FORCE_SPLITK": "2"}}),  # K pair
    (256, 256, 8192, {"in_fmt": "f16", "env": {"GEMM_FORCE_SPLITK": "8", "GEMM_SPLITK_CLUSTER": "0"}}),
    (1300, 2000, 515, {"beta": -1.0, "env": {"GEMM_TAIL_SPLIT": "3", "GEMM_FORCE_TILE": "128x128"}}),
    (1300, 2000, 515, {"env": {"GEMM_TAIL_SPLIT": "3", "GEMM_FORCE_TILE": "128x128", "GEMM_FUSED_REDUCE": "1"}}),
    (1, 3000, 1000, {}),                                                    # column-stream GEMV
    (1, 3000, 1000, {"tb": True, "beta": 0.5}),                            # row-dot GEMV
    (3000, 1, 1000, {"ta": True}),
    (1, 500, 300, {"tb": True, "offsets": (1, 1, 1)}),                     # generic GEMV
    (100, 70, 0, {"beta": 2.0}),                                            # K == 0
    (300, 520, 333, {"in_fmt": "tf32", "ta": True, "tb": False}),          # TF32 transposes
]


def parity() -> None:
    assert gemm.gemm_debug_build() == 1, gemm.LIB_PATH
    plan = gemm.Plan(0)
    for M, N, K, kw in PATH_CASES:
        run_case(plan, M, N, K, seed=M + N + K, **kw)  # asserts the error word stays clear
    run_case_ex(plan, 300, 260, 515, c_fmt="f32", d_fmt="bf16", beta=0.5, seed=3)
    print("ok", len(PATH_CASES) + 1)


# path forced, sites whose check fails: the last output element of a ragged
# fp32 output is written with a plain store by each of these
SHRINK_CASES = [
    ("tc", 130, 130, 64, {"GEMM_FORCE_TILE": "128x128", "GEMM_FORCE_SPLITK": "1", "GEMM_TAIL_SPLIT": "0",
                          "GEMM_SPLITK_CLUSTER": "0"}, "epilogue_store"),
    ("tc_splitk_cluster", 130, 130, 256, {"GEMM_SPLITK_CLUSTER": "1", "GEMM_FORCE_SPLITK": "2"}, "epilogue_store"),
    ("tc_splitk", 130, 130, 256, {"GEMM_FORCE_TILE": "128x128", "GEMM_FORCE_SPLITK": "2",
                                  "GEMM_SPLITK_CLUSTER": "0"}, "tile_reduce"),
    ("gemv_colstream", 1, 1000, 512, {}, "gemv"),
    ("scale", 130, 130, 0, {}, "scale"),
]


def shrink() -> None:
    import torch
    assert gemm.gemm_debug_build() == 1 and os.environ.get("GEMM_DEBUG_SHRINK") == "4"
    for path, M, N, K, env, site in SHRINK_CASES:
        os.environ.update(env)
        plan = gemm.Plan(0)
        lda, ldb, ldc = round_up(max(K, 1), 8), round_up(N, 8), round_up(N, 4)
        A = inputs.matrix(M, K, 5, inputs.TENSOR_A, "bf16", ld=lda)
        B = inputs.matrix(K, N, 5, inputs.TENSOR_B, "bf16", ld=ldb)
        C0 = np.full((M, ldc), np.nan, np.float32)
        Ad, Bd, Cd = to_device(A, "bf16"), to_device(B, "bf16"), to_device(C0, "f32")
        st = gemm.gemm_run(plan.handle, M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb, Cd.data_ptr(), ldc,
                           1.0, 0.0, gemm.GEMM_BF16_F32, 0, 0, 0, 0.0, torch.cuda.current_stream().cuda_stream)
        assert st == gemm.GEMM_OK, (path, gemm.gemm_status_string(st))
        torch.cuda.synchronize()
        assert plan.last_config()["path"] == path, (path, plan.last_config())
        assert plan.poll_error() == gemm.GEMM_ERR_DEBUG_CHECK, path
        bits = gemm.gemm_plan_last_error_bits(plan.handle)
        assert bits & gemm.DBG_FLAG and gemm.debug_sites(bits) == [site], (path, hex(bits))
        assert (bits & 0xFFFF) == 0, (path, hex(bits))  # no wait ran out
        out = from_device(Cd, "f32").reshape(M, ldc)[:, :N].astype(np.float64)
        assert np.isnan(out[M - 1, N - 1]), path  # the skipped store
        exact, _ = oracle.gemm(M, N, K, A, B, lda=lda, ldb=ldb, in_fmt="bf16", out_fmt="f32")
        got, ref = out.ravel()[:-1], np.asarray(exact, np.float64).ravel()[:-1]
        tol = 1e-5 * max(K, 1) + 2.0 ** -21 * np.abs(ref)  # |A|, |B| <= 1
        assert np.all(np.abs(got - ref) <= tol), path
        plan.close()
        for k in env:
            os.environ.pop(k)
    print("ok", len(SHRINK_CASES))


if __name__ == "__main__":
    {"parity": parity, "shrink": shrink}[sys.argv[1]]()
