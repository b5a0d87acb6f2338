"""The debug build of the library (device-side checks of every plain global
access and every TMA coordinate, include/gemm.h: gemm_debug_build), run in
child processes because the binding loads one library per process.

- Every kernel path (one-CTA, pair and K-pair tiles, split-K with the
  reduction kernel and in the kernel, tail split, the three GEMV kernels, the
  K == 0 kernel, the TF32 transposes, a separate C and D) gives the oracle's
  results under the checks, and no check fails: the kernels stay inside the
  call's buffers and keep the TMA copy rules.
- With the output's range taken 4 bytes short (GEMM_DEBUG_SHRINK, read by the
  debug build only), each path that writes the last output element with a
  plain store skips it and reports the failing site through
  gemm_plan_poll_error / gemm_plan_last_error_bits; nothing faults (every
  access stays inside the real buffer) and every other element is right.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(mode, extra_env=None):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_mma_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, GEMM_DEBUG="1", **(extra_env or {}))
    for k in [k for k in env if k.startswith("GEMM_") and k not in ("GEMM_DEBUG", "GEMM_DEBUG_SHRINK")]:
        env.pop(k)
    r = subprocess.run([sys.executable, "-m", "tests.debug_cases", mode], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().startswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]


def test_debug_build_every_path_matches_oracle_without_a_failed_check():
    _run("parity")


def test_debug_build_skips_and_reports_an_out_of_range_store():
    _run("shrink", {"GEMM_DEBUG_SHRINK": "4"})
