"""FLOP / byte accounting and the roofline used by the benchmark.

"Matrix Multiplication Background User's Guide", section 2 (Math and Memory
Bounds): a GEMM performs M*N*K fused multiply-adds, 2*M*N*K floating-point
operations; its arithmetic intensity is those FLOPs over the bytes moved
(A, B read and C written -- and read again when beta != 0); it is
memory-bound when that intensity is below the GPU's ops:byte ratio.  The
attainable rate is min(peak FLOP/s, intensity * memory bandwidth).
"""
from __future__ import annotations

ELEM_BYTES = {"bf16": 2, "f16": 2, "f32": 4, "tf32": 4}


def gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def gemm_bytes(M: int, N: int, K: int, in_fmt: str = "bf16", out_fmt: str = "f32",
               beta: bool = False) -> int:
    """Algorithmic bytes: A and B read once, C written once (and read once if beta != 0)."""
    ib, cb = ELEM_BYTES[in_fmt], ELEM_BYTES[out_fmt]
    return (M * K + K * N) * ib + M * N * cb * (2 if beta else 1)


def intensity(M: int, N: int, K: int, in_fmt: str = "bf16", out_fmt: str = "f32",
              beta: bool = False) -> float:
    return gemm_flops(M, N, K) / gemm_bytes(M, N, K, in_fmt, out_fmt, beta)


def tflops(flops: float, seconds: float) -> float:
    return flops / seconds / 1e12


def attainable(ai: float, peak_flops: float, bandwidth: float) -> float:
    """min(peak, AI * BW) in FLOP/s."""
    return min(peak_flops, ai * bandwidth)


def bound(ai: float, peak_flops: float, bandwidth: float) -> str:
    return "tensor" if ai * bandwidth >= peak_flops else "hbm"
