"""Seeded synthetic inputs for the GEMM path (shared by tests, bench and smoke).

This module holds no GEMM arithmetic: it only draws numbers and rounds them to
the operand format.  Both the CUDA path and the CPU oracle receive the arrays
it returns; neither computes them.

Generator (counter-based, so any entry can be regenerated from its index):

    ctr   = seed * 2^40 + tensor_id * 2^36 + idx          (mod 2^64)
    h     = splitmix64(ctr)
    u     = (h >> 40) * 2^-24                             in [0, 1)
    value = 2u - 1                                        in [-1, 1)

splitmix64 is the finaliser published with the SplitMix generator (Steele,
Lea and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014;
constants as in Vigna's splitmix64.c).  ``value`` has at most 24 significant
bits, so it is exact in fp32; it is then rounded once, to nearest-even, to
bf16 or fp16.  ``idx`` is the row-major index in the stored (rows x cols)
matrix, ignoring any padding columns (ld > cols), which are filled with a NaN
sentinel so that a kernel that reads them produces NaN.

Tensor ids: A = 0, B = 1, C = 2 (the bench and tests use these).
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TENSOR_A, TENSOR_B, TENSOR_C = 0, 1, 2
BF16_NAN = np.uint16(0x7FC1)
F16_NAN = np.uint16(0x7E01)


def splitmix64(x: np.ndarray) -> np.ndarray:
    z = x.astype(np.uint64) + _GOLDEN
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def counters(seed: int, tensor_id: int, idx: np.ndarray) -> np.ndarray:
    if not (0 <= seed < 2 ** 24 and 0 <= tensor_id < 16):
        raise ValueError("seed must be < 2^24 and tensor_id < 16")
    idx = np.asarray(idx, dtype=np.uint64)
    base = np.uint64((seed << 40) | (tensor_id << 36))
    return base | idx


def uniform_pm1(seed: int, tensor_id: int, idx: np.ndarray) -> np.ndarray:
    """Values in [-1, 1) as float32 (exact) for the given linear indices."""
    h = splitmix64(counters(seed, tensor_id, idx))
    u = (h >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
    return (2.0 * u - 1.0).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest-even) and return the uint16 patterns."""
    w = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (w + np.uint64(0x7FFF) + ((w >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def _encode(vals: np.ndarray, fmt: str) -> np.ndarray:
    if fmt == "bf16":
        return f32_to_bf16_bits(vals)
    if fmt == "f16":
        return f32_to_f16_bits(vals)
    if fmt in ("f32", "tf32"):  # a TF32 operand is a full fp32 word; the tensor core drops its low bits
        return vals.astype(np.float32)
    raise ValueError(fmt)


def matrix(rows: int, cols: int, seed: int, tensor_id: int, fmt: str = "bf16",
           ld: int | None = None, chunk: int = 1 << 23) -> np.ndarray:
    """Stored matrix of shape (rows, ld): uint16 bit patterns for bf16/fp16,
    float32 for f32 and tf32.  Entry (r, c) with c < cols is drawn from index r*cols+c."""
    ld = cols if ld is None else ld
    if ld < cols:
        raise ValueError("ld < cols")
    dtype = np.float32 if fmt in ("f32", "tf32") else np.uint16
    total = rows * cols
    flat = np.empty(total, dtype=dtype)
    for s in range(0, total, chunk):
        e = min(total, s + chunk)
        flat[s:e] = _encode(uniform_pm1(seed, tensor_id, np.arange(s, e, dtype=np.uint64)), fmt)
    dense = flat.reshape(rows, cols) if rows and cols else flat.reshape(rows, cols)
    if ld == cols:
        return dense
    out = np.empty((rows, ld), dtype=dtype)
    out[:, cols:] = {"bf16": BF16_NAN, "f16": F16_NAN}.get(fmt, np.float32(np.nan))
    out[:, :cols] = dense
    return out


def entries(seed: int, tensor_id: int, cols: int, r: np.ndarray, c: np.ndarray,
            fmt: str = "bf16") -> np.ndarray:
    """Regenerate individual entries (r, c) of matrix(rows, cols, seed, tensor_id)."""
    idx = np.asarray(r, dtype=np.uint64) * np.uint64(cols) + np.asarray(c, dtype=np.uint64)
    return _encode(uniform_pm1(seed, tensor_id, idx), fmt)


def config_seed(index: int) -> int:
    """Seed for the workload with the given 0-based index in the config list."""
    return 1234 + index
