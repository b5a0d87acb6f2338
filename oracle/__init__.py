"""CPU oracle for the dense GEMM path: ctypes binding of ``oracle.c``.

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``; the
product package never imports it.

The computation follows "Matrix Multiplication Background User's Guide",
section 2 (A is M x K, B is K x N, C is M x N, one K-long dot product per
output) with the BLAS reading D = act(alpha*op(A)@op(B) + beta*C), and
"Learning Triton One Kernel at a Time: Matrix Multiplication", section Naive
GEMM (one dot product per row/column pair).  Inputs are decoded exactly to
fp64, accumulated in fp64 in ascending k, and rounded once (nearest-even) to
the output format.  See ``oracle.c`` for the full statement.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

BF16, F16, F32, TF32 = 0, 1, 2, 3
FMT_NAMES = {"bf16": BF16, "f16": F16, "f32": F32, "tf32": TF32}

_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (plain C11, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, vp, d, i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int
        lib.oracle_decode.argtypes = [ctypes.c_uint32, i]
        lib.oracle_decode.restype = d
        lib.oracle_round_bf16.argtypes = [d]
        lib.oracle_round_bf16.restype = ctypes.c_uint16
        lib.oracle_round_f16.argtypes = [d]
        lib.oracle_round_f16.restype = ctypes.c_uint16
        lib.oracle_round_f32.argtypes = [d]
        lib.oracle_round_f32.restype = ctypes.c_float
        lib.oracle_entry.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, d, d,
                                     i, i, i, i, i, d]
        lib.oracle_entry.restype = d
        lib.oracle_gemm.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, d, d,
                                    i, i, i, i, i, i, d, vp, vp]
        lib.oracle_gemm.restype = i
        lib.oracle_sample.argtypes = [i64, vp, vp, i64, vp, i64, vp, i64, vp, i64, d, d,
                                      i, i, i, i, i, i, d, vp, vp]
        lib.oracle_sample.restype = i
        _lib = lib
    return _lib


def _fmt(f) -> int:
    return FMT_NAMES[f] if isinstance(f, str) else int(f)


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _ld(a, ld):
    if ld is not None:
        return int(ld)
    return int(a.shape[1]) if a is not None and a.ndim == 2 else 1


def _out_array(shape, fmt):
    return np.empty(shape, dtype=np.float32 if fmt == F32 else np.uint16)


def gemm(M, N, K, A, B, *, lda=None, ldb=None, C=None, ldc=None, alpha=1.0, beta=0.0,
         in_fmt="bf16", out_fmt="f32", transA=False, transB=False, act=0, slope=0.0, c_fmt=None):
    """Full M x N result.  A, B (and C) are the STORED arrays: uint16 bit
    patterns for bf16/fp16, float32 for fp32; row strides lda/ldb/ldc default
    to the arrays' widths.  C is in c_fmt (default: out_fmt, C updated in
    place).  Returns (exact_f64[M,N], rounded[M,N])."""
    lib = _load()
    fi, fo = _fmt(in_fmt), _fmt(out_fmt)
    fc = _fmt(c_fmt if c_fmt is not None else out_fmt)
    exact = np.empty((M, N), dtype=np.float64)
    out = _out_array((M, N), fo)
    rc = lib.oracle_gemm(M, N, K, _ptr(A), _ld(A, lda), _ptr(B), _ld(B, ldb),
                         _ptr(C), _ld(C, ldc), float(alpha), float(beta), fi, fo, fc,
                         int(bool(transA)), int(bool(transB)), int(act), float(slope),
                         exact.ctypes.data, out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return exact, out


def sample(rows, cols, K, A, B, *, lda=None, ldb=None, C=None, ldc=None, alpha=1.0,
           beta=0.0, in_fmt="bf16", out_fmt="f32", transA=False, transB=False, act=0,
           slope=0.0, c_fmt=None):
    """Entries (rows[t], cols[t]) only; same values as gemm() at those places."""
    lib = _load()
    fi, fo = _fmt(in_fmt), _fmt(out_fmt)
    fc = _fmt(c_fmt if c_fmt is not None else out_fmt)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    n = rows.shape[0]
    exact = np.empty(n, dtype=np.float64)
    out = _out_array(n, fo)
    rc = lib.oracle_sample(n, rows.ctypes.data, cols.ctypes.data, K, _ptr(A), _ld(A, lda),
                           _ptr(B), _ld(B, ldb), _ptr(C), _ld(C, ldc), float(alpha),
                           float(beta), fi, fo, fc, int(bool(transA)), int(bool(transB)),
                           int(act), float(slope), exact.ctypes.data, out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_sample rejected its arguments")
    return exact, out


def decode(bits, fmt) -> float:
    return _load().oracle_decode(int(bits), _fmt(fmt))


def round_bf16(x: float) -> int:
    return int(_load().oracle_round_bf16(float(x)))


def round_f16(x: float) -> int:
    return int(_load().oracle_round_f16(float(x)))


def round_f32(x: float) -> float:
    return float(_load().oracle_round_f32(float(x)))
