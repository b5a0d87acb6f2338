"""Shared helper of the GPU parity tests: seeded inputs -> C ABI on the GPU ->
comparison with the CPU oracle, element by element.

Tolerance (fp32 accumulation against the fp64 oracle):
    |C_gpu - C_oracle| <= 1e-5 * K * max|A| * max|B| * max(1, |alpha|)
                          + 2^-21 * (|C_oracle| + |beta| * |C_in|)
                          + 1 ulp of the output format at |C_oracle| (16-bit outputs)
The first term is the accumulation bound; the second covers the fp32
rounding of alpha*acc, beta*C and the activation; the ulp term covers the
final rounding to bf16/fp16, where the GPU rounds an fp32 value and the
oracle rounds the fp64 one, so a tie can break either way.

GELU and SiLU are smooth: an error e in their argument moves the result by
at most L*e, L = max|f'| (1.07 for GELU, at x = sqrt 2; 1.10 for SiLU, near
x = 2.4), so the first two terms are taken with |C_oracle| replaced by the
value before the activation and multiplied by 1.1; their fp32 evaluation
(erfcf / expf within a few ulp, then two roundings) adds 2^-20 * |C_oracle|.
"""
from __future__ import annotations

import os

import numpy as np

import oracle
from dense_gemm_mma_gb300 import gemm, inputs

ESIZE = {"bf16": 2, "f16": 2, "f32": 4, "tf32": 4}


def decode(bits, fmt):
    bits = np.asarray(bits)
    if fmt == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if fmt == "f16":
        return bits.astype(np.uint16).view(np.float16).astype(np.float64)
    return bits.astype(np.float64)


def ulp(x, fmt):
    if fmt == "f32":
        return np.zeros_like(x)
    p, emin = (8, -126) if fmt == "bf16" else (11, -14)
    _, e = np.frexp(np.abs(x))
    ex = np.maximum(e - 1, emin)
    return np.ldexp(1.0, ex - (p - 1))


def round_up(x, m):
    return (x + m - 1) // m * m


def to_device(arr, fmt):
    import torch
    if fmt in ("f32", "tf32"):
        return torch.from_numpy(np.ascontiguousarray(arr)).cuda()
    t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16))
    return t.view(torch.bfloat16 if fmt == "bf16" else torch.float16).cuda()


def from_device(t, fmt):
    import torch
    t = t.cpu()
    if fmt in ("f32", "tf32"):
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def sample_positions(M, N, n=4096, seed=99):
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, n))
    cols = list(rng.integers(0, N, n))
    edge_r = sorted({r for r in (0, M - 1) + tuple(x for b in range(0, M, 256)
                                                      for x in (b, b + 127, b + 128, b + 255))
                     if 0 <= r < M})
    edge_c = sorted({c for c in (0, N - 1) + tuple(x for b in range(0, N, 256)
                                                      for x in (b, b + 63, b + 64, b + 127, b + 128, b + 255))
                     if 0 <= c < N})
    for r in (0, M - 1):
        for c in (0, N - 1):
            rows.append(r)
            cols.append(c)
    for c in rng.integers(0, N, 64):
        rows.append(M - 1)
        cols.append(int(c))
    for r in rng.integers(0, M, 64):
        rows.append(int(r))
        cols.append(N - 1)
    for r in edge_r[:64]:
        for c in edge_c[:16]:
            rows.append(r)
            cols.append(c)
    return np.array(rows, dtype=np.int64), np.array(cols, dtype=np.int64)


class Result:
    pass


def run_case(plan, M, N, K, in_fmt="bf16", out_fmt="f32", ta=False, tb=False, alpha=1.0,
             beta=0.0, act=0, slope=0.0, seed=1, pad=(0, 0, 0), sample=None, env=None,
             check=True, repeat=1, offsets=(0, 0, 0)):
    """Run one GEMM through the C ABI and compare with the oracle.

    pad: extra elements added to lda/ldb/ldc beyond the smallest legal
    (16-byte multiple) leading dimension; the padding holds NaN sentinels,
    which the kernels must neither read nor write.  sample: None for a full
    check, else a number of sampled output entries.  offsets: element offsets
    of A/B/C inside their buffers (misaligned pointers for the GEMV paths)."""
    import torch
    old_env = {}
    for k, v in (env or {}).items():
        old_env[k] = os.environ.get(k)
        os.environ[k] = v
    try:
        a_rows, a_cols = (K, M) if ta else (M, K)
        b_rows, b_cols = (N, K) if tb else (K, N)
        ie, ce = ESIZE[in_fmt], ESIZE[out_fmt]
        lda = round_up(max(a_cols, 1), 16 // ie) + pad[0]
        ldb = round_up(max(b_cols, 1), 16 // ie) + pad[1]
        ldc = round_up(max(N, 1), 16 // ce) + pad[2]
        A = inputs.matrix(a_rows, a_cols, seed, inputs.TENSOR_A, in_fmt, ld=lda)
        B = inputs.matrix(b_rows, b_cols, seed, inputs.TENSOR_B, in_fmt, ld=ldb)
        if beta != 0.0:
            C0 = inputs.matrix(M, N, seed, inputs.TENSOR_C, out_fmt, ld=ldc)
        else:
            C0 = inputs.matrix(M, N, seed, inputs.TENSOR_C, out_fmt, ld=ldc)
            C0[:, :N] = inputs.BF16_NAN if out_fmt == "bf16" else (
                inputs.F16_NAN if out_fmt == "f16" else np.float32(np.nan))
        dev = [to_device(np.concatenate([np.zeros(o, X.dtype), X.ravel()]), f)
               for X, f, o in ((A, in_fmt, offsets[0]), (B, in_fmt, offsets[1]), (C0, out_fmt, offsets[2]))]
        Ad, Bd, Cd = dev
        dtype = gemm.DTYPES[(in_fmt, out_fmt)]
        stream = torch.cuda.current_stream().cuda_stream
        outs = []
        for _ in range(repeat):
            Cd.copy_(to_device(np.concatenate([np.zeros(offsets[2], C0.dtype), C0.ravel()]), out_fmt))
            st = gemm.gemm_run(plan.handle, M, N, K, Ad.data_ptr() + offsets[0] * ie, lda,
                               Bd.data_ptr() + offsets[1] * ie, ldb,
                               Cd.data_ptr() + offsets[2] * ce, ldc, alpha, beta, dtype,
                               int(ta), int(tb), act, slope, stream)
            assert st == gemm.GEMM_OK, gemm.gemm_status_string(st)
            torch.cuda.synchronize()
            assert plan.poll_error() == gemm.GEMM_OK, "watchdog fired"
            outs.append(from_device(Cd, out_fmt)[offsets[2]:].reshape(M, ldc))
        res = Result()
        res.info = plan.last_config()
        res.outputs = outs
        out = outs[0]
        if not check:
            return res
        # padding columns untouched (bitwise)
        if ldc > N:
            assert np.array_equal(out[:, N:].view(np.uint8), C0[:, N:].view(np.uint8)), "ld padding written"
        a_dec = decode(A[:, :a_cols], in_fmt)
        b_dec = decode(B[:, :b_cols], in_fmt)
        amax = float(np.abs(a_dec).max()) if a_dec.size else 0.0
        bmax = float(np.abs(b_dec).max()) if b_dec.size else 0.0
        cin = decode(C0[:, :N], out_fmt) if beta != 0.0 else np.zeros((M, N))
        if sample is None:
            exact, rounded = oracle.gemm(M, N, K, A, B, lda=lda, ldb=ldb, C=C0, ldc=ldc, alpha=alpha,
                                         beta=beta, in_fmt=in_fmt, out_fmt=out_fmt, transA=ta,
                                         transB=tb, act=act, slope=slope)
            got = decode(out[:, :N], out_fmt)
            cterm = np.abs(cin)
        else:
            rows, cols = sample_positions(M, N, sample, seed)
            exact, rounded = oracle.sample(rows, cols, K, A, B, lda=lda, ldb=ldb, C=C0, ldc=ldc,
                                           alpha=alpha, beta=beta, in_fmt=in_fmt, out_fmt=out_fmt,
                                           transA=ta, transB=tb, act=act, slope=slope)
            got = decode(out[rows, cols], out_fmt)
            cterm = np.abs(cin[rows, cols]) if beta != 0.0 else 0.0
        ref = decode(rounded, out_fmt)
        if act in (gemm.GEMM_ACT_GELU, gemm.GEMM_ACT_SILU):
            if sample is None:
                pre, _ = oracle.gemm(M, N, K, A, B, lda=lda, ldb=ldb, C=C0, ldc=ldc, alpha=alpha, beta=beta,
                                     in_fmt=in_fmt, out_fmt=out_fmt, transA=ta, transB=tb)
            else:
                pre, _ = oracle.sample(rows, cols, K, A, B, lda=lda, ldb=ldb, C=C0, ldc=ldc, alpha=alpha,
                                       beta=beta, in_fmt=in_fmt, out_fmt=out_fmt, transA=ta, transB=tb)
            tol = (1.1 * (1e-5 * K * amax * bmax * max(1.0, abs(alpha))
                          + 2.0 ** -21 * (np.abs(pre) + abs(beta) * cterm))
                   + 2.0 ** -20 * np.abs(exact) + ulp(exact, out_fmt))
        else:
            tol = (1e-5 * K * amax * bmax * max(1.0, abs(alpha))
                   + 2.0 ** -21 * (np.abs(exact) + abs(beta) * cterm) + ulp(exact, out_fmt))
        err = np.abs(got - ref)
        bad = ~(err <= tol)
        if bad.any():
            idx = np.argwhere(bad)[:5]
            raise AssertionError(
                f"{int(bad.sum())} of {bad.size} outputs off ({M}x{N}x{K} {in_fmt}->{out_fmt} "
                f"ta={ta} tb={tb} info={res.info}); first: " +
                "; ".join(f"{tuple(i)} gpu={got[tuple(i)]!r} oracle={ref[tuple(i)]!r} tol={np.broadcast_to(tol, bad.shape)[tuple(i)]:.3g}" for i in idx))
        res.max_err = float(err.max()) if err.size else 0.0
        return res
    finally:
        for k, v in old_env.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


TYPES = {"bf16": gemm.GEMM_TYPE_BF16, "f16": gemm.GEMM_TYPE_F16, "f32": gemm.GEMM_TYPE_F32,
         "tf32": gemm.GEMM_TYPE_TF32}


def run_case_ex(plan, M, N, K, in_fmt="bf16", c_fmt="f32", d_fmt="bf16", ta=False, tb=False, alpha=1.0,
                beta=0.5, act=0, slope=0.0, seed=1, pad=(0, 0, 0, 0), sample=None, env=None, c_none=False):
    """gemm_run_ex with a separate C (c_fmt, row stride ldc) and output D
    (d_fmt, ldd): D is compared with the oracle as run_case compares C, C
    must come back bitwise unchanged, and D's row padding (NaN sentinels)
    must not be written."""
    import torch
    old_env = {}
    for k, v in (env or {}).items():
        old_env[k] = os.environ.get(k)
        os.environ[k] = v
    try:
        a_rows, a_cols = (K, M) if ta else (M, K)
        b_rows, b_cols = (N, K) if tb else (K, N)
        ie = ESIZE[in_fmt]
        lda = round_up(max(a_cols, 1), 16 // ie) + pad[0]
        ldb = round_up(max(b_cols, 1), 16 // ie) + pad[1]
        ldc = max(N, 1) + pad[2]                       # a separate C needs no 16-byte rows
        ldd = round_up(max(N, 1), 16 // ESIZE[d_fmt]) + pad[3]
        A = inputs.matrix(a_rows, a_cols, seed, inputs.TENSOR_A, in_fmt, ld=lda)
        B = inputs.matrix(b_rows, b_cols, seed, inputs.TENSOR_B, in_fmt, ld=ldb)
        C0 = inputs.matrix(M, N, seed, inputs.TENSOR_C, c_fmt, ld=ldc)
        nan = {"bf16": inputs.BF16_NAN, "f16": inputs.F16_NAN, "f32": np.float32(np.nan)}[d_fmt]
        D0 = np.full((M, ldd), nan, dtype=np.float32 if d_fmt == "f32" else np.uint16)
        Ad, Bd, Cd, Dd = (to_device(A, in_fmt), to_device(B, in_fmt), to_device(C0, c_fmt),
                          to_device(D0, d_fmt))
        stream = torch.cuda.current_stream().cuda_stream
        st = gemm.gemm_run_ex(plan.handle, M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb,
                              None if c_none else Cd.data_ptr(), ldc, TYPES[c_fmt], Dd.data_ptr(), ldd,
                              TYPES[d_fmt], alpha, beta, TYPES[in_fmt], int(ta), int(tb), act, slope, stream)
        assert st == gemm.GEMM_OK, gemm.gemm_status_string(st)
        torch.cuda.synchronize()
        assert plan.poll_error() == gemm.GEMM_OK, "watchdog fired"
        res = Result()
        res.info = plan.last_config()
        C_after = from_device(Cd, c_fmt).reshape(M, ldc)
        assert np.array_equal(C_after.view(np.uint8), C0.view(np.uint8)), "C was modified"
        D = from_device(Dd, d_fmt).reshape(M, ldd)
        if ldd > N:
            assert np.array_equal(D[:, N:].view(np.uint8), D0[:, N:].view(np.uint8)), "D padding written"
        a_dec = decode(A[:, :a_cols], in_fmt)
        b_dec = decode(B[:, :b_cols], in_fmt)
        amax = float(np.abs(a_dec).max()) if a_dec.size else 0.0
        bmax = float(np.abs(b_dec).max()) if b_dec.size else 0.0
        kw = dict(lda=lda, ldb=ldb, C=C0, ldc=ldc, alpha=alpha, beta=beta, in_fmt=in_fmt, out_fmt=d_fmt,
                  c_fmt=c_fmt, transA=ta, transB=tb)
        if sample is None:
            exact, rounded = oracle.gemm(M, N, K, A, B, act=act, slope=slope, **kw)
            pre, _ = oracle.gemm(M, N, K, A, B, **kw)
            got = decode(D[:, :N], d_fmt)
            cterm = np.abs(decode(C0[:, :N], c_fmt))
        else:
            rows, cols = sample_positions(M, N, sample, seed)
            exact, rounded = oracle.sample(rows, cols, K, A, B, act=act, slope=slope, **kw)
            pre, _ = oracle.sample(rows, cols, K, A, B, **kw)
            got = decode(D[rows, cols], d_fmt)
            cterm = np.abs(decode(C0[rows, cols], c_fmt))
        ref = decode(rounded, d_fmt)
        lip = 1.1 if act in (gemm.GEMM_ACT_GELU, gemm.GEMM_ACT_SILU) else 1.0
        tol = (lip * (1e-5 * K * amax * bmax * max(1.0, abs(alpha)) + 2.0 ** -21 * (np.abs(pre) + abs(beta) * cterm))
               + 2.0 ** -20 * np.abs(exact) + ulp(exact, d_fmt))
        err = np.abs(got - ref)
        bad = ~(err <= tol)
        if bad.any():
            idx = np.argwhere(bad)[:5]
            raise AssertionError(
                f"{int(bad.sum())} of {bad.size} outputs off ({M}x{N}x{K} {in_fmt}, C {c_fmt}, D {d_fmt}, "
                f"info={res.info}); first: " +
                "; ".join(f"{tuple(i)} gpu={got[tuple(i)]!r} oracle={ref[tuple(i)]!r}" for i in idx))
        return res
    finally:
        for k, v in old_env.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
