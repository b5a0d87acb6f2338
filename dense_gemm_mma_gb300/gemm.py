"""ctypes binding of libdgemm_gb300.so (include/gemm.h).

Argument marshalling only: every function here forwards to the C entry point
of the same name; the torch helpers at the bottom turn tensors into pointers,
leading dimensions and flags.  There is no fallback: if the shared library is
missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
# GEMM_DEBUG=1 in the environment (read at the first load) selects the debug
# build: device-side bounds and copy-rule checks (include/gemm.h, gemm_debug_build).
LIB_PATH = os.path.join(_PKG, "libdgemm_gb300_debug.so" if os.environ.get("GEMM_DEBUG") == "1"
                        else "libdgemm_gb300.so")

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_ALIGNMENT = 2
GEMM_ERR_UNSUPPORTED = 3
GEMM_ERR_NO_DEVICE = 4
GEMM_ERR_OUT_OF_MEMORY = 5
GEMM_ERR_CUDA = 6
GEMM_ERR_TIMEOUT = 7
GEMM_ERR_DEBUG_CHECK = 8
# bits of the plan's error word (gemm_plan_last_error_bits)
DBG_FLAG = 1 << 30
DBG_SITES = {0: "tma", 1: "epilogue_store", 2: "epilogue_load", 3: "split_in_kernel", 4: "tile_reduce",
             5: "gemv", 6: "scale", 7: "transpose"}

GEMM_OP_N, GEMM_OP_T = 0, 1
GEMM_TYPE_BF16, GEMM_TYPE_F16, GEMM_TYPE_F32, GEMM_TYPE_TF32 = 0, 1, 2, 3
GEMM_BF16_F32, GEMM_BF16_BF16, GEMM_F16_F32, GEMM_F16_F16, GEMM_TF32_F32 = 0, 1, 2, 3, 4
GEMM_ACT_NONE, GEMM_ACT_LEAKY_RELU, GEMM_ACT_RELU, GEMM_ACT_GELU, GEMM_ACT_SILU = 0, 1, 2, 3, 4

PATH_NAMES = {0: "none", 1: "tc", 2: "tc_splitk", 3: "gemv_rowdot", 4: "gemv_colstream",
              5: "gemv_generic", 6: "scale", 7: "tc_splitk_cluster", 8: "tc_tail_split"}

DTYPES = {("bf16", "f32"): GEMM_BF16_F32, ("bf16", "bf16"): GEMM_BF16_BF16,
          ("f16", "f32"): GEMM_F16_F32, ("f16", "f16"): GEMM_F16_F16, ("tf32", "f32"): GEMM_TF32_F32}


class gemm_epilogue_t(ctypes.Structure):
    _fields_ = [("act", ctypes.c_int32), ("slope", ctypes.c_float)]


class gemm_config_info_t(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int32), ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
        ("tile_k", ctypes.c_int32), ("cta_per_tile", ctypes.c_int32), ("splitk", ctypes.c_int32),
        ("stages", ctypes.c_int32), ("raster_group", ctypes.c_int32), ("grid", ctypes.c_int32),
        ("sms", ctypes.c_int32), ("tiles", ctypes.c_int64), ("units", ctypes.c_int64),
        ("waves", ctypes.c_double), ("tail_fraction", ctypes.c_double),
        ("useful_fraction", ctypes.c_double), ("launches", ctypes.c_int32),
        ("tail_tiles", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64),
    ]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["path"] = PATH_NAMES.get(self.path, str(self.path))
        return d


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gemm_status_string(status)}")


_lib = None

# name -> (restype, argtypes)
_I64, _VP, _F, _I32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int32
_SIGNATURES = {
    "gemm_plan_create": (_I32, [ctypes.POINTER(_VP), ctypes.c_int]),
    "gemm_run": (_I32, [_VP, _I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64, _F, _F,
                        _I32, _I32, _I32, gemm_epilogue_t, _VP]),
    "gemm_plan_destroy": (_I32, [_VP]),
    "gemm_status_string": (ctypes.c_char_p, [_I32]),
    "gemm_plan_last_config": (_I32, [_VP, ctypes.POINTER(gemm_config_info_t)]),
    "gemm_plan_poll_error": (_I32, [_VP, _VP]),
    "gemm_plan_set_watchdog": (_I32, [_VP, ctypes.c_uint64]),
    "gemm_plan_selftest_watchdog": (_I32, [_VP, _VP]),
    "gemm_check_args": (_I32, [_I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64, _F,
                               _I32, _I32, _I32, gemm_epilogue_t]),
    "gemm_choose_config": (_I32, [_I64, _I64, _I64, _I32, _I32, _I32, _I32,
                                  ctypes.POINTER(gemm_config_info_t)]),
    "gemm_quantization": (_I32, [_I64, _I64, _I32, _I32, _I32, _I32, _I32,
                                 ctypes.POINTER(gemm_config_info_t)]),
    "gemm_gemv_noalloc": (_I32, [_I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64, _F, _F,
                                 _I32, _I32, _I32, gemm_epilogue_t, _VP]),
    "gemm_plan_set_autotune": (_I32, [_VP, ctypes.c_int]),
    "gemm_run_ex": (_I32, [_VP, _I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64, _I32, _VP, _I64, _I32,
                           _F, _F, _I32, _I32, _I32, gemm_epilogue_t, _VP]),
    "gemm_check_args_ex": (_I32, [_I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64, _I32, _VP, _I64, _I32,
                                  _F, _F, _I32, _I32, _I32, gemm_epilogue_t]),
    "gemm_plan_tuned_count": (_I32, [_VP, ctypes.POINTER(_I64)]),
    "gemm_plan_last_error_bits": (_I32, [_VP, ctypes.POINTER(_I64)]),
    "gemm_debug_build": (ctypes.c_int, []),
}


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the shared library (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is None:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is not built; run __graft_entry__.build() "
                               "(python -m dense_gemm_mma_gb300.build)")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_symbols() -> list[str]:
    return list(_SIGNATURES)


# ---------------------------------------------------------------- C entry points

def gemm_status_string(status: int) -> str:
    return load().gemm_status_string(status).decode()


def gemm_plan_create(device: int = 0) -> int:
    h = _VP()
    st = load().gemm_plan_create(ctypes.byref(h), device)
    if st != GEMM_OK:
        raise GemmError(st, "gemm_plan_create")
    return h.value


def gemm_plan_destroy(plan: int) -> int:
    return load().gemm_plan_destroy(plan)


def gemm_run(plan, M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, dtype, transA, transB,
             act=GEMM_ACT_NONE, slope=0.0, stream=None) -> int:
    return load().gemm_run(plan, M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, dtype,
                           transA, transB, gemm_epilogue_t(act, slope), stream)


def gemm_run_ex(plan, M, N, K, A, lda, B, ldb, C, ldc, c_type, D, ldd, d_type, alpha, beta, ab_type,
                transA, transB, act=GEMM_ACT_NONE, slope=0.0, stream=None) -> int:
    return load().gemm_run_ex(plan, M, N, K, A, lda, B, ldb, C, ldc, c_type, D, ldd, d_type, alpha, beta,
                              ab_type, transA, transB, gemm_epilogue_t(act, slope), stream)


def gemm_check_args_ex(M, N, K, A, lda, B, ldb, C, ldc, c_type, D, ldd, d_type, alpha, beta, ab_type,
                       transA, transB, act=GEMM_ACT_NONE, slope=0.0) -> int:
    return load().gemm_check_args_ex(M, N, K, A, lda, B, ldb, C, ldc, c_type, D, ldd, d_type, alpha, beta,
                                     ab_type, transA, transB, gemm_epilogue_t(act, slope))


def gemm_plan_last_config(plan) -> gemm_config_info_t:
    info = gemm_config_info_t()
    st = load().gemm_plan_last_config(plan, ctypes.byref(info))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_plan_last_config")
    return info


def gemm_plan_poll_error(plan, stream=None) -> int:
    return load().gemm_plan_poll_error(plan, stream)


def gemm_plan_last_error_bits(plan) -> int:
    v = _I64()
    st = load().gemm_plan_last_error_bits(plan, ctypes.byref(v))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_plan_last_error_bits")
    return v.value


def gemm_debug_build() -> int:
    return load().gemm_debug_build()


def debug_sites(bits: int) -> list[str]:
    """Names of the debug-build check sites set in an error word."""
    return [name for s, name in DBG_SITES.items() if bits & (1 << (16 + s))]


def gemm_plan_set_watchdog(plan, timeout_ns: int) -> int:
    return load().gemm_plan_set_watchdog(plan, timeout_ns)


def gemm_plan_selftest_watchdog(plan, stream=None) -> int:
    return load().gemm_plan_selftest_watchdog(plan, stream)


def gemm_check_args(M, N, K, A, lda, B, ldb, C, ldc, alpha, dtype, transA, transB,
                    act=GEMM_ACT_NONE, slope=0.0) -> int:
    return load().gemm_check_args(M, N, K, A, lda, B, ldb, C, ldc, alpha, dtype, transA,
                                  transB, gemm_epilogue_t(act, slope))


def gemm_choose_config(M, N, K, dtype, transA, transB, sms) -> gemm_config_info_t:
    info = gemm_config_info_t()
    st = load().gemm_choose_config(M, N, K, dtype, transA, transB, sms, ctypes.byref(info))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_choose_config")
    return info


def gemm_quantization(M, N, tile_m, tile_n, splitk, sms, ctas_per_sm=1) -> gemm_config_info_t:
    info = gemm_config_info_t()
    st = load().gemm_quantization(M, N, tile_m, tile_n, splitk, sms, ctas_per_sm,
                                  ctypes.byref(info))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_quantization")
    return info


def gemm_gemv_noalloc(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, dtype, transA, transB,
                      act=GEMM_ACT_NONE, slope=0.0, stream=None) -> int:
    return load().gemm_gemv_noalloc(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, dtype,
                                    transA, transB, gemm_epilogue_t(act, slope), stream)


def gemm_plan_set_autotune(plan, enable: bool) -> int:
    return load().gemm_plan_set_autotune(plan, int(bool(enable)))


def gemm_plan_tuned_count(plan) -> int:
    n = _I64()
    st = load().gemm_plan_tuned_count(plan, ctypes.byref(n))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_plan_tuned_count")
    return n.value


# ------------------------------------------------------------------ torch helpers

def _operand(t, trans: bool):
    """(pointer, ld) of a stored 2-D operand whose rows are contiguous."""
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("operands must be 2-D with contiguous rows")
    return t.data_ptr(), max(t.stride(0), t.shape[1], 1)


class Plan:
    """Owns a gemm_plan_t on one device."""

    def __init__(self, device: int = 0):
        self.handle = gemm_plan_create(device)

    def close(self):
        if self.handle:
            gemm_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def run(self, A, B, C, *, alpha=1.0, beta=0.0, transA=False, transB=False,
            act=GEMM_ACT_NONE, slope=0.0, stream=None, M=None, N=None, K=None) -> int:
        """C <- act(alpha*op(A)@op(B) + beta*C) on torch tensors holding the
        STORED matrices (A is K x M when transA, B is N x K when transB)."""
        import torch
        # fp32 operands are read as TF32 by the tensor cores (GEMM_TF32_F32)
        in_t = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "tf32"}[A.dtype]
        out_t = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[C.dtype]
        if B.dtype != A.dtype:
            raise ValueError("A and B must have the same dtype")
        dtype = DTYPES[(in_t, out_t)]
        a, lda = _operand(A, transA)
        b, ldb = _operand(B, transB)
        c, ldc = _operand(C, False)
        M = C.shape[0] if M is None else M
        N = C.shape[1] if N is None else N
        K = (A.shape[0] if transA else A.shape[1]) if K is None else K
        if stream is None:
            stream = torch.cuda.current_stream(C.device).cuda_stream
        return gemm_run(self.handle, M, N, K, a, lda, b, ldb, c, ldc, alpha, beta, dtype,
                        int(transA), int(transB), act, slope, stream)

    def last_config(self) -> dict:
        return gemm_plan_last_config(self.handle).as_dict()

    def poll_error(self, stream=None) -> int:
        return gemm_plan_poll_error(self.handle, stream)
