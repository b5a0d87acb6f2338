"""CPU tests of the product's host logic: the C ABI loads and exports what
include/gemm.h declares, argument checks, the tile/wave quantization
arithmetic against the figures printed in "Matrix Multiplication Background
User's Guide" sections 2 and 3, the planner's invariants, and the FLOP/byte
accounting of the benchmark."""
import json
import os
import re

import pytest

from dense_gemm_mma_gb300 import gemm as g
from dense_gemm_mma_gb300 import roofline as rl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FIG = json.load(open(os.path.join(ROOT, "tests", "golden", "guide_figures.json")))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    import __graft_entry__
    __graft_entry__.build_library()
    g.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gemm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    import ctypes
    lib = g.load()
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(g.exported_symbols()) == names
    # nothing else is exported under the gemm_ prefix
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", g.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = sorted(set(re.findall(r" T (gemm_\w+)", out)))
    assert exported == names
    assert isinstance(ctypes.sizeof(g.gemm_config_info_t), int)
    assert ctypes.sizeof(g.gemm_config_info_t) == 96


def test_status_strings():
    for s in range(9):
        assert g.gemm_status_string(s).startswith("GEMM_")
    assert "debug" in g.gemm_status_string(g.GEMM_ERR_DEBUG_CHECK)
    assert "unknown" in g.gemm_status_string(99)


def test_debug_build_exports_the_same_symbols():
    """The debug build (device-side checks) is the same C ABI: the same
    exported gemm_* functions; gemm_debug_build tells the two apart."""
    import ctypes
    import subprocess
    from dense_gemm_mma_gb300 import build as b
    path = b.build(debug=True)
    assert path.endswith("libdgemm_gb300_debug.so")
    names = declared_functions()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    assert sorted(set(re.findall(r" T (gemm_\w+)", out))) == names
    dbg = ctypes.CDLL(path)  # loaded beside the release library: no call touches a device
    assert dbg.gemm_debug_build() == 1
    assert g.gemm_debug_build() == 0
    assert g.debug_sites(g.DBG_FLAG | (1 << 17) | (1 << 21)) == ["epilogue_store", "gemv"]


def test_no_device_without_gpu():
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    with pytest.raises(g.GemmError) as e:
        g.gemm_plan_create(0)
    assert e.value.status == g.GEMM_ERR_NO_DEVICE
    assert g.load().gemm_run(None, 4, 4, 4, 16, 8, 16, 8, 16, 8, 1.0, 0.0, 0, 0, 0,
                             g.gemm_epilogue_t(0, 0.0), None) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_plan_destroy(None) == g.GEMM_OK


# -------------------------------------------------------------- argument checks

A16, B16, C16 = 1 << 32, 2 << 32, 3 << 32   # fake, 16-byte aligned, 4 GiB apart (never dereferenced)


def chk(M, N, K, A=A16, lda=None, B=B16, ldb=None, C=C16, ldc=None, alpha=1.0, dtype=0,
        ta=0, tb=0, act=0):
    lda = lda if lda is not None else max(1, (M if ta else K))
    ldb = ldb if ldb is not None else max(1, (K if tb else N))
    ldc = ldc if ldc is not None else max(1, N)
    return g.gemm_check_args(M, N, K, A, lda, B, ldb, C, ldc, alpha, dtype, ta, tb, act)


def test_check_args_accepts_good_calls():
    assert chk(512, 512, 512) == g.GEMM_OK
    assert chk(8192, 128, 8192, tb=1) == g.GEMM_OK
    assert chk(24, 40, 16, ta=1, tb=1, dtype=3) == g.GEMM_OK


def test_check_args_ex_separate_c():
    """gemm_run_ex: D keeps gemm_run's rules for C; a separate C needs its
    element alignment, may be NULL only with beta == 0, and must not overlap D."""
    T16, TF, TH = g.GEMM_TYPE_BF16, g.GEMM_TYPE_F32, g.GEMM_TYPE_F16
    OK, E, AL = g.GEMM_OK, g.GEMM_ERR_INVALID_ARG, g.GEMM_ERR_ALIGNMENT
    A, B = 0x100000, 0x200000
    D, C = 0x400000, 0x800000            # 16-byte aligned, far apart

    def ex(M=64, N=64, K=64, c=C, ldc=64, c_type=TF, d=D, ldd=64, d_type=T16, beta=0.5, ab=T16):
        return g.gemm_check_args_ex(M, N, K, A, K, B, N, c, ldc, c_type, d, ldd, d_type, 1.0, beta, ab, 0, 0)
    assert ex() == OK                                        # fp32 C in, bf16 D out
    assert ex(c_type=TH) == OK and ex(c_type=T16) == OK      # any C type
    assert ex(c=None, beta=0.0) == OK                        # C unused
    assert ex(c=None) == E                                   # beta != 0 needs C
    assert ex(ldc=32) == E                                   # ldc < N
    assert ex(c=C + 2) == AL and ex(c=C + 4) == OK           # fp32 C: 4-byte alignment only
    assert ex(d=D + 4) == AL                                 # D: 16 bytes on the tensor-core path
    assert ex(d_type=TH) == E                                # 16-bit D must be the operand type
    assert ex(d_type=TF) == OK
    assert ex(ab=TF) == E                                    # fp32 operands: not a dtype of this library
    assert ex(c=D, c_type=T16) == OK                         # in place: same matrix
    assert ex(c=D, c_type=TF) == E and ex(c=D, c_type=T16, ldc=72) == E
    assert ex(c=D + 64 * 64) == E                            # overlaps D (D spans 64*64*2 bytes)
    assert ex(c=D + 64 * 64 * 2) == OK                       # right after D


def test_check_args_rejects_output_overlapping_operands():
    """C is written while A and B are read: a C that shares a byte with A or B
    is rejected before any launch (gemm_run), and so is a D of gemm_run_ex that
    shares one with A or B.  Slices of one parent whose rows interleave without
    sharing a byte are accepted."""
    E, OK = g.GEMM_ERR_INVALID_ARG, g.GEMM_OK
    M, N, K = 64, 32, 128                      # A 64 x 128 bf16 (16 KiB), B 128 x 32 (8 KiB), C fp32 8 KiB
    a_bytes, b_bytes = M * K * 2, K * N * 2
    assert chk(M, N, K) == OK
    assert chk(M, N, K, C=A16 + 4096) == E                     # C inside A
    assert chk(M, N, K, C=B16 + 1024) == E                     # C inside B
    assert chk(M, N, K, C=A16 + a_bytes - 16) == E             # C straddles the end of A
    assert chk(M, N, K, C=A16 - 16) == E                       # C's last row runs into A's first
    assert chk(M, N, K, C=A16 + a_bytes) == OK                 # right after A
    assert chk(M, N, K, C=B16 - M * N * 4) == OK               # right before B
    for ta in (0, 1):                                          # stored K x M when transposed
        for tb in (0, 1):
            assert chk(M, N, K, ta=ta, tb=tb) == OK
            assert chk(M, N, K, ta=ta, tb=tb, C=A16 + a_bytes // 2) == E
            assert chk(M, N, K, ta=ta, tb=tb, C=B16 + b_bytes // 2) == E
            assert chk(M, N, K, ta=ta, tb=tb, C=A16 + a_bytes) == OK
    # A and C as column slices of one parent with 256 fp32-sized... (bf16 parent,
    # ld 512 elements = 1 KiB rows): A in bytes [0, 256) of every row, C (bf16 out)
    # in bytes [512, 576): rows interleave, no byte is shared
    P, ld = A16, 512
    assert chk(M, N, K, A=P, lda=ld, C=P + 512, ldc=ld, dtype=1) == OK
    assert chk(M, N, K, A=P, lda=ld, C=P + 240, ldc=ld, dtype=1) == E      # C's rows start inside A's
    assert chk(M, N, K, A=P, lda=ld, C=P + 1024 - 64, ldc=ld, dtype=1) == OK  # ends where A's next row starts
    assert chk(M, N, K, A=P, lda=ld, C=P + 1024 - 62, ldc=ld, dtype=1) == E   # ... two bytes into it
    # different leading dimensions: C's rows (ld 64 bf16 = 128 B) walk across A's (1 KiB apart)
    assert chk(M, N, K, A=P, lda=ld, C=P + 256, ldc=64, dtype=1) == E
    assert chk(2, N, K, A=P, lda=ld, C=P + 256, ldc=64, dtype=1) == OK       # two C rows in A's gap
    # nothing of A or B is read: no rule (K == 0, alpha == 0)
    assert chk(M, N, 0, C=A16) == OK
    assert chk(M, N, K, C=A16, alpha=0.0) == OK
    # gemm_run_ex: D against A and B
    T16, TF = g.GEMM_TYPE_BF16, g.GEMM_TYPE_F32

    def ex(d, c=None, beta=0.0):
        return g.gemm_check_args_ex(M, N, K, A16, K, B16, N, c, N, TF, d, N, TF, 1.0, beta, T16, 0, 0)
    assert ex(C16) == OK
    assert ex(A16 + 1024) == E and ex(B16 + 1024) == E
    assert ex(C16, c=A16, beta=1.0) == OK     # a separate C may overlap A: both are only read


def test_check_args_rejects():
    E, AL, U = g.GEMM_ERR_INVALID_ARG, g.GEMM_ERR_ALIGNMENT, g.GEMM_ERR_UNSUPPORTED
    assert chk(-1, 8, 8) == E
    assert chk(8, -1, 8) == E
    assert chk(8, 8, -1) == E
    assert chk(8, 8, 8, dtype=5) == E
    assert chk(8, 8, 8, ta=2) == E
    assert chk(8, 8, 8, act=5) == E and chk(8, 8, 8, act=-1) == E
    for act in (g.GEMM_ACT_RELU, g.GEMM_ACT_GELU, g.GEMM_ACT_SILU):
        assert chk(8, 8, 8, act=act) == g.GEMM_OK
    assert chk(2 ** 31, 8, 8) == U
    assert chk(8, 8, 16, lda=8) == E                 # lda < K
    assert chk(8, 16, 8, ldb=8) == E                 # ldb < N
    assert chk(8, 16, 8, ldc=8) == E                 # ldc < N
    assert chk(16, 8, 8, ta=1, lda=8) == E           # transposed A: lda >= M
    assert chk(8, 16, 8, tb=1, ldb=4) == E           # transposed B: ldb >= K
    assert chk(8, 8, 8, C=0) == E
    assert chk(8, 8, 8, A=0) == E
    assert chk(8, 8, 8, B=0) == E
    assert chk(8, 8, 8, A=A16 + 2) == AL             # tensor-core path: 16-byte pointers
    assert chk(8, 8, 8, C=C16 + 8) == AL
    assert chk(8, 8, 12, lda=12) == AL               # lda * 2 not a multiple of 16
    assert chk(8, 12, 8, ldc=12, dtype=1) == AL      # bf16 C: ldc * 2
    assert chk(8, 8, 8, A=A16 + 1) == AL             # not even element-aligned
    assert chk(8, 8, 8, C=C16 + 2) == AL             # fp32 C needs 4-byte alignment


def test_check_args_degenerate_and_gemv_relaxations():
    assert chk(0, 8, 8, A=0, B=0, C=0) == g.GEMM_OK          # nothing to do
    assert chk(8, 0, 8, A=0, B=0, C=0) == g.GEMM_OK
    assert chk(8, 8, 0, A=0, B=0) == g.GEMM_OK               # C <- beta*C, A/B unused
    assert chk(8, 8, 8, A=0, B=0, alpha=0.0) == g.GEMM_OK    # alpha == 0: A/B unused
    # GEMV: vectors need only element alignment, strides are free
    assert chk(1, 100, 7, A=A16 + 2, ldb=100) == g.GEMM_OK
    assert chk(100, 1, 7, B=B16 + 2, ldb=1, lda=7, ldc=3, C=C16 + 4) == g.GEMM_OK


# --------------------------------------------------- tile / wave quantization pins

def test_wave_quantization_matches_guide_fig8():
    w = FIG["wave_quantization"]
    tm, tn = w["tile"]
    for case in w["cases"]:
        q = g.gemm_quantization(w["M"], case["N"], tm, tn, 1, w["sms"])
        assert q.tiles == case["tiles"] == w["m_tiles"] * case["n_tiles"]
        assert int(q.waves) == case["full_waves"]
        tail = q.units % w["sms"]
        assert tail == case["tail_tiles"]
        if "tail_percent" in case:
            assert round(100 * q.tail_fraction, 2) == case["tail_percent"]
    for n in w["full_wave_N"]:
        full = g.gemm_quantization(w["M"], n, tm, tn, 1, w["sms"])
        after = g.gemm_quantization(w["M"], n + 8, tm, tn, 1, w["sms"])
        assert full.tail_fraction == 0.0 and full.waves == int(full.waves)
        assert after.tail_fraction > 0.0           # a new wave starts right after


def test_tile_quantization_matches_guide_fig7_and_fig6():
    t = FIG["tile_quantization"]
    tm, tn = t["tile"]
    for n in range(t["N_from"], t["N_to"] + 1, t["N_step"]):
        q = g.gemm_quantization(t["M"], n, tm, tn, 1, 108)
        assert q.tiles == (t["M"] // tm) * t["n_tiles"]
    assert g.gemm_quantization(t["M"], 128, tm, tn, 1, 108).tiles == (t["M"] // tm) * t["n_tiles_at_128"]
    q136 = g.gemm_quantization(t["M"], 136, tm, tn, 1, 108)
    second_tile_useful = (136 - tn) / tn
    assert round(100 * second_tile_useful, 2) == t["second_tile_useful_percent_at_136"]
    assert q136.useful_fraction == pytest.approx(136 / 256)
    f = FIG["fig6"]
    best = g.gemm_quantization(*f["best"], *f["tile"], 1, 108)
    worst = g.gemm_quantization(*f["worst"], *f["tile"], 1, 108)
    assert best.tiles == f["tiles_best"] and worst.tiles == f["tiles_worst"]
    assert worst.tiles / best.tiles == f["math_ratio"]
    extra = (f["worst"][0] * f["worst"][1]) / (f["best"][0] * f["best"][1]) - 1
    assert round(100 * extra, 2) == f["extra_useful_percent"]


def test_arithmetic_intensity_matches_guide_section2():
    a = FIG["arithmetic_intensity"]
    for c in a["cases"]:
        ai = rl.intensity(c["M"], c["N"], c["K"], c["fmt"], c["fmt"])
        assert round(ai, c["decimals"]) == c["value"] or int(ai) == c["value"]
        on_v100 = "math" if ai > a["v100_ops_per_byte"] else "memory"
        assert on_v100 == c["bound_on_v100"]
    # GEMV intensity stays below 1 FLOP/B
    assert rl.intensity(1, 8192, 8192, "f16", "f16") < a["gemv_intensity_below"]
    assert rl.intensity(8192, 1, 8192, "bf16", "f32") < a["gemv_intensity_below"]


def test_tflops_formula_matches_t4_benchmark():
    t = FIG["t4_benchmark"]
    v = rl.tflops(rl.gemm_flops(t["M"], t["N"], t["K"]), t["median_latency_ms"] / 1e3)
    assert abs(v - t["tflops"]) <= t["tflops_std"]
    assert round(v, 2) == round(t["tflops"], 2)


def test_roofline_bound():
    assert rl.bound(rl.intensity(8192, 8192, 8192, "bf16", "bf16"), 2.25e15, 8e12) == "tensor"
    assert rl.bound(rl.intensity(8192, 128, 8192, "bf16", "f32"), 2.25e15, 8e12) == "hbm"
    assert rl.attainable(100.0, 2.25e15, 8e12) == 8e14


# ----------------------------------------------------------------------- planner

@pytest.mark.parametrize("M,N,K", [(512, 512, 512), (8192, 8192, 8192), (8192, 128, 8192),
                                   (6912, 2048, 4096), (27648, 136, 4096), (2304, 1544, 4096),
                                   (256, 256, 65536), (2, 2, 1), (129, 257, 10000)])
def test_planner_invariants(M, N, K):
    for sms in (108, 148, 152):
        c = g.gemm_choose_config(M, N, K, g.GEMM_BF16_F32, 0, 0, sms)
        assert c.path in (1, 2, 7, 8)
        assert (c.tile_m, c.cta_per_tile) in ((128, 1), (256, 2), (128, 2))
        assert (c.tile_m, c.cta_per_tile) != (128, 2) or (c.path == 7 and c.splitk == 2)
        assert c.tile_n in (64, 128, 256) and c.tile_k == 64
        assert 1 <= c.grid <= sms and c.grid <= c.units * c.cta_per_tile
        assert c.grid % c.cta_per_tile == 0
        slots = sms // 2 if c.tile_m == 256 else sms
        if c.path == 8:       # whole tiles for the full waves, K slices for the last wave's tiles
            assert 0 < c.tail_tiles < slots and c.tiles >= slots
            assert c.tail_tiles == c.tiles % slots
            assert c.units == c.tiles - c.tail_tiles + c.tail_tiles * c.splitk
            assert c.tail_tiles * c.splitk <= slots
        elif c.path == 2:     # every tile split
            assert c.tail_tiles == c.tiles and c.units == c.tiles * c.splitk
        else:
            assert c.tail_tiles == 0 and c.units == c.tiles * c.splitk
        kb = -(-K // 64)
        assert 1 <= c.splitk <= kb
        per = -(-kb // c.splitk)
        assert -(-kb // per) == c.splitk                  # no empty K slice
        assert (c.path in (2, 7, 8)) == (c.splitk > 1)
        assert c.launches == (2 if c.path in (2, 8) else 1)
        assert c.workspace_bytes == c.tail_tiles * c.splitk * c.tile_m * c.tile_n * 4


def test_planner_splits_small_output_with_long_k():
    c = g.gemm_choose_config(256, 256, 65536, g.GEMM_F16_F32, 0, 0, 152)
    assert c.splitk > 1 and c.units >= 64
    big = g.gemm_choose_config(8192, 8192, 8192, g.GEMM_BF16_BF16, 0, 0, 152)
    assert big.tile_n == 256 and big.tile_m == 256 and big.cta_per_tile == 2
    assert big.path in (1, 8) and (big.path == 1) == (big.splitk == 1)


def test_planner_gemv_paths():
    assert g.PATH_NAMES[g.gemm_choose_config(1, 8192, 8192, 0, 0, 0, 152).path] == "gemv_colstream"
    assert g.PATH_NAMES[g.gemm_choose_config(1, 8192, 8192, 0, 0, 1, 152).path] == "gemv_rowdot"
    assert g.PATH_NAMES[g.gemm_choose_config(8192, 1, 8192, 0, 0, 0, 152).path] == "gemv_rowdot"
    assert g.PATH_NAMES[g.gemm_choose_config(8192, 1, 8192, 0, 1, 0, 152).path] == "gemv_colstream"
    assert g.PATH_NAMES[g.gemm_choose_config(0, 5, 5, 0, 0, 0, 152).path] == "none"
    assert g.PATH_NAMES[g.gemm_choose_config(5, 5, 0, 0, 0, 0, 152).path] == "scale"


def test_planner_forced_pair(monkeypatch):
    monkeypatch.setenv("GEMM_FORCE_TILE", "256x256")
    c = g.gemm_choose_config(1000, 1000, 1000, 0, 0, 0, 152)
    assert c.tile_m == 256 and c.tile_n == 256 and c.cta_per_tile == 2
    assert c.tiles == 4 * 4 and c.grid == 2 * c.units


def test_planner_tf32():
    """TF32: 32 K elements per 128-byte stage row, tensor-core path for every
    shape (GEMV shapes included)."""
    c = g.gemm_choose_config(8192, 8192, 8192, g.GEMM_TF32_F32, 0, 1, 152)
    assert c.tile_k == 32 and c.path in (1, 8)
    for shape in [(1, 4096, 4096), (4096, 1, 4096)]:
        c = g.gemm_choose_config(*shape, g.GEMM_TF32_F32, 0, 1, 152)
        assert c.path in (1, 2, 7, 8) and c.tile_k == 32
    ok = g.GEMM_OK
    chk = lambda *a, **k: g.gemm_check_args(*a, **k)
    A, B, C = 0x100000, 0x200000, 0x300000
    assert chk(64, 64, 64, A, 64, B, 64, C, 64, 1.0, g.GEMM_TF32_F32, 0, 1) == ok
    assert chk(64, 64, 62, A, 62, B, 62, C, 64, 1.0, g.GEMM_TF32_F32, 0, 1) == g.GEMM_ERR_ALIGNMENT  # ld % 4
    assert chk(64, 3, 64, A, 64, B, 64, C + 4, 5, 1.0, g.GEMM_TF32_F32, 0, 1) == ok   # N < 4: C 4-byte aligned
    assert chk(64, 64, 64, A, 64, B, 64, C, 64, 1.0, 5, 0, 1) == g.GEMM_ERR_INVALID_ARG


def test_planner_kpair_switch(monkeypatch):
    """GEMM_SPLITK_CLUSTER=1 takes the on-chip two-slice reduction (a cluster
    of two CTAs per 128-row tile, one launch); =0 never does."""
    monkeypatch.setenv("GEMM_SPLITK_CLUSTER", "1")
    c = g.gemm_choose_config(1024, 1024, 4096, 0, 0, 0, 152)
    assert g.PATH_NAMES[c.path] == "tc_splitk_cluster"
    assert (c.tile_m, c.cta_per_tile, c.splitk, c.launches) == (128, 2, 2, 1)
    assert c.units == 2 * c.tiles and c.grid == 2 * min(c.tiles, 76)
    monkeypatch.setenv("GEMM_SPLITK_CLUSTER", "0")
    for shape in [(8192, 128, 8192), (8192, 256, 8192), (1024, 1024, 4096)]:
        assert g.gemm_choose_config(*shape, 0, 0, 0, 152).path in (1, 2)
    # K of one k-block cannot be halved: the switch is ignored
    monkeypatch.setenv("GEMM_SPLITK_CLUSTER", "1")
    c = g.gemm_choose_config(1024, 1024, 64, 0, 0, 0, 152)
    assert c.path in (1, 2) and c.splitk == 1


def test_planner_kpair_over_several_waves():
    """A K pair whose tiles take more than one wave of clusters is chosen only
    where the best other choice needs more than one wave too: 27648 x 128 x
    4096, where it measured faster on GB300, takes it; shapes where a one-wave
    tile measured faster keep that tile (1024 x 2048 x 1024: 14.7 us as 128
    one-CTA tiles against 16.4 us as 128 K-pair clusters)."""
    for shape in [(27648, 128, 4096)]:
        c = g.gemm_choose_config(*shape, 0, 0, 0, 152)
        assert g.PATH_NAMES[c.path] == "tc_splitk_cluster", shape
        assert c.tiles > 76 and c.waves > 1.0
    for shape in [(1536, 1536, 1536), (1280, 1280, 1280), (4096, 512, 4096), (2048, 1024, 4096),
                  (1024, 4096, 1024), (2048, 2048, 1024), (1024, 2048, 1024), (2048, 1024, 1024)]:
        c = g.gemm_choose_config(*shape, 0, 0, 0, 152)
        assert g.PATH_NAMES[c.path] == "tc" and c.waves <= 1.0, (shape, c.as_dict())


def test_gemv_colstream_grid_is_one_wave():
    """The column-stream GEMV's K split never asks for more CTAs than four per
    SM: a split rounded up left a few CTAs to run alone in a second wave
    (1 x 5000 x 8192: 610 CTAs for 608 slots)."""
    for sms in (152, 148, 132):
        for n in (5000, 8192, 3000, 16384, 777, 4096 + 512, 40000):
            for k in (8192, 4096, 1000):
                c = g.gemm_choose_config(1, n, k, 0, 0, 0, sms)
                assert g.PATH_NAMES[c.path] == "gemv_colstream"
                panels = -(-n // 512)
                assert c.grid <= max(4 * sms, panels), (sms, n, k, c.grid)
                assert c.grid == panels * c.splitk


def test_planner_tail_split(monkeypatch):
    """Config 5's second-wave shapes: 2304 x 2176 x 4096 has 81 tiles of
    256 x 256 for 76 CTA pairs, so 5 tiles would run alone in a second wave;
    the tail split runs 76 whole tiles and splits the 5 along K."""
    c = g.gemm_choose_config(2304, 2176, 4096, g.GEMM_F16_F32, 0, 0, 152)
    assert g.PATH_NAMES[c.path] == "tc_tail_split" and c.tiles == 81 and c.tail_tiles == 5
    assert c.units == 76 + 5 * c.splitk and c.launches == 2
    # a full last wave has no tail to split
    assert g.gemm_choose_config(2304, 1984, 4096, g.GEMM_F16_F32, 0, 0, 152).path == 1
    monkeypatch.setenv("GEMM_TAIL_SPLIT", "0")
    assert g.gemm_choose_config(2304, 2176, 4096, g.GEMM_F16_F32, 0, 0, 152).path != 8
    monkeypatch.setenv("GEMM_TAIL_SPLIT", "3")
    monkeypatch.setenv("GEMM_FORCE_TILE", "128x128")
    c = g.gemm_choose_config(300, 2000, 1000, g.GEMM_F16_F32, 0, 0, 20)
    assert c.path == 8 and c.splitk == 3 and c.tiles == 3 * 16 and c.tail_tiles == 48 % 20


def test_planner_log_lines():
    """GEMM_LOG=1 prints one line per planned call on stderr: the shape, the types,
    and the decisions (path, tile, split, grid, waves, tail, launches, workspace)."""
    import subprocess
    import sys
    code = ("from dense_gemm_mma_gb300 import gemm as g; "
            "g.gemm_choose_config(256, 256, 65536, g.GEMM_F16_F32, 0, 0, 152); "
            "g.gemm_choose_config(1, 8192, 8192, g.GEMM_BF16_F32, 0, 1, 152)")
    env = dict(os.environ, GEMM_LOG="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT)
    lines = [l for l in r.stderr.splitlines() if l.startswith("gemm_log")]
    assert len(lines) == 2, r.stderr
    assert "256x256x65536 f16->f32 op(A)=N op(B)=N -> tc_splitk tile 128x" in lines[0]
    assert "launches 2" in lines[0] and "workspace" in lines[0]
    assert "1x8192x8192 bf16->f32 op(A)=N op(B)=T -> gemv_rowdot" in lines[1]
    env.pop("GEMM_LOG")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT)
    assert "gemm_log" not in r.stderr


def test_fused_reduction_is_opt_in(monkeypatch):
    """GEMM_FUSED_REDUCE=1 sums K slices that all run at once inside the GEMM
    kernel (one launch); by default the tile reduction kernel does (two)."""
    c = g.gemm_choose_config(256, 256, 65536, g.GEMM_F16_F32, 0, 0, 152)
    assert c.path == 2 and c.launches == 2
    monkeypatch.setenv("GEMM_FUSED_REDUCE", "1")
    c = g.gemm_choose_config(256, 256, 65536, g.GEMM_F16_F32, 0, 0, 152)
    assert c.path == 2 and c.launches == 1 and c.tail_tiles * c.splitk <= c.grid // c.cta_per_tile
    # more slices than CTAs: the reduction kernel all the same
    monkeypatch.setenv("GEMM_FORCE_SPLITK", "64")
    monkeypatch.setenv("GEMM_FORCE_TILE", "128x64")
    c = g.gemm_choose_config(256, 256, 65536, g.GEMM_F16_F32, 0, 0, 152)
    assert c.units > 152 and c.launches == 2


def test_planner_env_overrides(monkeypatch):
    monkeypatch.setenv("GEMM_FORCE_TILE", "128x128")
    monkeypatch.setenv("GEMM_FORCE_SPLITK", "4")
    c = g.gemm_choose_config(1024, 1024, 4096, 0, 0, 0, 152)
    assert c.tile_n == 128 and c.splitk == 4
    monkeypatch.setenv("GEMM_RASTER_GROUP", "3")
    assert g.gemm_choose_config(1024, 1024, 4096, 0, 0, 0, 152).raster_group == 3


# (M, N, K, dtype) -> (path, tile_m, tile_n, splitk): the planner's pick on 152
# SMs, each timed on GB300 against the earlier model's pick in alternating
# processes (L2 flushed, means of 30 calls) and faster by the margin noted.
MEASURED_PICKS = [
    ((12288, 128, 8192, 0), ("tc", 128, 128, 1)),              # 59.1 -> 45.4 us
    ((7680, 512, 12288, 0), ("tc", 256, 256, 1)),              # 86.0 -> 66.2 us
    ((11264, 256, 8192, 0), ("tc", 256, 256, 1)),              # 59.5 -> 47.8 us
    ((24576, 64, 8192, 0), ("tc_tail_split", 128, 64, 3)),    # 89.3 -> 73.1 us
    ((19456, 64, 8192, 0), ("tc", 128, 64, 1)),               # 62.4 -> 56.1 us
    ((1152, 4096, 4096, 2), ("tc", 128, 256, 1)),             # 41.8 -> 33.9 us
    ((8192, 128, 8192, 0), ("tc_splitk_cluster", 128, 128, 2)),
    ((256, 256, 65536, 2), ("tc_splitk", 128, 128, 32)),
]


@pytest.mark.parametrize("shape,pick", MEASURED_PICKS, ids=["x".join(map(str, s[:3])) for s, _ in MEASURED_PICKS])
def test_planner_keeps_the_measured_picks(shape, pick):
    M, N, K, dt = shape
    c = g.gemm_choose_config(M, N, K, dt, 0, 0, 152)
    assert (g.PATH_NAMES[c.path], c.tile_m, c.tile_n, c.splitk) == pick, c.as_dict()
