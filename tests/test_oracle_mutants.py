"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a scratch copy of oracle.c (never in the
committed source), builds it on the CPU, and checks that at least one pin of
tests/test_oracle.py fails against the planted copy.  The pins run in a child
process, so a planted out-of-bounds read that crashes also counts as caught.
"""
import importlib.util
import inspect
import json
import os
import subprocess
import sys

import pytest

import tests.test_oracle as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_DIR = os.path.join(ROOT, "oracle")

MUTANTS = {
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k + 1 < K; ++k)"),
    "transposed_b_index": ("return load_in(B, fmt, trans ? j * ldb + k : k * ldb + j);",
                           "return load_in(B, fmt, trans ? k * ldb + j : j * ldb + k);"),
    "transA_ignored": ("return load_in(A, fmt, trans ? k * lda + i : i * lda + k);",
                       "return load_in(A, fmt, i * lda + k);"),
    "beta_sign": ("if (beta != 0.0) d += beta *", "if (beta != 0.0) d -= beta *"),
    "c_read_when_beta_zero": ("if (beta != 0.0) d += beta *", "d += beta *"),
    "alpha_dropped": ("double d = alpha * s;", "double d = s;"),
    "act_before_alpha": ("double d = alpha * s;",
                         "if (act == 1 && s < 0.0) s = slope * s;\n  double d = alpha * s;"),
    "truncating_round": ("return nearbyint(x / q) * q;", "return trunc(x / q) * q;"),
    "f16_subnormal_scale": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    "bf16_wrong_precision": ("double r = round_to_precision(x, 8, -126);",
                             "double r = round_to_precision(x, 9, -126);"),
    "gelu_wrong_sign": ("return 0.5 * d * erfc(-d / sqrt(2.0));", "return 0.5 * d * erfc(d / sqrt(2.0));"),
    "gelu_half_dropped": ("return 0.5 * d * erfc(-d / sqrt(2.0));", "return d * erfc(-d / sqrt(2.0));"),
    "silu_wrong_sign": ("return d / (1.0 + exp(-d));", "return d / (1.0 + exp(d));"),
    "relu_as_identity": ("case 2: return d < 0.0 ? 0.0 : d;", "case 2: return d;"),
    "tf32_rounds_instead": ("w &= 0xFFFFE000u;", "w = (w + 0x1000u) & 0xFFFFE000u;"),
    "tf32_keeps_11_bits": ("w &= 0xFFFFE000u;", "w &= 0xFFFFF000u;"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(os.path.join(ORACLE_DIR, "oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    d = tmp_path / name
    d.mkdir()
    csrc = d / "oracle.c"
    csrc.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{name}",
                                                  os.path.join(ORACLE_DIR, "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(csrc)
    mod._LIB = str(d / "liboracle.so")
    mod._lib = None
    mod.build(force=True)
    return mod


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if name.startswith("test_") and "oracle_lib" in inspect.signature(fn).parameters:
            out.append(fn)
    return out


def _run_pin(fn, lib):
    params = inspect.signature(fn).parameters
    marks = getattr(fn, "pytestmark", [])
    variants = [{}]
    for m in marks:
        if m.name == "parametrize":
            argnames = [a.strip() for a in m.args[0].split(",")]
            variants = [dict(zip(argnames, v if isinstance(v, tuple) else (v,)))
                        for v in m.args[1]]
    for kw in variants:
        kw = {k: v for k, v in kw.items() if k in params}
        fn(oracle_lib=lib, **kw)


def _caught_in_child(tmp_path, name):
    """Run every pin against the mutant in a child process; return the pins
    that failed (a crash of the child counts as one failure)."""
    code = (
        "import json, pathlib, sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import tests.test_oracle_mutants as tm\n"
        f"old, new = tm.MUTANTS[{name!r}]\n"
        f"lib = tm._build_mutant(pathlib.Path({str(tmp_path)!r}), {name!r}, old, new)\n"
        "caught = []\n"
        "for fn in tm._pin_functions():\n"
        "    print('RUNNING', fn.__name__, flush=True)\n"
        "    try:\n"
        "        tm._run_pin(fn, lib)\n"
        "    except (AssertionError, ValueError, IndexError, OverflowError):\n"
        "        caught.append(fn.__name__)\n"
        "print('CAUGHT', json.dumps(caught), flush=True)\n"
    )
    r = subprocess.run([sys.executable, "-W", "ignore", "-c", code], capture_output=True,
                       text=True, timeout=600, cwd=ROOT)
    for line in r.stdout.splitlines():
        if line.startswith("CAUGHT "):
            return json.loads(line[len("CAUGHT "):])
    running = [ln.split()[1] for ln in r.stdout.splitlines() if ln.startswith("RUNNING ")]
    assert r.returncode != 0, r.stderr[-2000:]
    return [f"{running[-1] if running else '?'} (child exited {r.returncode})"]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    caught = _caught_in_child(tmp_path, name)
    assert caught, f"no pin caught the planted mistake {name}"


def test_unmodified_copy_passes_every_pin(tmp_path):
    lib = _build_mutant(tmp_path, "none", "#include <math.h>", "#include <math.h>")
    for fn in _pin_functions():
        _run_pin(fn, lib)
