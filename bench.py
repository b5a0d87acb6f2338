"""Benchmark of the dense GEMM / GEMV path on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload skinny|square|small|tile|wave]

Default workload ("skinny", the configuration the headline metric is quoted
on): one step is four calls of the C ABI, all memory-bound on GB300 --
  skinny GEMM 8192 x 128 x 8192, bf16 -> fp32, B row-major
  skinny GEMM 8192 x 128 x 8192, bf16 -> fp32, B given transposed-contiguous
  GEMV 1 x 8192 x 8192, bf16 -> fp32, B row-major (column-stream kernel)
  GEMV 1 x 8192 x 8192, bf16 -> fp32, B transposed (row-dot kernel)
`value` is the step's algorithmic bytes (A, B read once, C written once)
over its device time, in GB/s; per-call TFLOP/s and GB/s are in `parts`.

Timing: inputs are resident in HBM; each call streams more than the 129 MB L2
from buffers no other call of the step touches, and a 512 MiB read flushes
L2 between steps (outside the timed events) without leaving dirty lines.  Every call is bracketed by
CUDA events on the stream it is launched on; the step time is the sum.
`e2e` repeats the step through the same C ABI with the inputs copied from
pinned host memory and the outputs copied back inside the timed region.
`cpu_baseline` times the CPU oracle (single thread) on a bounded sample of
the same step's outputs.  `other_configs` (default workload only) adds, outside
the step, each call of the other configurations -- 8192^3 bf16 -> bf16, 8192^3
with beta = 0.5 and LeakyReLU, 6912 x 2048 x 4096 and split-K 256 x 256 x 65536
-- timed alone between its own events with L2 flushed, in TFLOP/s and as a
fraction of the roofline.  `--impl reference` times that oracle as the
reference arm.  Under torchrun (N > 1) every rank runs the same workload on
its own GPU (replicas: the path needs no exchange between GPUs).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dense_gemm_mma_gb300 import inputs, roofline as rl  # noqa: E402

METRIC = "GEMM TFLOP/s & % of GB300 dense BF16 roofline; GEMV GB/s vs HBM peak"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ workloads

class Call:
    """One gemm_run of a workload: shape, types, flags and epilogue."""

    def __init__(self, name, M, N, K, in_fmt="bf16", out_fmt="f32", ta=False, tb=False,
                 alpha=1.0, beta=0.0, act=0, slope=0.0, seed=0, ldb=None, ldc=None, group=None):
        self.name, self.M, self.N, self.K = name, M, N, K
        self.in_fmt, self.out_fmt, self.ta, self.tb = in_fmt, out_fmt, ta, tb
        self.alpha, self.beta, self.act, self.slope, self.seed = alpha, beta, act, slope, seed
        self.ldb_override, self.ldc_override, self.group = ldb, ldc, group

    @property
    def flops(self):
        return rl.gemm_flops(self.M, self.N, self.K)

    @property
    def bytes(self):
        return rl.gemm_bytes(self.M, self.N, self.K, self.in_fmt, self.out_fmt, self.beta != 0.0)

    def desc(self):
        return {"name": self.name, "M": self.M, "N": self.N, "K": self.K, "in": self.in_fmt,
                "out": self.out_fmt, "transA": self.ta, "transB": self.tb, "alpha": self.alpha,
                "beta": self.beta, "act": "leaky_relu" if self.act else "none", "slope": self.slope}


def workload(name: str):
    if name == "skinny":
        s = inputs.config_seed(1)
        return ("skinny_gemm_8192x128x8192_and_gemv_1x8192x8192_bf16", [
            Call("skinny_NN", 8192, 128, 8192, seed=s),
            Call("skinny_NT", 8192, 128, 8192, tb=True, seed=s),
            Call("gemv_N", 1, 8192, 8192, seed=s),
            Call("gemv_T", 1, 8192, 8192, tb=True, seed=s)])
    if name == "square":
        s = inputs.config_seed(2)
        return ("square_gemm_8192_cubed_bf16", [
            Call("square_bf16_out", 8192, 8192, 8192, out_fmt="bf16", seed=s),
            Call("square_beta_leaky", 8192, 8192, 8192, out_fmt="f32", beta=0.5, act=1, slope=0.01,
                 seed=s)])
    if name == "tf32":
        s = inputs.config_seed(2)
        return ("square_gemm_8192_cubed_tf32", [
            Call("square_tf32_NT", 8192, 8192, 8192, in_fmt="tf32", tb=True, seed=s),
            Call("square_tf32_NN", 8192, 8192, 8192, in_fmt="tf32", seed=s)])
    if name == "small":
        return ("gemm_512_cubed_bf16", [Call("gemm_512", 512, 512, 512, seed=inputs.config_seed(0))])
    if name == "tile":
        s = inputs.config_seed(3)
        calls = [Call("tile_6912x2048x4096", 6912, 2048, 4096, seed=s)]
        calls += [Call(f"tile_27648xN{n}x4096", 27648, n, 4096, seed=s, ldb=256, ldc=256, group="m27648")
                  for n in range(128, 257, 8)]
        return ("tile_quantization_sweep_bf16", calls)
    if name == "wave":
        s = inputs.config_seed(4)
        calls = [Call(f"wave_2304xN{n}x4096", 2304, n, 4096, in_fmt="f16", seed=s, ldb=6400,
                      ldc=6400, group="m2304") for n in range(1024, 6401, 8)]
        calls.append(Call("splitk_256x256x65536", 256, 256, 65536, in_fmt="f16", seed=s))
        return ("wave_quantization_sweep_f16_and_splitk", calls)
    raise SystemExit(f"unknown workload {name}")


# --------------------------------------------------------------------- helpers

def stored_shapes(c: Call):
    a = (c.K, c.M) if c.ta else (c.M, c.K)
    b = (c.N, c.K) if c.tb else (c.K, c.N)
    return a, b


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 20 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "clocks.mem,temperature.gpu")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        def parse(s):
            p = [x.strip() for x in s.split(",")]
            try:
                r = {"sm": float(p[1]), "max": float(p[2]), "power": float(p[3]),
                     "hw_slowdown": p[5], "hw_thermal": p[6], "sw_thermal": p[7], "sw_power": p[8]}
            except (ValueError, IndexError):
                return None
            for key, i in (("mem", 9), ("temp", 10)):  # (absent or "N/A" on some drivers)
                try:
                    r[key] = float(p[i])
                except (ValueError, IndexError):
                    r[key] = None
            return r
        rows = [(t, parse(s)) for t, s in self.samples]
        rows = [(t, r) for t, r in rows if r is not None]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        inside = [r for t, r in rows if t0 <= t <= t1]
        note = "samples inside the timed region"
        if not inside:  # timed region shorter than the sampling period: nearest samples
            inside = [min(rows, key=lambda tr: min(abs(tr[0] - t0), abs(tr[0] - t1)))[1]]
            note = "timed region shorter than the 20 ms sampling period; nearest sample"
        reasons = set()
        for r in inside:
            for key, name in (("hw_slowdown", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        mem = [r["mem"] for r in inside if r["mem"] is not None]
        temp = [r["temp"] for r in inside if r["temp"] is not None]
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["max"] for r in inside),
                "mem_mhz": statistics.median(mem) if mem else None,
                "gpu_temp_c_max": max(temp) if temp else None,
                "power_w_max": max(r["power"] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside), "note": note}


def ref_tiling(c, sms: int):
    """Tile and wave quantization of the call under a fixed 256 x 128 tiling, one
    tile per SM ("Matrix Multiplication Background User's Guide", section 3.2,
    quotes its tail-wave example for 256 x 128 tiles on 108 SMs), for comparison
    with the tiling the planner chose.  None for GEMV shapes."""
    from dense_gemm_mma_gb300 import gemm
    if c.M < 2 or c.N < 2 or sms <= 0:
        return None
    q = gemm.gemm_quantization(c.M, c.N, 256, 128, 1, sms, 1)
    return {"tiles": q.tiles, "waves": round(q.waves, 3), "tail_fraction": round(q.tail_fraction, 4)}


# Dense tensor-core peak of a call's operand type in TFLOP/s: the measured bf16
# figure, times the nominal TF32 / bf16 ratio (1.1 / 2.25 PFLOP/s) for TF32.
def tensor_peak(c, peaks) -> float:
    return peaks["bf16_tflops"] * (1.1 / 2.25 if c.in_fmt == "tf32" else 1.0)


def max_over_ranks(value: float, dist, device) -> float:
    """Largest `value` over all ranks (the slowest replica sets the job time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, steps: int, step_bytes: float, max_ms: float) -> float:
    """Whole-job GB/s: the bytes every replica processed over the slowest replica's time."""
    return world * steps * step_bytes / (max_ms / 1e3) / 1e9


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------ CPU oracle leg

def oracle_sample(calls, host, fraction: float):
    """Time the CPU oracle on `fraction` of every call's output rows (for
    GEMV: of its outputs).  Returns (seconds, bytes-equivalent, description)."""
    import oracle
    oracle.build()
    total_s = 0.0
    total_bytes = 0.0
    parts = []
    for c in calls:
        A, B = host[c.name]["A"], host[c.name]["B"]
        if c.M == 1:
            n = max(1, int(round(c.N * fraction)))
            rows = np.zeros(n, dtype=np.int64)
            cols = np.linspace(0, c.N - 1, n).astype(np.int64)
        else:
            n_rows = max(1, int(round(c.M * fraction)))
            r = np.linspace(0, c.M - 1, n_rows).astype(np.int64)
            rows = np.repeat(r, c.N)
            cols = np.tile(np.arange(c.N, dtype=np.int64), n_rows)
        t = time.perf_counter()
        oracle.sample(rows, cols, c.K, A, B, lda=A.shape[1], ldb=B.shape[1], alpha=c.alpha,
                      beta=0.0, in_fmt=c.in_fmt, out_fmt=c.out_fmt, transA=c.ta, transB=c.tb,
                      act=c.act, slope=c.slope)
        dt = time.perf_counter() - t
        frac = len(rows) / float(c.M * c.N)
        total_s += dt
        total_bytes += c.bytes * frac
        parts.append(f"{c.name}: {len(rows)} outputs")
    return total_s, total_bytes, "; ".join(parts)


# --------------------------------------------------------------------- main

def run_reference(args, wl_name, calls, rank):
    if rank != 0:
        return 0
    t_gen = time.time()
    host = {}
    for c in calls:
        (ar, ac), (br, bc) = stored_shapes(c)
        host[c.name] = {"A": inputs.matrix(ar, ac, c.seed, inputs.TENSOR_A, c.in_fmt),
                        "B": inputs.matrix(br, bc, c.seed, inputs.TENSOR_B, c.in_fmt)}
    frac = args.ref_fraction
    for _ in range(args.warmup if args.warmup < 2 else 1):
        oracle_sample(calls[:1], host, frac / 8)
    secs, byts = 0.0, 0.0
    desc = ""
    for _ in range(args.steps):
        s, b, desc = oracle_sample(calls, host, frac)
        secs += s
        byts += b
    value = byts / secs / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": calls[0].in_fmt,
            "data": "synthetic", "config": {"workload": wl_name, "calls": [c.desc() for c in calls],
                                            "parallelism": "none"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: {desc} (fraction {frac} of every call's outputs)"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0,
            "note": f"CPU fp64 oracle, single thread; input generation {time.time() - t_gen:.1f} s untimed"}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="skinny", choices=["skinny", "square", "small", "tile", "wave", "tf32"])
    ap.add_argument("--cpu-fraction", type=float, default=None,
                    help="fraction of each call's outputs the cpu_baseline oracle computes")
    ap.add_argument("--ref-fraction", type=float, default=1.0 / 512)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the per-call timing of the compute-bound and split-K configurations "
                         "that the default run adds under `other_configs`")
    ap.add_argument("--other-reps", type=int, default=20)
    ap.add_argument("--only", default=None,
                    help="comma-separated call names: run only these calls of the workload "
                         "(e.g. one call for a profiler capture)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--autotune", action="store_true",
                    help="benchmark mode: time the planner's leading candidates once per shape "
                         "(during warm-up) and keep the fastest")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3  # at least three warm-up steps
    ws, rank, local = dist_env()
    wl_name, calls = workload(args.workload)
    if args.only:
        keep = set(args.only.split(","))
        calls = [c for c in calls if c.name in keep]
        if not calls:
            raise SystemExit(f"--only matches no call of workload {args.workload}")
        wl_name += "_only_" + "_".join(c.name for c in calls)
    if args.impl == "reference":
        return run_reference(args, wl_name, calls, rank)

    import torch
    from dense_gemm_mma_gb300 import gemm

    import __graft_entry__
    __graft_entry__.build_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    plan = gemm.Plan(local)
    if args.autotune:
        gemm.gemm_plan_set_autotune(plan.handle, True)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    # ---- inputs: generated once on the host, copied to distinct device buffers
    t_gen = time.time()
    host, devbuf = {}, {}
    shared = {}
    for c in calls:
        (ar, ac), (br, bc) = stored_shapes(c)
        key_a = (ar, ac, c.seed, c.in_fmt)
        if key_a not in shared:
            shared[key_a] = inputs.matrix(ar, ac, c.seed, inputs.TENSOR_A, c.in_fmt)
        A = shared[key_a]
        if c.ldb_override and not c.tb:
            bc_full = c.ldb_override
            key_b = (br, bc_full, c.seed, c.in_fmt, "grp")
            if key_b not in shared:
                shared[key_b] = inputs.matrix(br, bc_full, c.seed, inputs.TENSOR_B, c.in_fmt)
            B = shared[key_b]
        else:
            B = inputs.matrix(br, bc, c.seed, inputs.TENSOR_B, c.in_fmt)
        host[c.name] = {"A": A, "B": B}
    torch_dt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}

    def to_dev(arr, fmt):
        t = torch.from_numpy(arr.view(np.int16) if arr.dtype == np.uint16 else arr)
        return t.view(torch_dt[fmt]).to(dev) if arr.dtype == np.uint16 else t.to(dev)

    # Every call gets its own device copies (calls of a sweep group share theirs).
    group_buf = {}
    for c in calls:
        h = host[c.name]
        if c.group and c.group in group_buf:
            devbuf[c.name] = group_buf[c.group]
            continue
        Ad = to_dev(h["A"], c.in_fmt)
        Bd = to_dev(h["B"], c.in_fmt)
        ldc = c.ldc_override or c.N
        if c.beta != 0.0:
            Cin = inputs.matrix(c.M, ldc, c.seed, inputs.TENSOR_C, c.out_fmt)
            Cd = to_dev(Cin, c.out_fmt)
            C0 = Cd.clone()
        else:
            Cd = torch.empty((c.M, ldc), dtype=torch_dt[c.out_fmt], device=dev)
            C0 = None
        devbuf[c.name] = {"A": Ad, "B": Bd, "C": Cd, "C0": C0}
        if c.group:
            group_buf[c.group] = devbuf[c.name]
    gen_s = time.time() - t_gen
    # L2 flush: reading 512 MiB leaves L2 full of clean lines of this buffer,
    # so no dirty data is written back inside a timed call.
    flush = torch.zeros(512 * 2 ** 20 // 4, dtype=torch.float32, device=dev)
    flush_out = torch.zeros((), dtype=torch.float32, device=dev)

    def flush_l2():
        torch.sum(flush, dim=0, out=flush_out)

    def launch(c, bufs, a_ptr=None, b_ptr=None, c_ptr=None):
        (ar, ac), (br, bc) = stored_shapes(c)
        lda = ac
        ldb = c.ldb_override if (c.ldb_override and not c.tb) else bc
        ldc = c.ldc_override or c.N
        st = gemm.gemm_run(plan.handle, c.M, c.N, c.K,
                           a_ptr or bufs["A"].data_ptr(), lda, b_ptr or bufs["B"].data_ptr(), ldb,
                           c_ptr or bufs["C"].data_ptr(), ldc, c.alpha, c.beta,
                           gemm.DTYPES[(c.in_fmt, c.out_fmt)], int(c.ta), int(c.tb), c.act, c.slope,
                           sptr)
        if st != gemm.GEMM_OK:
            raise RuntimeError(f"{c.name}: {gemm.gemm_status_string(st)}")
        return gemm.gemm_plan_last_config(plan.handle)

    n = len(calls)
    infos = [None] * n

    def one_step(events=None, flush_each=False):
        launches = 0
        for i, c in enumerate(calls):
            if flush_each:
                flush_l2()
            if events is not None:
                events[i][0].record(stream)
            info = launch(c, devbuf[c.name])
            if events is not None:
                events[i][1].record(stream)
            infos[i] = info
            launches += info.launches
        return launches

    # warm-up
    for _ in range(args.warmup):
        flush_l2()
        one_step()
    torch.cuda.synchronize(dev)
    if plan.poll_error() != gemm.GEMM_OK:
        raise RuntimeError("watchdog fired during warm-up")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    # A workload whose calls read buffers no other call touches is timed a step
    # at a time (one event pair around its calls, which run back to back as a
    # user's would); the calls of a sweep share A and B, so each is timed on
    # its own with L2 flushed before it.
    sweep = any(c.group for c in calls)
    new_ev = lambda: torch.cuda.Event(enable_timing=True)
    ev = [[[new_ev(), new_ev()] for _ in range(n)] for _ in range(args.steps)]
    step_ev = [[new_ev(), new_ev()] for _ in range(args.steps)]

    def restore_c():
        # beta != 0 calls update C in place: restore it outside the timed events
        for c in calls:
            if devbuf[c.name]["C0"] is not None:
                devbuf[c.name]["C"].copy_(devbuf[c.name]["C0"])

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_begin = time.time()
    gpu_launches = 0
    for s in range(args.steps):
        flush_l2()
        restore_c()
        if sweep:
            gpu_launches += one_step(ev[s], flush_each=True)
        else:
            step_ev[s][0].record(stream)
            gpu_launches += one_step()
            step_ev[s][1].record(stream)
            # the per-call breakdown (parts, roofline): the same step again,
            # each call between its own events, right after the timed step so
            # that both see the same clocks and power state
            flush_l2()
            restore_c()
            gpu_launches += one_step(ev[s])
    torch.cuda.synchronize(dev)
    t_end = time.time()
    if dist is not None:
        dist.barrier()
    call_ms = np.array([[ev[s][i][0].elapsed_time(ev[s][i][1]) for i in range(n)]
                        for s in range(args.steps)])
    step_ms = call_ms.sum(axis=1) if sweep else \
        np.array([step_ev[s][0].elapsed_time(step_ev[s][1]) for s in range(args.steps)])
    time.sleep(0.3)
    sampler.stop()
    if plan.poll_error() != gemm.GEMM_OK:
        raise RuntimeError("watchdog fired during the timed region")
    total_ms = max_over_ranks(float(step_ms.sum()), dist, dev)
    step_bytes = sum(c.bytes for c in calls)
    step_flops = sum(c.flops for c in calls)
    value = job_throughput(ws, args.steps, step_bytes, total_ms)

    peaks, peak_src = load_peaks()
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mean_call = call_ms.mean(axis=0)
    parts = []
    for i, c in enumerate(calls):
        sec = mean_call[i] / 1e3
        info = infos[i].as_dict()
        ai = c.flops / c.bytes
        att = rl.attainable(ai, tensor_peak(c, peaks) * 1e12, peaks["hbm_gbs"] * 1e9)
        parts.append({
            "name": c.name, "us": round(mean_call[i] * 1e3, 2),
            "us_median": round(float(np.median(call_ms[:, i])) * 1e3, 2),
            "us_iqr": round(float(np.subtract(*np.percentile(call_ms[:, i], [75, 25]))) * 1e3, 2),
            "tflops": round(c.flops / sec / 1e12, 2), "gbs": round(c.bytes / sec / 1e9, 1),
            "intensity": round(ai, 1), "bound": rl.bound(ai, tensor_peak(c, peaks) * 1e12, peaks["hbm_gbs"] * 1e9),
            "frac_of_roofline": round(c.flops / sec / att, 3),
            "frac_of_nominal_roofline": round(c.flops / sec / rl.attainable(
                ai, (1.1e15 if c.in_fmt == "tf32" else 2.25e15), 8e12), 3),
            "path": info["path"], "tile": f"{info['tile_m']}x{info['tile_n']}", "splitk": info["splitk"],
            "grid": info["grid"], "units": info["units"], "waves": round(info["waves"], 3),
            "tail_fraction": round(info["tail_fraction"], 4), "launches": info["launches"],
            "ref_256x128": ref_tiling(c, n_sms)})
    dom = int(np.argmax(mean_call))
    dc = calls[dom]
    dom_sec = mean_call[dom] / 1e3
    dom_ai = dc.flops / dc.bytes
    dom_bound = rl.bound(dom_ai, tensor_peak(dc, peaks) * 1e12, peaks["hbm_gbs"] * 1e9)
    if dom_bound == "hbm":
        achieved, peak, unit = dc.bytes / dom_sec / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = dc.flops / dom_sec / 1e12, round(tensor_peak(dc, peaks), 1), "TFLOP/s"
    roof = {"bound": dom_bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic_for(dc.name),
            "kernel": dc.name, "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
            "algorithmic_bytes_per_launch": dc.bytes, "algorithmic_flops_per_launch": dc.flops}

    # ---- end to end: host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, calls, host, devbuf, launch, stream, dev, torch, step_bytes, ws, dist)

    # ---- CPU oracle baseline (rank 0, N == 1 only)
    cpu = None
    if not args.no_cpu and rank == 0 and ws == 1:
        frac = args.cpu_fraction or {"skinny": 1 / 4, "square": 1 / 8192, "tf32": 1 / 8192, "small": 1 / 8,
                                     "tile": 1 / 4096, "wave": 1 / 2048}[args.workload]
        secs, byts, desc = oracle_sample(calls, host, frac)
        cpu = {"value": round(byts / secs / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{desc} (fraction {frac:g} of each call's outputs; {secs:.1f} s)",
               "tflops": round(sum(c.flops for c in calls) * (byts / step_bytes) / secs / 1e12, 9)}

    # ---- the other configurations, each call timed alone (outside the step)
    others = None
    if args.workload == "skinny" and not args.no_others:
        others = measure_others(args, plan, launch, flush_l2, stream, dev, torch, peaks, n_sms, local)

    clocks = sampler.summary(t_begin, t_end)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": calls[0].in_fmt, "data": "synthetic",
            "config": {"workload": wl_name, "calls": [c.desc() for c in calls],
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                       "l2": ("flushed before every call (512 MiB read, untimed); the calls of a sweep "
                              "share A and B" if sweep else
                              "flushed between steps (512 MiB read, untimed); each call reads "
                              "device buffers no other call of the step touches"),
                       "timing": ("each call between its own CUDA events; ms_per_step is their sum" if sweep
                                  else "one CUDA event pair around each step's calls, which run back "
                                       "to back; every timed step is followed by the same step with "
                                       "events around each call, for parts and roofline"),
                       "planner": "benchmark mode (timed once per shape in warm-up)" if args.autotune
                                  else "cost model",
                       "step_bytes": step_bytes, "step_flops": step_flops,
                       "step_tflops": round(ws * args.steps * step_flops / (total_ms / 1e3) / 1e12, 2),
                       "input_generation_s": round(gen_s, 1)},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": gpu_launches,
            "clocks": clocks, "parts": parts, "other_configs": others,
        }
        print(json.dumps(line), flush=True)
    plan.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def other_calls():
    """The compute-bound square GEMM (both runs), the 6912 x 2048 x 4096 tile case and
    the 256 x 256 x 65536 split-K case, on their own configurations' seeds."""
    s2, s3, s4 = inputs.config_seed(2), inputs.config_seed(3), inputs.config_seed(4)
    return [
        Call("square_bf16_out", 8192, 8192, 8192, out_fmt="bf16", seed=s2),
        Call("square_beta_leaky", 8192, 8192, 8192, out_fmt="f32", beta=0.5, act=1, slope=0.01, seed=s2),
        Call("tile_6912x2048x4096", 6912, 2048, 4096, seed=s3),
        Call("splitk_256x256x65536", 256, 256, 65536, in_fmt="f16", seed=s4),
    ]


def measure_others(args, plan, launch, flush_l2, stream, dev, torch, peaks, n_sms, gpu_index):
    """Each call of other_calls() between its own CUDA events on the launching
    stream, L2 flushed before every call (untimed), C restored before a beta call
    (untimed), after three untimed warm-up calls; reports the median, TFLOP/s and
    the fraction of the roofline against the measured peaks, with the clocks
    sampled while these calls ran."""
    from dense_gemm_mma_gb300 import gemm
    torch_dt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}

    def to_dev(arr, fmt):
        if arr.dtype == np.uint16:
            return torch.from_numpy(arr.view(np.int16)).view(torch_dt[fmt]).to(dev)
        return torch.from_numpy(arr).to(dev)

    t_gen = time.time()
    calls = other_calls()
    host_cache, bufs = {}, {}
    for c in calls:
        (ar, ac), (br, bc) = stored_shapes(c)
        key = (c.M, c.N, c.K, c.in_fmt, c.seed)
        if key not in host_cache:
            host_cache[key] = (to_dev(inputs.matrix(ar, ac, c.seed, inputs.TENSOR_A, c.in_fmt), c.in_fmt),
                               to_dev(inputs.matrix(br, bc, c.seed, inputs.TENSOR_B, c.in_fmt), c.in_fmt))
        Ad, Bd = host_cache[key]
        if c.beta != 0.0:
            Cd = to_dev(inputs.matrix(c.M, c.N, c.seed, inputs.TENSOR_C, c.out_fmt), c.out_fmt)
            C0 = Cd.clone()
        else:
            Cd, C0 = torch.empty((c.M, c.N), dtype=torch_dt[c.out_fmt], device=dev), None
        bufs[c.name] = {"A": Ad, "B": Bd, "C": Cd, "C0": C0}
    gen_s = time.time() - t_gen
    reps = max(3, args.other_reps)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)] for _ in calls]
    infos = []
    sampler = ClockSampler(gpu_index)
    sampler.start()
    time.sleep(0.3)
    t0 = time.time()
    for i, c in enumerate(calls):
        b = bufs[c.name]
        for _ in range(3):  # warm-up
            flush_l2()
            launch(c, b)
        for r in range(reps):
            flush_l2()
            if b["C0"] is not None:
                b["C"].copy_(b["C0"])
            ev[i][r][0].record(stream)
            info = launch(c, b)
            ev[i][r][1].record(stream)
        infos.append(info)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    time.sleep(0.3)
    sampler.stop()
    if plan.poll_error() != gemm.GEMM_OK:
        raise RuntimeError("watchdog fired while timing the other configurations")
    out = []
    for i, c in enumerate(calls):
        ms = np.array([a.elapsed_time(z) for a, z in ev[i]])
        med = float(np.median(ms)) / 1e3
        ai = c.flops / c.bytes
        tpk = tensor_peak(c, peaks) * 1e12
        att = rl.attainable(ai, tpk, peaks["hbm_gbs"] * 1e9)
        info = infos[i].as_dict()
        out.append({
            **c.desc(), "us_median": round(med * 1e6, 2), "us_min": round(float(ms.min()) * 1e3, 2),
            "us_iqr": round(float(np.subtract(*np.percentile(ms, [75, 25]))) * 1e3, 2),
            "tflops": round(c.flops / med / 1e12, 2), "gbs": round(c.bytes / med / 1e9, 1),
            "intensity": round(ai, 1), "bound": rl.bound(ai, tpk, peaks["hbm_gbs"] * 1e9),
            "frac_of_roofline": round(c.flops / med / att, 3),
            "frac_of_nominal_roofline": round(c.flops / med / rl.attainable(ai, 2.25e15, 8e12), 3),
            "path": info["path"], "tile": f"{info['tile_m']}x{info['tile_n']}", "splitk": info["splitk"],
            "grid": info["grid"], "waves": round(info["waves"], 3), "launches": info["launches"]})
    del bufs, host_cache
    torch.cuda.empty_cache()
    sweeps = measure_sweeps(args, plan, launch, flush_l2, stream, dev, torch, peaks, to_dev)
    return {"timing": (f"each call alone between its own CUDA events, L2 flushed before every call, "
                       f"3 warm-up + {reps} timed calls each; median; roofline = min(measured bf16 "
                       f"burst peak, intensity x measured copy bandwidth)"),
            "input_generation_s": round(gen_s, 1), "calls": out, "clocks": sampler.summary(t0, t1),
            "sweeps": sweeps}


def sweep_calls():
    """Samples of the two quantization sweeps: 2304 x N x 4096 fp16 for every
    32nd N from 1024 to 6400 (169 of the 673 shapes; the tile count per wave
    goes through every residue), and 27648 x N x 4096 bf16 for N = 128 ... 256
    in steps of 8 (all 17)."""
    s3, s4 = inputs.config_seed(3), inputs.config_seed(4)
    wave = [Call(f"wave_2304xN{n}x4096", 2304, n, 4096, in_fmt="f16", seed=s4, ldb=6400, ldc=6400)
            for n in range(1024, 6401, 32)]
    tile = [Call(f"tile_27648xN{n}x4096", 27648, n, 4096, seed=s3, ldb=256, ldc=256)
            for n in range(128, 257, 8)]
    return {"wave_2304xNx4096_f16": wave, "tile_27648xNx4096_bf16": tile}


def measure_sweeps(args, plan, launch, flush_l2, stream, dev, torch, peaks, to_dev):
    """Each call of each sweep sample alone between its own CUDA events, L2
    flushed before every call, one warm-up and 5 timed calls (median); the
    calls of a sweep share A, B (the widest N) and C.  Reported per sweep:
    the median, the range and the fraction of the roofline, and every call's
    time."""
    from dense_gemm_mma_gb300 import gemm
    out = {}
    for name, calls in sweep_calls().items():
        c0 = calls[0]
        n_max = max(c.N for c in calls)
        A = to_dev(inputs.matrix(c0.M, c0.K, c0.seed, inputs.TENSOR_A, c0.in_fmt), c0.in_fmt)
        B = to_dev(inputs.matrix(c0.K, n_max, c0.seed, inputs.TENSOR_B, c0.in_fmt), c0.in_fmt)
        C = torch.empty((c0.M, n_max), dtype=torch.float32, device=dev)
        b = {"A": A, "B": B, "C": C, "C0": None}
        reps = 5
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)] for _ in calls]
        infos = []
        for i, c in enumerate(calls):
            flush_l2()
            launch(c, b)
            for r in range(reps):
                flush_l2()
                ev[i][r][0].record(stream)
                info = launch(c, b)
                ev[i][r][1].record(stream)
            infos.append(info.as_dict())
        torch.cuda.synchronize(dev)
        if plan.poll_error() != gemm.GEMM_OK:
            raise RuntimeError(f"watchdog fired in sweep {name}")
        us = np.array([float(np.median([a.elapsed_time(z) for a, z in ev[i]])) * 1e3 for i in range(len(calls))])
        tfl = np.array([c.flops / (u * 1e-6) / 1e12 for c, u in zip(calls, us)])
        gbs = np.array([c.bytes / (u * 1e-6) / 1e9 for c, u in zip(calls, us)])
        frac = []
        for c, u in zip(calls, us):
            ai = c.flops / c.bytes
            att = rl.attainable(ai, tensor_peak(c, peaks) * 1e12, peaks["hbm_gbs"] * 1e9)
            frac.append(c.flops / (u * 1e-6) / att)
        frac = np.array(frac)
        bound = rl.bound(c0.flops / c0.bytes, tensor_peak(c0, peaks) * 1e12, peaks["hbm_gbs"] * 1e9)
        out[name] = {
            "shapes": len(calls), "bound": bound, "N": [c.N for c in calls], "us": [round(float(u), 2) for u in us],
            "tflops_median": round(float(np.median(tfl)), 1), "tflops_min": round(float(tfl.min()), 1),
            "tflops_max": round(float(tfl.max()), 1), "gbs_median": round(float(np.median(gbs)), 1),
            "gbs_min": round(float(gbs.min()), 1), "gbs_max": round(float(gbs.max()), 1),
            "frac_of_roofline_median": round(float(np.median(frac)), 3),
            "paths": {p: sum(1 for i in infos if i["path"] == p) for p in sorted({i["path"] for i in infos})}}
        del A, B, C, b
        torch.cuda.empty_cache()
    return out


def traffic_for(kernel_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel sources as they are now (else null)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = source_digest()
    for line in open(path):
        p = line.split()
        if len(p) >= 3 and p[0] == kernel_name and p[1] == want:
            return float(p[2])
    return None


def source_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_gemm_mma_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:12]


def measure_e2e(args, calls, host, devbuf, launch, stream, dev, torch, step_bytes, ws, dist):
    """Same step through the C ABI, with every input copied from pinned host
    memory and every output copied back inside the timed region (copies on a
    second stream, overlapping the previous calls' kernels)."""
    pinned_in, pinned_out = [], []
    h2d = d2h = 0
    seen = set()
    plan_items = []
    for c in calls:
        b = devbuf[c.name]
        items = []
        for key in ("A", "B"):
            t = b[key]
            if id(t) in seen:
                continue
            seen.add(id(t))
            p = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            p.copy_(t)
            items.append((p, t))
            h2d += t.numel() * t.element_size()
        if b["C0"] is not None:
            p = torch.empty(b["C0"].shape, dtype=b["C0"].dtype, pin_memory=True)
            p.copy_(b["C0"])
            items.append((p, b["C"]))
            h2d += b["C0"].numel() * b["C0"].element_size()
        out = torch.empty(b["C"].shape, dtype=b["C"].dtype, pin_memory=True)
        d2h += b["C"].numel() * b["C"].element_size()
        plan_items.append((c, b, items, out))
    steps = max(1, min(args.steps, 20))
    # Pipelined as a user would run it: inputs go up on a copy stream while
    # the previous calls compute; each call waits for its own inputs, and a
    # buffer is refilled only after the call that read it has finished.
    copy_stream = torch.cuda.Stream(device=dev)
    n = len(plan_items)
    ready = [torch.cuda.Event() for _ in range(n)]
    done = [torch.cuda.Event() for _ in range(n)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def run_step(first):
        for i, (c, b, items, out) in enumerate(plan_items):
            with torch.cuda.stream(copy_stream):
                if not first:
                    copy_stream.wait_event(done[i])
                for p, t in items:
                    t.copy_(p, non_blocking=True)
                ready[i].record(copy_stream)
            stream.wait_event(ready[i])
            launch(c, b)
            out.copy_(b["C"], non_blocking=True)
            done[i].record(stream)

    run_step(True)  # warm-up
    torch.cuda.synchronize(dev)
    e0.record(stream)
    copy_stream.wait_event(e0)
    for s in range(steps):
        run_step(s == 0)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(float(e0.elapsed_time(e1)), dist, dev)
    return {"value": round(job_throughput(ws, steps, step_bytes, ms), 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(ms / steps, 4)}


if __name__ == "__main__":
    sys.exit(main())
