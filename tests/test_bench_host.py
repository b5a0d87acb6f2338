"""CPU tests of bench.py's host logic: the reference arm's JSON line and the
rank aggregation of replicas (world size 2 over gloo)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1",
                        "--ref-fraction", str(1 / 2048)], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"].startswith("skinny")


def test_job_throughput_formula():
    import bench
    # two replicas, 3 steps of 1 GB each, slowest replica 1.5 s -> 4 GB/s
    assert bench.job_throughput(2, 3, 1e9, 1500.0) == pytest.approx(4.0)
    assert bench.max_over_ranks(7.5, None, None) == 7.5


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [12.0, 20.0][rank]
    worst = bench.max_over_ranks(ms, dist, "cpu")
    q.put((rank, worst, bench.job_throughput(world, 10, 1e8, worst)))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_gloo():
    import multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, gbs in out:
        assert worst == 20.0                      # max over ranks
        assert gbs == pytest.approx(2 * 10 * 1e8 / 0.020 / 1e9)


def test_reference_tiling_matches_the_guides_tail_wave_example():
    """The guide's section 3.2 example: 2304 x 1536 x 4096 with 256 x 128 tiles
    fills 108 SMs exactly (108 tiles); N = 1544 needs 117 tiles, a second wave
    with 9 of 108 SMs busy (8.33%)."""
    import bench
    import __graft_entry__
    __graft_entry__.build_library()
    full = bench.ref_tiling(bench.Call("x", 2304, 1536, 4096), 108)
    assert full == {"tiles": 108, "waves": 1.0, "tail_fraction": 0.0}
    tail = bench.ref_tiling(bench.Call("x", 2304, 1544, 4096), 108)
    assert tail["tiles"] == 117 and tail["tail_fraction"] == round(9 / 108, 4)
    assert bench.ref_tiling(bench.Call("gemv", 1, 8192, 8192), 152) is None


def test_sweep_samples_on_the_default_line():
    """The default bench line carries samples of both quantization sweeps:
    every 32nd N of 2304 x N x 4096 fp16 (169 shapes, all inside the shared
    6400-column B and C) and all 17 N of 27648 x N x 4096 bf16."""
    import bench
    sw = bench.sweep_calls()
    wave, tile = sw["wave_2304xNx4096_f16"], sw["tile_27648xNx4096_bf16"]
    assert [c.N for c in wave] == list(range(1024, 6401, 32)) and len(wave) == 169
    assert [c.N for c in tile] == list(range(128, 257, 8)) and len(tile) == 17
    for calls, ld in ((wave, 6400), (tile, 256)):
        for c in calls:
            assert c.ldb_override == ld and c.ldc_override == ld and c.N <= ld and not c.tb
    assert {c.in_fmt for c in wave} == {"f16"} and {c.in_fmt for c in tile} == {"bf16"}


def test_clock_summary_reads_memory_clock_and_temperature():
    """The clock record: SM clock median, memory clock median and the hottest
    GPU temperature of the samples inside the timed region; a field the
    driver reports as N/A is left out, not an error."""
    import time
    import bench
    c = bench.ClockSampler(0)
    t = time.time()
    na = "Not Active"
    c.samples = [(t, f"0, 2070, 2070, 170.5, 0x0, {na}, {na}, {na}, {na}, 3996, 45"),
                 (t + 0.01, f"0, 2060, 2070, 171.0, 0x0, {na}, {na}, {na}, Active, N/A, 46"),
                 (t + 5.0, f"0, 1000, 2070, 900.0, 0x0, Active, {na}, {na}, {na}, 3996, 90")]
    s = c.summary(t - 1, t + 1)
    assert s["sm_mhz"] == 2065.0 and s["sm_max_mhz"] == 2070.0 and s["mem_mhz"] == 3996.0
    assert s["gpu_temp_c_max"] == 46.0 and s["power_w_max"] == 171.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 2
