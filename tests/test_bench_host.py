"""Host-side pieces of bench.py, on CPU: the reference (oracle) arm's JSON
line, the clock-record parser, and the max-over-ranks timing reduction with
two gloo ranks."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "TFLOP/s" and d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == bench.LONG  # the GPU arm's `value` workload


def test_reference_arm_non_zero_rank_does_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1"], capture_output=True, text=True, timeout=120, env=env,
                       cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_clock_summary_parses_nvidia_smi_records():
    s = bench.ClockSampler(0)
    s.lines = [
        "300, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "1500, 2070, 1300.5, 0x4, Not Active, Not Active, Not Active, Active",
        "1400, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "1450, 2070, 1380.0, 0x4, Not Active, Not Active, Not Active, Active",
    ]
    out = s.summary()
    assert out["sm_mhz"] == 1450.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 4


def _free_port():
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        return so.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    r, w, _ = bench.dist_init()
    # each replica times its own work; the slowest replica sets the time
    out = bench.max_over_ranks([1.0 + r, 10.0 - r], w)
    bench.barrier(w)
    q.put((r, out))
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 10.0]
