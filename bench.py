#!/usr/bin/env python
"""Benchmark of the fused attention forward on GB300.

One step is one pass of the whole hot path over one batch of synthetic
input: the prefill kernel on the causal B=2, H=16, N=4096, d=128 workload,
the prefill kernel on the causal B=1, H=32, N=16384, d=128 long-sequence
workload (the largest single-GPU prefill workload of the study, whose
attention fwd TFLOP/s against the bf16 tensor peak is the line's `value`),
and the split-K decode (split kernel + combine kernel) on the
B=64, H=32, Nk=8192, d=128 decode workload (HBM GB/s).  L2 is flushed before
every step: a 256 MiB write, then a 256 MiB read of another buffer, so no dirty
line of the flush is left for the timed kernels to write back.  Each kernel is timed with CUDA events on the
stream it is launched on.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs N independent replicas (one per GPU, launched by torchrun): the
path has no exchange step.  ``--impl reference`` times the fp64 CPU oracle on
the host cores instead, on bounded samples of the same workload.
Prints one JSON line (rank 0).
"""
import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s & % of BF16 tensor peak; decode-shape HBM GB/s"
HEADLINE = "b2h16n4096d128_causal"
LONG = "b1h32n16384d128_causal"
DECODE = "decode_b64h32nk8192d128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
LAUNCH_COVER_CYCLES = 400_000  # ~0.2 ms device-side spin before each timed step
CPU_SAMPLE_SECONDS = 10.0
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gbattn", "reference"], default="gbattn")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (for quick runs)")
    ap.add_argument("--case", default=None,
                    help="run only this workload's kernel(s) (profiling runs); prints its time")
    ap.add_argument("--shape", default=None,
                    help="with --case custom: B,H,Nq,Nk,d,causal of a profiling workload")
    ap.add_argument("--mma-rates", action="store_true",
                    help="time the tensor-core issue forms (attn_bench_mma_rate) and print "
                         "one JSON line: single-CTA and CTA-pair products, lone and "
                         "converged issuer, with and without waits and softmax-like warps")
    ap.add_argument("--pass", dest="which",
                    choices=["fwd", "bwd", "fp8", "mx", "merge", "pair"], default="fwd",
                    help="with --case: time the forward (default), the backward call, the "
                         "forward on FP8 (E4M3) operands, (decode) MXFP8 keys and values, "
                         "attn_merge of 4 shard results of the workload's shape, or the "
                         "forward on CTA-pair products (attn_fwd_cta_pair)")
    a = ap.parse_args()
    a.warmup = max(3, a.warmup)
    a.steps = max(1, a.steps)
    return a


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def _sources_sha(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "attention_flashattention_fwd_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


PREFILL_SOURCES = ["prefill_sm103.cu", "sm103_ptx.cuh", "gbattn_internal.h"]
PAIR_SOURCES = ["prefill_pair_sm103.cu", "sm103_ptx.cuh", "gbattn_internal.h"]
DECODE_SOURCES = ["decode_sm103.cu", "sm103_ptx.cuh", "gbattn_internal.h"]
BACKWARD_SOURCES = ["backward_sm103.cu", "sm103_ptx.cuh", "gbattn_internal.h"]
FP8_PEAK_RATIO = 2.0  # nominal dense fp8 : bf16 tensor rate (4.5 : 2.25 PFLOP/s)
# ex2.approx.f32 per clock per SM on GB300 (measured: 4 cycles per warp instruction
# per SM sub-partition); the SFU roofline of the softmax's exponentials
SFU_EX2_PER_CLK_SM = 32.0


def visible_pairs(w):
    """(query, key) pairs a prefill workload scores: one exponential each."""
    if not w.causal:
        return w.B * w.H * w.Nq * w.Nk
    off = w.Nk - w.Nq  # query i sees keys j <= i + off
    return w.B * w.H * (w.Nq * (off + 1) + w.Nq * (w.Nq - 1) // 2)
MERGE_PARTS = 4  # key shards merged by attn_merge in the context-parallel measurement
MERGE_SOURCES = ["merge_sm103.cu", "sm103_ptx.cuh", "gbattn_internal.h"]
# FLOPs of the backward: five products of the forward's size (S and dP
# recomputed, dV, dK, dQ) against the forward's two.
BWD_FLOP_RATIO = 2.5


def profiled_traffic(profile_name, sources):
    """DRAM bytes per launch recorded in profiles/<profile_name>.md by an ncu
    capture, or None when the kernel sources changed since the capture."""
    path = os.path.join(ROOT, "profiles", profile_name + ".md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    s = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != _sources_sha(sources):
        return None
    return int(m.group(1))


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU is timed."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax = float(f[1])
            except ValueError:
                continue
            for name, val in zip(names, f[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": [], "samples": 0}
        loaded = [x for x in sm if smax is None or x > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- distribution

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(values, world, device=None):
    """Element-wise maximum of a list of floats over all ranks (the slowest
    replica sets the time)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.cpu().tolist()


# ------------------------------------------------------------------ oracle

def oracle_rows_tflops(w, q, k, v, rows):
    """Run the fp64 oracle on `rows` of workload `w`; returns (TFLOP/s, seconds,
    FLOPs, o, lse).  FLOPs per row = 4 d (visible keys), the same count the
    GPU metric uses (4 B H Nq Nk d, halved for causal)."""
    import numpy as np

    import oracle
    visible = (rows[:, 1] + 1) if w.causal else np.full(len(rows), w.Nk)
    flops = float(4 * w.d * visible.sum())
    t0 = time.perf_counter()
    o, lse = oracle.attention_rows(q, k, v, rows, causal=w.causal, scale=w.scale)
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, dt, flops, o, lse


def head_rows(w, bh, stride=1, offset=0):
    import numpy as np
    i = np.arange(offset, w.Nq, stride, dtype=np.int64)
    return np.stack([np.full_like(i, bh), i], axis=1)


def cpu_baseline_leg(w, q_bits, k_bits, v_bits, o_gpu=None, lse_gpu=None):
    """Time the oracle, as it stands, on whole heads of workload `w` until about
    CPU_SAMPLE_SECONDS have passed."""
    import numpy as np

    import oracle
    BH = w.B * w.H
    tot_flops, tot_s, heads = 0.0, 0.0, 0
    worst_o, worst_l = 0.0, 0.0
    order = np.random.default_rng(2024).permutation(BH)
    for bh in order:
        rows = head_rows(w, int(bh))
        _, dt, fl, o, lse = oracle_rows_tflops(w, q_bits, k_bits, v_bits, rows)
        tot_flops += fl
        tot_s += dt
        heads += 1
        if o_gpu is not None:
            og = o_gpu[int(bh)].astype(np.float64)
            worst_o = max(worst_o, float(np.abs(og - o).max()))
            worst_l = max(worst_l, float(np.abs(lse_gpu[int(bh)] - lse).max()))
        if tot_s >= CPU_SAMPLE_SECONDS:
            break
    out = {"value": tot_flops / tot_s / 1e12, "unit": "TFLOP/s", "cores": oracle.threads_used(),
           "kind": "oracle",
           "sample": f"{heads} of {BH} (b,h) heads of {w.name}, all {w.Nq} query rows each "
                     f"({tot_flops / 1e9:.1f} GFLOP in {tot_s:.1f} s, fp64 naive, OpenMP over rows)"}
    if o_gpu is not None:
        out["gpu_vs_oracle_on_sample"] = {"o_max_abs": worst_o, "lse_max_abs": worst_l}
    return out


# ------------------------------------------------------------- reference arm

def run_reference(args):
    # rank 0 alone times the oracle; the other ranks exit at once without work
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import torch  # noqa: F401

    import oracle
    from attention_flashattention_fwd_gb300.inputs import WORKLOADS, bf16_bits, make_workload
    w = WORKLOADS[LONG]
    q, k, v = make_workload(w, device="cpu")
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    BH = w.B * w.H
    stride = 32  # a step = every 32nd query row of one head (512 rows, ~2.1 GFLOP)
    times, flops = [], []
    for s in range(args.warmup + args.steps):
        rows = head_rows(w, s % BH, stride=stride, offset=s % stride)
        _, dt, fl, _, _ = oracle_rows_tflops(w, qb, kb, vb, rows)
        if s >= args.warmup:
            times.append(dt)
            flops.append(fl)
    value = sum(flops) / sum(times) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                   "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads_used(),
                         "kind": "oracle",
                         "sample": f"each step: every {stride}th query row of one (b,h) head of "
                                   f"{w.name} (fp64 naive)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def run_mma_rates(steps=4096, reps=5):
    """The tensor-core issue rates behind the kernels' issuer design (PDC
    Lecture 7 §7.13 for the CTA pair): every product of either form keeps each
    SM's tensor core busy for 64 cycles, so 64 x products / issuer cycles is the
    fraction of the time the tensor core is busy."""
    import torch

    from attention_flashattention_fwd_gb300 import binding
    torch.cuda.init()
    rows = []
    for busy in (0, 1):
        for waits in (0, 1):
            for issuer in (0, 1):
                for form in (1, 2):
                    r = binding.bench_mma_rate(form, issuer=issuer, busy=busy, waits=waits,
                                               steps=steps, reps=reps)
                    products = steps * 8
                    flops = products * 2 * 128 * 128 * 16 * r["sms"]  # either form, per SM
                    rows.append({"form": "cta_pair_m256" if form == 2 else "single_cta_m128",
                                 "issuer": "warp" if issuer else "lane", "busy": busy,
                                 "waits": waits, "sms": r["sms"], "ms": round(r["ms"], 4),
                                 "cycles_per_product": round(r["cycles"] / products, 1),
                                 "tensor_busy": round(64 * products / r["cycles"], 3),
                                 "tflops": round(flops / (r["ms"] * 1e-3) / 1e12, 1)})
    if binding.device_error() != 0:
        raise RuntimeError("attn_bench_mma_rate: a bounded wait ran out")
    print(json.dumps({"metric": "tensor-core issue rate", "steps": steps, "reps": reps,
                      "rows": rows}), flush=True)


def run_case(args):
    """One workload alone: W warm-up launches then K timed launches (used to
    profile a single kernel with ncu)."""
    import torch

    from attention_flashattention_fwd_gb300 import binding
    from attention_flashattention_fwd_gb300.inputs import (EXTRA_WORKLOADS, WORKLOADS, Workload,
                                                           make_workload)
    if args.case == "custom":
        B, H, Nq, Nk, d, causal = (int(x) for x in args.shape.split(","))
        w = Workload(f"b{B}h{H}q{Nq}k{Nk}d{d}{'_causal' if causal else ''}", B, H, Nq, Nk, d,
                     bool(causal), seed=2000)
    else:
        w = WORKLOADS[args.case] if args.case in WORKLOADS else EXTRA_WORKLOADS[args.case]
    binding.load()
    dev = torch.device("cuda", 0)
    q, k, v = make_workload(w, device=dev)
    o, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    ws = None
    if w.decode:
        ws = torch.empty(max(1, binding.decode_workspace_bytes(w.B, w.H, w.Nk, w.d)),
                         dtype=torch.uint8, device=dev)

    def launch():
        if w.decode:
            binding.attn_fwd_decode(q, k, v, scale=w.scale, out=o, lse=lse, workspace=ws)
        else:
            binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)

    flop_ratio = 1.0
    if args.which == "bwd":
        if w.decode:
            raise SystemExit("--pass bwd needs a prefill workload")
        launch()  # o, lse of these inputs
        g = torch.Generator(device=dev).manual_seed(w.seed + 7)
        dout = torch.randn(q.shape, generator=g, device=dev).to(torch.bfloat16)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        bws = torch.empty(binding.bwd_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d),
                          dtype=torch.uint8, device=dev)
        flop_ratio = BWD_FLOP_RATIO

        def launch():  # noqa: F811  (the timed call is the backward)
            binding.attn_bwd(q, k, v, o, lse, dout, causal=w.causal, scale=w.scale, dq=dq, dk=dk,
                             dv=dv, workspace=bws)
    elif args.which == "merge":
        if w.decode:
            raise SystemExit("--pass merge needs a prefill workload")
        launch()  # o, lse of these inputs, as the shards' results
        o_parts = torch.stack([o] * MERGE_PARTS).contiguous()
        l_parts = torch.stack([lse - float(s) for s in range(MERGE_PARTS)]).contiguous()
        om, lm = torch.empty_like(o), torch.empty_like(lse)
        merge_bytes = (MERGE_PARTS + 1) * (o.nbytes + lse.nbytes)

        def launch():  # noqa: F811  (the timed call is the merge)
            binding.attn_merge(o_parts, l_parts, out=om, lse=lm)
    elif args.which == "mx":
        if not w.decode:
            raise SystemExit("--pass mx needs a decode workload")
        from attention_flashattention_fwd_gb300.inputs import make_workload_mx
        del q, k, v
        qx, k8x, ksx, v8x, vsx = make_workload_mx(w, device=dev)
        mx_bytes = sum(t.nbytes for t in (qx, k8x, ksx, v8x, vsx, o, lse))

        def launch():  # noqa: F811  (the timed call is the MX decode)
            binding.attn_fwd_decode_mx(qx, k8x, ksx, v8x, vsx, scale=w.scale, out=o, lse=lse,
                                       workspace=ws)
    elif args.which == "pair":
        if w.decode or w.d != 128:
            raise SystemExit("--pass pair needs a d = 128 prefill workload")

        def launch():  # noqa: F811  (the timed call is the CTA-pair forward)
            binding.attn_fwd_cta_pair(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)
    elif args.which == "fp8":
        if w.decode or w.d != 128:
            raise SystemExit("--pass fp8 needs a d = 128 prefill workload")
        from attention_flashattention_fwd_gb300.inputs import make_workload_fp8
        del q, k, v
        q8, k8, vt8, ds8 = make_workload_fp8(w, device=dev)

        def launch():  # noqa: F811  (the timed call is the FP8 forward)
            binding.attn_fwd_fp8(q8, k8, vt8, *ds8, causal=w.causal, scale=w.scale, out=o,
                                 lse=lse)

    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(LAUNCH_COVER_CYCLES)
    e0.record()
    for _ in range(args.steps):
        launch()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    if binding.device_error() != 0:
        raise RuntimeError("a kernel reported a device-side error")
    if args.which == "mx":
        val = (mx_bytes / ms / 1e6, "GB/s")
    elif args.which == "merge":
        val = (merge_bytes / ms / 1e6, "GB/s")
    else:
        val = (w.algorithmic_bytes() / ms / 1e6, "GB/s") if w.decode else (
        flop_ratio * w.flops() / ms / 1e9, "TFLOP/s")
    print(json.dumps({"case": w.name, "pass": args.which, "ms_per_launch": ms, "value": val[0],
                      "unit": val[1], "steps": args.steps, "warmup": args.warmup,
                      "l2": "not flushed"}))


def run_gpu(args):
    rank, world, local = dist_init()
    import numpy as np
    import torch

    from attention_flashattention_fwd_gb300 import binding
    from attention_flashattention_fwd_gb300.inputs import WORKLOADS, bf16_bits, make_workload

    binding.load()  # raises if the CUDA library is missing: no fallback
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()

    w3, w4, w5 = WORKLOADS[HEADLINE], WORKLOADS[LONG], WORKLOADS[DECODE]
    q3, k3, v3 = make_workload(w3, device=dev)
    q4, k4, v4 = make_workload(w4, device=dev)
    q5, k5, v5 = make_workload(w5, device=dev)
    o3, l3 = torch.empty_like(q3), torch.empty(q3.shape[:3], dtype=torch.float32, device=dev)
    o4, l4 = torch.empty_like(q4), torch.empty(q4.shape[:3], dtype=torch.float32, device=dev)
    o5, l5 = torch.empty_like(q5), torch.empty(q5.shape[:3], dtype=torch.float32, device=dev)
    ws5 = torch.empty(max(1, binding.decode_workspace_bytes(w5.B, w5.H, w5.Nk, w5.d)),
                      dtype=torch.uint8, device=dev)
    splits = binding.decode_workspace_bytes(w5.B, w5.H, w5.Nk, w5.d) > 0
    launches_per_step = 1 + 1 + (2 if splits else 1)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another one: the write evicts
        # every line the previous work left, and the read evicts the written
        # buffer's dirty lines, so the next timed kernel neither hits in L2 nor
        # pays for writing back lines it did not produce
        flush.zero_()
        flush_rd.max()

    stream = torch.cuda.current_stream()

    def step(ev):
        flush_l2()
        # keep the GPU busy while the host enqueues this step's launches, so the
        # events below time the kernels and not host-side launch latency
        torch.cuda._sleep(LAUNCH_COVER_CYCLES)
        ev[0].record(stream)
        binding.attn_fwd(q3, k3, v3, causal=True, scale=w3.scale, out=o3, lse=l3, stream=stream)
        ev[1].record(stream)
        binding.attn_fwd(q4, k4, v4, causal=True, scale=w4.scale, out=o4, lse=l4, stream=stream)
        ev[2].record(stream)
        binding.attn_fwd_decode(q5, k5, v5, scale=w5.scale, out=o5, lse=l5, workspace=ws5,
                                stream=stream)
        ev[3].record(stream)

    def mk():
        return [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    for _ in range(args.warmup):
        step(mk())
    torch.cuda.synchronize()

    def timed_region():
        evs = [mk() for _ in range(args.steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
        barrier(world)
        torch.cuda.synchronize()
        sampler.start()
        t0.record(stream)
        for ev in evs:
            step(ev)
        t1.record(stream)
        torch.cuda.synchronize()
        sampler.stop()
        barrier(world)
        ms = [0.0, 0.0, 0.0]
        for ev in evs:
            for i in range(3):
                ms[i] += ev[i].elapsed_time(ev[i + 1])
        return ms, t0.elapsed_time(t1), sampler.summary()

    ms, total_ms, clocks = timed_region()
    if any(r in clocks["reasons"] for r in BAD_REASONS):
        ms, total_ms, clocks = timed_region()  # re-measure once
        clocks["remeasured"] = True
    if binding.device_error() != 0:
        raise RuntimeError("a kernel reported a device-side error during the benchmark")
    ms3, ms4, ms5, total_ms = max_over_ranks(ms + [total_ms], world, device=dev)
    K = args.steps

    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sfu_mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or 2070.0
    sfu_peak = SFU_EX2_PER_CLK_SM * n_sms * sfu_mhz * 1e6 / 1e12  # Texp/s

    def prefill_part(w, ms_sum, sources, prof):
        per_launch = ms_sum / K
        tflops = world * K * w.flops() / (ms_sum * 1e-3) / 1e12
        achieved = w.flops() / (per_launch * 1e-3) / 1e12
        exps = visible_pairs(w)
        exp_rate = exps / (per_launch * 1e-3) / 1e12
        return {
            "workload": w.name, "value": tflops, "unit": "TFLOP/s", "ms_per_launch": per_launch,
            "frac_of_2250": achieved / 2250.0,
            "roofline": {"bound": "tensor", "achieved": achieved,
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16_tflops"],
                         "traffic": profiled_traffic(prof, sources),
                         "peak_source": f"{peak_src} bf16 burst"},
            # secondary: the softmax's exponentials against the SFU rate
            "sfu": {"exps_per_launch": exps, "achieved": exp_rate, "peak": sfu_peak,
                    "unit": "Texp/s", "frac": exp_rate / sfu_peak,
                    "peak_source": f"{SFU_EX2_PER_CLK_SM:g} ex2/clk/SM x {n_sms} SMs x "
                                   f"{sfu_mhz:g} MHz"},
        }

    p3 = prefill_part(w3, ms3, PREFILL_SOURCES, "ncu_prefill_" + HEADLINE)
    p4 = prefill_part(w4, ms4, PREFILL_SOURCES, "ncu_prefill_" + LONG)
    per5 = ms5 / K
    gbs = w5.algorithmic_bytes() / (per5 * 1e-3) / 1e9
    p5 = {"workload": w5.name, "value": world * gbs, "unit": "GB/s", "ms_per_call": per5,
          "frac_of_8000": gbs / 8000.0,
          "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                       "frac": gbs / peaks["hbm_gbs"],
                       "traffic": profiled_traffic("ncu_decode_" + DECODE, DECODE_SOURCES),
                       "peak_source": f"{peak_src} HBM copy"}}

    # ---- end to end through the C ABI with host buffers (the long workload,
    # the line's `value`): pinned host q, k, v in, pinned host o, lse out
    qh, kh, vh = (t.cpu().pin_memory() for t in (q4, k4, v4))
    oh = torch.empty(q4.shape, dtype=torch.bfloat16).pin_memory()
    lh = torch.empty(q4.shape[:3], dtype=torch.float32).pin_memory()
    e2e_steps = min(K, 10)
    for _ in range(3):
        binding.attn_fwd_from_host(qh, kh, vh, oh, lh, q4, k4, v4, o4, l4, causal=True,
                                   scale=w4.scale, stream=stream)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        binding.attn_fwd_from_host(qh, kh, vh, oh, lh, q4, k4, v4, o4, l4, causal=True,
                                   scale=w4.scale, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    (e2e_ms,) = max_over_ranks([e0.elapsed_time(e1)], world, device=dev)
    # the host link's own rate right now: the same step's bytes as plain
    # copies, inputs in on `stream` while the results go out on a second
    # stream, no kernel.  A copy-only step is the floor under an end-to-end
    # step, and the link is shared with the rest of the machine, so it is
    # measured beside the number it bounds.
    out_stream = torch.cuda.Stream(device=dev)
    h2d_b = int(qh.nbytes + kh.nbytes + vh.nbytes)
    d2h_b = int(oh.nbytes + lh.nbytes)

    def link_pass():
        out_stream.wait_stream(stream)  # both directions start after the last pass
        with torch.cuda.stream(stream):
            for dst, src in ((q4, qh), (k4, kh), (v4, vh)):
                dst.copy_(src, non_blocking=True)
        with torch.cuda.stream(out_stream):
            oh.copy_(o4, non_blocking=True)
            lh.copy_(l4, non_blocking=True)

    def link_rate(fn):
        fn()
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(e2e_steps):
            fn()
            stream.wait_stream(out_stream)
        c1.record(stream)
        torch.cuda.synchronize()
        return c0.elapsed_time(c1) / e2e_steps

    def h2d_only():
        with torch.cuda.stream(stream):
            for dst, src in ((q4, qh), (k4, kh), (v4, vh)):
                dst.copy_(src, non_blocking=True)

    def d2h_only():
        with torch.cuda.stream(out_stream):
            out_stream.wait_stream(stream)
            oh.copy_(o4, non_blocking=True)
            lh.copy_(l4, non_blocking=True)

    # one pass in: concurrent copies in both directions ends when the inputs
    # have landed (they are the larger side); the copies alone give each
    # direction's rate
    copy_ms = link_rate(link_pass)
    h2d_ms, d2h_ms = link_rate(h2d_only), link_rate(d2h_only)
    (copy_ms, h2d_ms, d2h_ms) = max_over_ranks([copy_ms, h2d_ms, d2h_ms], world, device=dev)
    e2e = {"value": world * e2e_steps * w4.flops() / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b,
           "ms_per_step": e2e_ms / e2e_steps,
           "path": "attn_fwd_from_host (pinned host q,k,v -> device -> kernel -> host o,lse)",
           # the end-to-end step against the copy-only step of the same bytes
           "link": {"copy_only_ms_per_step": copy_ms,
                    "h2d_gbs": h2d_b / (h2d_ms * 1e-3) / 1e9,
                    "d2h_gbs": d2h_b / (d2h_ms * 1e-3) / 1e9,
                    "frac": copy_ms / (e2e_ms / e2e_steps),
                    "note": "frac = copy-only ms / end-to-end ms, both measured in this run"}}
    del qh, kh, vh, oh, lh

    # ---- the backward pass (next-row widening; not part of the timed step):
    # attn_bwd on the headline workload with the step's own o and lse, timed
    # call by call with CUDA events after an L2 flush
    g = torch.Generator(device=dev).manual_seed(w3.seed + 7)
    dout3 = torch.randn(q3.shape, generator=g, device=dev).to(torch.bfloat16)
    dq3, dk3, dv3 = torch.empty_like(q3), torch.empty_like(k3), torch.empty_like(v3)
    bws = torch.empty(binding.bwd_workspace_bytes(w3.B, w3.H, w3.Nq, w3.Nk, w3.d),
                      dtype=torch.uint8, device=dev)
    binding.attn_fwd(q3, k3, v3, causal=True, scale=w3.scale, out=o3, lse=l3, stream=stream)

    def bwd_call():
        binding.attn_bwd(q3, k3, v3, o3, l3, dout3, causal=True, scale=w3.scale, dq=dq3, dk=dk3,
                         dv=dv3, workspace=bws, stream=stream)

    for _ in range(3):
        bwd_call()
    torch.cuda.synchronize()
    bwd_reps = min(K, 20)
    bwd_ms = 0.0
    for _ in range(bwd_reps):
        flush_l2()
        torch.cuda._sleep(LAUNCH_COVER_CYCLES)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        bwd_call()
        b1.record(stream)
        torch.cuda.synchronize()
        bwd_ms += b0.elapsed_time(b1)
    if binding.device_error() != 0:
        raise RuntimeError("a kernel reported a device-side error in the backward")
    (bwd_ms,) = max_over_ranks([bwd_ms], world, device=dev)
    bwd_per = bwd_ms / bwd_reps
    bwd_flops = BWD_FLOP_RATIO * w3.flops()
    bwd_tf = bwd_flops / (bwd_per * 1e-3) / 1e12
    backward = {
        "workload": w3.name, "value": world * bwd_tf, "unit": "TFLOP/s", "ms_per_call": bwd_per,
        "calls": bwd_reps, "flops_per_call": bwd_flops,
        "timed": "attn_bwd call: prep + main + dQ convert kernels, L2 flushed before each call",
        "roofline": {"bound": "tensor", "achieved": bwd_tf, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": bwd_tf / peaks["bf16_tflops"],
                     "traffic": profiled_traffic("ncu_backward_" + HEADLINE, BACKWARD_SOURCES),
                     "peak_source": f"{peak_src} bf16 burst"},
    }

    # ---- non-causal prefill at d = 128, N = 4096 (not part of the timed step)
    from attention_flashattention_fwd_gb300.inputs import EXTRA_WORKLOADS
    wn = EXTRA_WORKLOADS["b2h16n4096d128"]
    qn, kn, vn = make_workload(wn, device=dev)
    on, ln = torch.empty_like(qn), torch.empty(qn.shape[:3], dtype=torch.float32, device=dev)
    for _ in range(3):
        binding.attn_fwd(qn, kn, vn, causal=False, scale=wn.scale, out=on, lse=ln, stream=stream)
    torch.cuda.synchronize()
    n_ms = 0.0
    for _ in range(bwd_reps):
        flush_l2()
        torch.cuda._sleep(LAUNCH_COVER_CYCLES)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        binding.attn_fwd(qn, kn, vn, causal=False, scale=wn.scale, out=on, lse=ln, stream=stream)
        b1.record(stream)
        torch.cuda.synchronize()
        n_ms += b0.elapsed_time(b1)
    (n_ms,) = max_over_ranks([n_ms], world, device=dev)
    noncausal = prefill_part(wn, n_ms * K / bwd_reps, PREFILL_SOURCES, "ncu_prefill_" + wn.name)
    noncausal["calls"] = bwd_reps
    del qn, kn, vn, on, ln

    # ---- the same headline workload through attn_fwd_cta_pair: CTA-pair
    # (cta_group::2) products, bit-identical output (not part of the timed step)
    op, lp = torch.empty_like(o3), torch.empty_like(l3)
    for _ in range(3):
        binding.attn_fwd_cta_pair(q3, k3, v3, causal=True, scale=w3.scale, out=op, lse=lp,
                                  stream=stream)
    torch.cuda.synchronize()
    c_ms = 0.0
    for _ in range(bwd_reps):
        flush_l2()
        torch.cuda._sleep(LAUNCH_COVER_CYCLES)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        binding.attn_fwd_cta_pair(q3, k3, v3, causal=True, scale=w3.scale, out=op, lse=lp,
                                  stream=stream)
        b1.record(stream)
        torch.cuda.synchronize()
        c_ms += b0.elapsed_time(b1)
    if binding.device_error() != 0:
        raise RuntimeError("a kernel reported a device-side error in the CTA-pair forward")
    (c_ms,) = max_over_ranks([c_ms], world, device=dev)
    cta_pair = prefill_part(w3, c_ms * K / bwd_reps, PAIR_SOURCES, "ncu_prefill_pair_" + w3.name)
    cta_pair["calls"] = bwd_reps
    cta_pair["entry"] = "attn_fwd_cta_pair (tcgen05.mma.cta_group::2, M = 256 over two SMs)"
    del op, lp

    # ---- FP8 (E4M3) operands on the headline workload (not part of the timed
    # step): the same Gaussian draws, per-tensor scaled to E4M3
    from attention_flashattention_fwd_gb300.inputs import make_workload_fp8
    q8, k8, vt8, ds8 = make_workload_fp8(w3, device=dev)
    o8, l8 = torch.empty_like(o3), torch.empty_like(l3)

    def fp8_call():
        binding.attn_fwd_fp8(q8, k8, vt8, *ds8, causal=True, scale=w3.scale, out=o8, lse=l8,
                             stream=stream)

    for _ in range(3):
        fp8_call()
    torch.cuda.synchronize()
    f_ms = 0.0
    for _ in range(bwd_reps):
        flush_l2()
        torch.cuda._sleep(LAUNCH_COVER_CYCLES)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        fp8_call()
        b1.record(stream)
        torch.cuda.synchronize()
        f_ms += b0.elapsed_time(b1)
    if binding.device_error() != 0:
        raise RuntimeError("a kernel reported a device-side error in the FP8 forward")
    (f_ms,) = max_over_ranks([f_ms], world, device=dev)
    f_per = f_ms / bwd_reps
    f_tf = w3.flops() / (f_per * 1e-3) / 1e12
    fp8_peak = FP8_PEAK_RATIO * peaks["bf16_tflops"]
    fp8 = {
        "workload": w3.name, "operands": "E4M3, one descale per tensor; V transposed",
        "value": world * f_tf, "unit": "TFLOP/s", "ms_per_call": f_per, "calls": bwd_reps,
        "frac_of_4500": f_tf / 4500.0,
        "roofline": {"bound": "tensor", "achieved": f_tf, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": f_tf / fp8_peak,
                     "traffic": profiled_traffic("ncu_prefill_fp8_" + w3.name, PREFILL_SOURCES),
                     "peak_source": f"{FP8_PEAK_RATIO:g} x {peak_src} bf16 burst"},
    }
    del q8, k8, vt8, o8, l8

    # ---- the decode workload with MXFP8 keys and values (not part of the timed
    # step): E4M3 codes with one E8M0 scale per 32 elements, half the bytes
    from attention_flashattention_fwd_gb300.inputs import make_workload_mx
    qx, k8x, ksx, v8x, vsx = make_workload_mx(w5, device=dev)
    ox, lx = torch.empty_like(o5), torch.empty_like(l5)

    def mx_call():
        binding.attn_fwd_decode_mx(qx, k8x, ksx, v8x, vsx, scale=w5.scale, out=ox, lse=lx,
                                   workspace=ws5, stream=stream)

    for _ in range(3):
        mx_call()
    torch.cuda.synchronize()
    x_ms = 0.0
    for _ in range(bwd_reps):
        flush_l2()
        torch.cuda._sleep(LAUNCH_COVER_CYCLES)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        mx_call()
        b1.record(stream)
        torch.cuda.synchronize()
        x_ms += b0.elapsed_time(b1)
    if binding.device_error() != 0:
        raise RuntimeError("a kernel reported a device-side error in the MX decode")
    (x_ms,) = max_over_ranks([x_ms], world, device=dev)
    x_per = x_ms / bwd_reps
    x_bytes = sum(t.nbytes for t in (qx, k8x, ksx, v8x, vsx, ox, lx))
    x_gbs = x_bytes / (x_per * 1e-3) / 1e9
    decode_mx = {
        "workload": w5.name, "operands": "K, V MXFP8 (E4M3 + one E8M0 scale per 32)",
        "value": world * x_gbs, "unit": "GB/s", "ms_per_call": x_per, "calls": bwd_reps,
        "bytes_per_call": x_bytes, "speedup_vs_bf16_decode": per5 / x_per,
        "roofline": {"bound": "hbm", "achieved": x_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": x_gbs / peaks["hbm_gbs"],
                     "traffic": profiled_traffic("ncu_decode_mx_" + DECODE, DECODE_SOURCES),
                     "peak_source": f"{peak_src} HBM copy"},
    }
    del qx, k8x, ksx, v8x, vsx, ox, lx

    # ---- the exchange step of key-sharded attention (not part of the timed step):
    # attn_merge of MERGE_PARTS shard results of the headline shape
    o_parts = torch.stack([o3] * MERGE_PARTS).contiguous()
    l_parts = torch.stack([l3 - float(s) for s in range(MERGE_PARTS)]).contiguous()
    om, lm = torch.empty_like(o3), torch.empty_like(l3)
    for _ in range(3):
        binding.attn_merge(o_parts, l_parts, out=om, lse=lm, stream=stream)
    torch.cuda.synchronize()
    m_ms = 0.0
    for _ in range(bwd_reps):
        flush_l2()
        torch.cuda._sleep(LAUNCH_COVER_CYCLES)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        binding.attn_merge(o_parts, l_parts, out=om, lse=lm, stream=stream)
        b1.record(stream)
        torch.cuda.synchronize()
        m_ms += b0.elapsed_time(b1)
    (m_ms,) = max_over_ranks([m_ms], world, device=dev)
    m_per = m_ms / bwd_reps
    m_bytes = (MERGE_PARTS + 1) * (o3.nbytes + l3.nbytes)
    m_gbs = m_bytes / (m_per * 1e-3) / 1e9
    merge = {
        "workload": f"{MERGE_PARTS} shard results of {w3.name}", "value": world * m_gbs,
        "unit": "GB/s", "ms_per_call": m_per, "calls": bwd_reps, "bytes_per_call": m_bytes,
        "roofline": {"bound": "hbm", "achieved": m_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": m_gbs / peaks["hbm_gbs"],
                     "traffic": profiled_traffic("ncu_merge_" + w3.name, MERGE_SOURCES),
                     "peak_source": f"{peak_src} HBM copy"},
    }

    line = {
        "metric": METRIC, "value": p4["value"], "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": total_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded iid Gaussian Q,K,V rounded to bf16)",
        "config": {"workload": LONG, "B": w4.B, "H": w4.H, "Nq": w4.Nq, "Nk": w4.Nk,
                   "d": w4.d, "causal": True, "scale": w4.scale,
                   "step": f"prefill {HEADLINE} + prefill {LONG} + decode {DECODE}",
                   "l2": "flushed before every step (256 MiB write, then a 256 MiB read)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": p4["roofline"],
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": launches_per_step * K,
        "parts": {HEADLINE: p3, LONG: p4, DECODE: p5},
        "noncausal": noncausal,
        "cta_pair": cta_pair,
        "fp8": fp8,
        "decode_mx": decode_mx,
        "backward": backward,
        "merge": merge,
    }

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        BH = w4.B * w4.H
        o_np = o4.reshape(BH, w4.Nq, w4.d).float().cpu().numpy()
        l_np = l4.reshape(BH, w4.Nq).cpu().numpy()
        line["cpu_baseline"] = cpu_baseline_leg(w4, bf16_bits(q4), bf16_bits(k4), bf16_bits(v4),
                                                o_np, l_np)

    # last: one compact entry per measured kernel (value, unit, fraction of its
    # measured roofline, ms per launch), so the end of the line holds them all
    def brief(part, ms_key):
        r = part["roofline"]
        return [round(part["value"], 1), part["unit"], round(r["frac"], 3),
                round(part[ms_key], 4)]

    line["summary"] = {
        "fields": ["value", "unit", "frac_of_measured_peak", "ms_per_launch"],
        "prefill_" + LONG: brief(p4, "ms_per_launch"),
        "prefill_" + HEADLINE: brief(p3, "ms_per_launch"),
        "prefill_" + wn.name: brief(noncausal, "ms_per_launch"),
        "cta_pair_" + w3.name: brief(cta_pair, "ms_per_launch"),
        "decode_" + w5.name.replace("decode_", ""): brief(p5, "ms_per_call"),
        "decode_mx_" + w5.name.replace("decode_", ""): brief(decode_mx, "ms_per_call"),
        "fp8_" + w3.name: brief(fp8, "ms_per_call"),
        "backward_" + w3.name: brief(backward, "ms_per_call"),
        "merge4_" + w3.name: brief(merge, "ms_per_call"),
        "e2e_" + LONG: [round(e2e["value"], 1), e2e["unit"], round(e2e["link"]["frac"], 3),
                         round(e2e["ms_per_step"], 4)],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.mma_rates:
        run_mma_rates()
        return
    if args.case:
        run_case(args)
        return
    run_gpu(args)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
