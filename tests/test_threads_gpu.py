"""Calls from several host threads at once.

The library's shared host state is a once-initialised table of kernel
attributes, a cached SM count per device and the streams and events of the
host-buffer path (its enqueue serialised by a mutex); everything else is per
call.  A fresh process starts six threads that make their first calls
together, so the one-time initialisation itself is raced: four run attn_fwd
on their own streams (both head sizes, causal and not), two run
attn_fwd_from_host.  Every result must equal a sequential rerun bit for bit
(the kernels are deterministic).
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent(r"""
    import sys, threading
    import torch
    from attention_flashattention_fwd_gb300 import binding
    from attention_flashattention_fwd_gb300.inputs import make_qkv

    def nan_full(shape, dtype, device=None, pin=False):
        t = torch.full(tuple(shape), float("nan"), dtype=dtype, device=device)
        return t.pin_memory() if pin else t

    dev = torch.device("cuda:0")
    torch.cuda.init()
    DEVICE_CASES = [  # B, H, Nq, Nk, d, causal
        (1, 3, 300, 300, 128, True), (2, 2, 257, 513, 64, False),
        (1, 5, 128, 640, 128, True), (3, 1, 700, 700, 64, True)]
    HOST_CASES = [(1, 4, 200, 200, 128, True), (2, 3, 130, 260, 64, False)]

    def dev_inputs(i):
        B, H, Nq, Nk, d, c = DEVICE_CASES[i]
        return make_qkv(B, H, Nq, Nk, d, seed=900 + i, device=dev), c

    def host_buffers(i):
        B, H, Nq, Nk, d, c = HOST_CASES[i]
        q, k, v = make_qkv(B, H, Nq, Nk, d, seed=950 + i, device="cpu")
        pin = lambda t: t.pin_memory()
        h = dict(q=pin(q), k=pin(k), v=pin(v),
                 o=nan_full((B, H, Nq, d), torch.bfloat16, pin=True),
                 lse=nan_full((B, H, Nq), torch.float32, pin=True))
        dd = dict(dq=nan_full(q.shape, q.dtype, dev), dk=nan_full(k.shape, k.dtype, dev),
                  dv=nan_full(v.shape, v.dtype, dev), do_=nan_full(q.shape, q.dtype, dev),
                  dlse=nan_full((B, H, Nq), torch.float32, dev))
        return h, dd, c

    dev_in = [dev_inputs(i) for i in range(len(DEVICE_CASES))]
    host_in = [host_buffers(i) for i in range(len(HOST_CASES))]
    results = {}
    errors = []
    gate = threading.Barrier(len(dev_in) + len(host_in))

    def run_dev(i):
        try:
            (q, k, v), c = dev_in[i]
            s = torch.cuda.Stream(device=dev)
            gate.wait()
            with torch.cuda.stream(s):
                for _ in range(3):
                    o, lse = binding.attn_fwd(q, k, v, causal=c, stream=s)
            s.synchronize()
            results[("dev", i)] = (o.cpu(), lse.cpu())
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    def run_host(i):
        try:
            h, dd, c = host_in[i]
            s = torch.cuda.Stream(device=dev)
            gate.wait()
            for _ in range(3):
                binding.attn_fwd_from_host(h["q"], h["k"], h["v"], h["o"], h["lse"], dd["dq"],
                                           dd["dk"], dd["dv"], dd["do_"], dd["dlse"], causal=c,
                                           stream=s)
            s.synchronize()
            results[("host", i)] = (h["o"].clone(), h["lse"].clone())
        except Exception as e:
            errors.append(repr(e))

    threads = [threading.Thread(target=run_dev, args=(i,)) for i in range(len(dev_in))]
    threads += [threading.Thread(target=run_host, args=(i,)) for i in range(len(host_in))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a thread did not finish"
    assert not errors, errors
    assert binding.device_error() == 0

    # sequential reruns on the default stream
    for i in range(len(dev_in)):
        (q, k, v), c = dev_in[i]
        o, lse = binding.attn_fwd(q, k, v, causal=c)
        torch.cuda.synchronize()
        ro, rl = results[("dev", i)]
        assert torch.equal(ro, o.cpu()) and torch.equal(rl, lse.cpu()), ("dev", i)
    for i in range(len(host_in)):
        h, dd, c = host_in[i]
        ro, rl = results[("host", i)]
        h["o"].fill_(float("nan"))
        h["lse"].fill_(float("nan"))
        binding.attn_fwd_from_host(h["q"], h["k"], h["v"], h["o"], h["lse"], dd["dq"], dd["dk"],
                                   dd["dv"], dd["do_"], dd["dlse"], causal=c)
        torch.cuda.synchronize()
        assert torch.equal(ro, h["o"]) and torch.equal(rl, h["lse"]), ("host", i)
    print("threads ok")
""")


def test_concurrent_first_calls_from_threads():
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and "threads ok" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])
