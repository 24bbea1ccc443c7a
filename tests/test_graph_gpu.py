"""CUDA-graph capture of the library's calls.

Every entry point only enqueues work on the caller's stream: kernel launches,
and for the host-buffer path copies plus event waits that fork the library's
own streams from the caller's stream and join them back.  Nothing synchronises
or allocates after the first call, so a whole sequence of calls can be captured
once and replayed with new inputs written into the same buffers.  The forward
kernels are deterministic (a fixed schedule, no atomics), so a replay must
reproduce the eager calls bit for bit; the backward's dQ is summed with
reduce-adds whose order varies, so it is compared within fp32 rounding.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import bf16_bits, make_qkv, make_qkv_fp8, make_qkv_mx
from tests.conftest import nan_full

pytestmark = pytest.mark.gpu

B, H, NQ, NK, D = 1, 4, 384, 512, 128


def _fill(bufs, seed):
    """Seeded inputs of the captured sequence, written in place."""
    dev = bufs["q"].device
    q, k, v = make_qkv(B, H, NQ, NK, D, seed=seed, device=dev)
    bufs["q"].copy_(q)
    bufs["k"].copy_(k)
    bufs["v"].copy_(v)
    half = NK // 2
    bufs["k0"].copy_(k[:, :, :half])
    bufs["k1"].copy_(k[:, :, half:])
    bufs["v0"].copy_(v[:, :, :half])
    bufs["v1"].copy_(v[:, :, half:])
    bufs["qd"].copy_(q[:, :, -1:])
    q8, k8, vt8, _ = make_qkv_fp8(B, H, NQ, NK, D, seed=seed + 1, device=dev)
    bufs["q8"].copy_(q8.view(torch.uint8))
    bufs["k8"].copy_(k8.view(torch.uint8))
    bufs["vt8"].copy_(vt8.view(torch.uint8))
    g = torch.Generator(device="cpu").manual_seed(seed + 2)
    bufs["dout"].copy_(torch.randn(B, H, NQ, D, generator=g).to(torch.bfloat16))
    _, kx, ksx, vx, vsx = make_qkv_mx(B, H, NK, D, seed=seed + 3, device=dev)
    for n, t in (("kx", kx), ("ksx", ksx), ("vx", vx), ("vsx", vsx)):
        bufs[n].copy_(t)


def _buffers(dev):
    bf, f32, u8 = torch.bfloat16, torch.float32, torch.uint8
    half = NK // 2
    z = lambda shape, dt: torch.zeros(shape, dtype=dt, device=dev)  # noqa: E731
    return {
        "q": z((B, H, NQ, D), bf), "k": z((B, H, NK, D), bf), "v": z((B, H, NK, D), bf),
        "k0": z((B, H, half, D), bf), "k1": z((B, H, half, D), bf),
        "v0": z((B, H, half, D), bf), "v1": z((B, H, half, D), bf),
        "qd": z((B, H, 1, D), bf),
        "q8": z((B, H, NQ, D), u8), "k8": z((B, H, NK, D), u8), "vt8": z((B, H, D, NK), u8),
        "dout": z((B, H, NQ, D), bf),
        "kx": z((B, H, NK, D), u8), "ksx": z((B, H, NK, D // 32), u8),
        "vx": z((B, H, NK, D), u8), "vsx": z((B, H, NK, D // 32), u8),
        "ox": z((B, H, 1, D), bf), "lx": z((B, H, 1), f32),
        # outputs
        "o": z((B, H, NQ, D), bf), "lse": z((B, H, NQ), f32),
        "o8": z((B, H, NQ, D), bf), "lse8": z((B, H, NQ), f32),
        "oc": z((B, H, NQ, D), bf), "lc": z((B, H, NQ), f32),
        "op": z((2, B, H, NQ, D), bf), "lp": z((2, B, H, NQ), f32),
        "om": z((B, H, NQ, D), bf), "lm": z((B, H, NQ), f32),
        "od": z((B, H, 1, D), bf), "ld": z((B, H, 1), f32),
        "dq": z((B, H, NQ, D), bf), "dk": z((B, H, NK, D), bf), "dv": z((B, H, NK, D), bf),
        "ws_dec": z(max(1, binding.decode_workspace_bytes(B, H, NK, D)), u8),
        "ws_bwd": z(binding.bwd_workspace_bytes(B, H, NQ, NK, D), u8),
    }


OUTPUTS = ("o", "lse", "oc", "lc", "o8", "lse8", "op", "lp", "om", "lm", "od", "ld", "ox", "lx", "dk", "dv")


def _step(b):
    """One pass over the entry points: causal prefill (single-CTA and CTA-pair
    products), FP8 prefill, two key shards merged, one decode row (bf16 and
    MXFP8 keys and values), and the backward of the causal prefill."""
    binding.attn_fwd(b["q"], b["k"], b["v"], causal=True, out=b["o"], lse=b["lse"])
    binding.attn_fwd_cta_pair(b["q"], b["k"], b["v"], causal=True, out=b["oc"], lse=b["lc"])
    binding.attn_fwd_fp8(b["q8"], b["k8"], b["vt8"], 0.05, 0.05, 0.05, causal=True,
                         out=b["o8"], lse=b["lse8"])
    binding.attn_fwd(b["q"], b["k0"], b["v0"], out=b["op"][0], lse=b["lp"][0])
    binding.attn_fwd(b["q"], b["k1"], b["v1"], out=b["op"][1], lse=b["lp"][1])
    binding.attn_merge(b["op"], b["lp"], out=b["om"], lse=b["lm"])
    binding.attn_fwd_decode(b["qd"], b["k"], b["v"], out=b["od"], lse=b["ld"],
                            workspace=b["ws_dec"])
    binding.attn_fwd_decode_mx(b["qd"], b["kx"], b["ksx"], b["vx"], b["vsx"], out=b["ox"],
                               lse=b["lx"], workspace=b["ws_dec"])
    binding.attn_bwd(b["q"], b["k"], b["v"], o=b["o"], lse=b["lse"], dout=b["dout"],
                     causal=True, dq=b["dq"], dk=b["dk"], dv=b["dv"], workspace=b["ws_bwd"])


def test_graph_replay_matches_eager_calls():
    dev = torch.device("cuda:0")
    b = _buffers(dev)
    _fill(b, seed=11)
    _step(b)  # first calls: one-time initialisation happens outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _step(b)
    for seed in (101, 202):
        _fill(b, seed)
        graph.replay()
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        replayed = {n: b[n].clone() for n in OUTPUTS + ("dq",)}
        _step(b)
        torch.cuda.synchronize()
        for n in OUTPUTS:
            assert torch.equal(replayed[n], b[n]), f"seed {seed}: {n} differs between replay and eager"
        dq_r, dq_e = replayed["dq"].float(), b["dq"].float()
        assert (dq_r - dq_e).abs().max() <= 2.0 ** -8 * dq_e.abs().max() + 1e-6
        # the replay computed attention, not stale buffers: the causal prefill
        # against the fp64 oracle on this seed's inputs
        ro, rl = oracle.attention(bf16_bits(b["q"]), bf16_bits(b["k"]), bf16_bits(b["v"]),
                                  causal=True)
        assert torch.equal(replayed["oc"], replayed["o"]) and torch.equal(replayed["lc"], replayed["lse"])
        e = np.abs(replayed["o"].float().cpu().numpy() - ro)
        el = np.abs(replayed["lse"].cpu().numpy() - rl)
        assert e.max() <= 2e-2 and e.mean() <= 1e-3 and el.max() <= 2e-3


def test_graph_replay_host_buffer_path():
    """attn_fwd_from_host captured: its H2D copies, the chunked kernels on the
    library's compute stream and the D2H copies on its copy-out stream become
    one graph; a replay after new values land in the pinned inputs returns the
    same host outputs as an eager call."""
    dev = torch.device("cuda:0")
    h = {n: nan_full(s, dt, pin=True) for n, s, dt in (
        ("q", (B, H, NQ, D), torch.bfloat16), ("k", (B, H, NK, D), torch.bfloat16),
        ("v", (B, H, NK, D), torch.bfloat16), ("o", (B, H, NQ, D), torch.bfloat16),
        ("lse", (B, H, NQ), torch.float32))}
    d = {"dq": nan_full((B, H, NQ, D), torch.bfloat16, dev),
         "dk": nan_full((B, H, NK, D), torch.bfloat16, dev),
         "dv": nan_full((B, H, NK, D), torch.bfloat16, dev),
         "do_": nan_full((B, H, NQ, D), torch.bfloat16, dev),
         "dlse": nan_full((B, H, NQ), torch.float32, dev)}

    def fill(seed):
        q, k, v = make_qkv(B, H, NQ, NK, D, seed=seed, device="cpu")
        h["q"].copy_(q)
        h["k"].copy_(k)
        h["v"].copy_(v)

    def call():
        binding.attn_fwd_from_host(h["q"], h["k"], h["v"], h["o"], h["lse"], d["dq"], d["dk"],
                                   d["dv"], d["do_"], d["dlse"], causal=True)

    fill(7)
    call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for seed in (303, 404):
        fill(seed)
        h["o"].fill_(float("nan"))
        h["lse"].fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        o_r, lse_r = h["o"].clone(), h["lse"].clone()
        call()
        torch.cuda.synchronize()
        assert torch.equal(o_r, h["o"]) and torch.equal(lse_r, h["lse"]), f"seed {seed}"
        ro, rl = oracle.attention(bf16_bits(h["q"]), bf16_bits(h["k"]), bf16_bits(h["v"]),
                                  causal=True)
        assert np.abs(o_r.float().numpy() - ro).max() <= 2e-2
        assert np.abs(lse_r.numpy() - rl).max() <= 2e-3
