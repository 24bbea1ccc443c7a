"""attn_fwd_decode_no_alloc: the decode entry point for callers that cannot
allocate device memory (a plugin whose host application owns all device
memory, or a serving loop that may not call cudaMalloc because it can
synchronise the device).  It keeps its split partials in a fixed scratch array
inside the library instead of a caller workspace.

The test calls it through the C ABI twice in a row, on different inputs (the
second call finds the first call's partials in the scratch), with outputs
filled with NaN beforehand.  It runs the same split plan and the same two
kernels as attn_fwd_decode, so each result must equal attn_fwd_decode's (with
its own workspace) bit for bit; both are also checked against the fp64 oracle
within the tolerances the other tests use.  One shape is decoded in a single
split, where the scratch is not used at all.  This file is named so that
pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import bf16_bits, make_qkv

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 2e-3
SCRATCH_BYTES = 2 << 20  # ATTN_DECODE_NO_ALLOC_SCRATCH_BYTES in include/gbattn.h

pytestmark = pytest.mark.gpu


def _no_alloc():
    lib = binding.load()
    fn = lib.attn_fwd_decode_no_alloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, P, P, I, I, I, I, F, P]
    fn.restype = I
    return fn


def _call(fn, q, k, v, o, lse, scale):
    B, H, _, d = q.shape
    Nk = k.shape[2]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
              ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()),
              ctypes.c_void_p(lse.data_ptr()), B, H, Nk, d, scale, stream)


# (8, 16, 4096, 128) and (3, 5, 3000, 64) split their keys; (4, 8, 500, 128)
# has one split by its size, (64, 40, 1000, 64) has 2560 heads, enough for one
# split each on a GB300 (16 CTAs per SM), though its workspace bound is not 0.
@pytest.mark.parametrize("B,H,Nk,d", [(8, 16, 4096, 128), (3, 5, 3000, 64), (4, 8, 500, 128),
                                      (64, 40, 1000, 64)])
def test_no_alloc_matches_decode_on_two_calls_in_a_row(B, H, Nk, d):
    fn = _no_alloc()
    assert binding.decode_workspace_bytes(B, H, Nk, d) <= SCRATCH_BYTES
    scale = d ** -0.5
    for seed in (71, 72):  # the second call sees the first call's scratch contents
        q, k, v = make_qkv(B, H, 1, Nk, d, seed=seed + Nk, device="cuda")
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, 1), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(fn, q, k, v, o, lse, scale) == 0
        ro = torch.full_like(q, float("nan"))
        rl = torch.full_like(lse, float("nan"))
        ws = torch.full((max(1, binding.decode_workspace_bytes(B, H, Nk, d)),), 0xFF,
                        dtype=torch.uint8, device="cuda")
        binding.attn_fwd_decode(q, k, v, scale=scale, out=ro, lse=rl, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(o, ro) and torch.equal(lse, rl), "differs from attn_fwd_decode"
        eo, el = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), scale=scale)
        e = np.abs(o.float().cpu().numpy() - eo)
        e_l = np.abs(lse.cpu().numpy() - el)
        assert e.max() <= O_MAX and e.mean() <= O_MEAN and e_l.max() <= LSE_MAX, (
            f"O max {e.max():.3g} mean {e.mean():.3g}, lse max {e_l.max():.3g}")
    assert binding.device_error() == 0


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    fn = _no_alloc()
    B, H, Nk, d = 64, 32, 8192, 128  # 16 splits x 2048 heads x 129 floats > 2 MiB
    assert binding.decode_workspace_bytes(B, H, Nk, d) > SCRATCH_BYTES
    q = torch.zeros((1, 1, 1, d), dtype=torch.bfloat16, device="cuda")  # never read
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 1), dtype=torch.float32, device="cuda")
    P = ctypes.c_void_p
    st = fn(P(q.data_ptr()), P(q.data_ptr()), P(q.data_ptr()), P(o.data_ptr()),
            P(lse.data_ptr()), B, H, Nk, d, 0.1, P(torch.cuda.current_stream().cuda_stream))
    assert st == 2  # ATTN_ERR_UNSUPPORTED, nothing launched
    torch.cuda.synchronize()
    assert binding.device_error() == 0
