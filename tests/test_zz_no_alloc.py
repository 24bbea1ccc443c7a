"""attn_fwd_decode_no_alloc: the decode entry point for callers that cannot
allocate device memory (a plugin whose host application owns all device
memory, or a serving loop that may not call cudaMalloc because it can
synchronise the device).  It keeps its split partials in a fixed scratch array
inside the library instead of a caller workspace.

The test calls it through the C ABI twice in a row, on different inputs, and
checks each result against the existing attn_fwd_decode entry point (with its
own workspace) within the tolerances the other tests use.  This file is named
so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import make_qkv

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


@pytest.mark.parametrize("B,H,Nk,d", [(8, 16, 4096, 128), (3, 5, 3000, 64)])
def test_no_alloc_matches_decode_on_two_calls_in_a_row(B, H, Nk, d):
    fn = _no_alloc()
    assert binding.decode_workspace_bytes(B, H, Nk, d) > 0  # the scratch is really used
    assert binding.decode_workspace_bytes(B, H, Nk, d) <= SCRATCH_BYTES
    scale = d ** -0.5
    for seed in (71, 72):  # the second call sees the first call's scratch contents
        q, k, v = make_qkv(B, H, 1, Nk, d, seed=seed, device="cuda")
        o = torch.empty_like(q)
        lse = torch.empty((B, H, 1), dtype=torch.float32, device="cuda")
        assert _call(fn, q, k, v, o, lse, scale) == 0
        ro, rl = binding.attn_fwd_decode(q, k, v, scale=scale)
        torch.cuda.synchronize()
        e = (o.float() - ro.float()).abs()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        assert e.max().item() <= O_MAX and e.mean().item() <= O_MEAN
        assert (lse - rl).abs().max().item() <= LSE_MAX


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    fn = _no_alloc()
    B, H, Nk, d = 64, 32, 8192, 128  # 2 splits x 2048 heads x 129 floats > 2 MiB
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
