"""The binding refuses buffers the kernels would write past or read from the
wrong device: a caller's output of the wrong shape, dtype or layout, a
workspace or sequence-length tensor on the host, a host-buffer argument of the
wrong dtype.  Each is a ValueError raised before the C entry point is called,
and nothing is written."""
import pytest
import torch

from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

B, H, NQ, NK, D = 1, 2, 130, 260, 64


def _qkv():
    return make_qkv(B, H, NQ, NK, D, seed=404, device="cuda")


@pytest.mark.parametrize("bad", [
    dict(out=torch.empty((B, H, NQ - 1, D), dtype=torch.bfloat16)),          # shape
    dict(out=torch.empty((B, H, NQ, D), dtype=torch.float16)),               # dtype
    dict(out=torch.empty((B, H, D, NQ), dtype=torch.bfloat16).transpose(2, 3)),  # layout
    dict(lse=torch.empty((B, H, NQ + 1), dtype=torch.float32)),
    dict(lse=torch.empty((B, H, NQ), dtype=torch.float64)),
], ids=["out_shape", "out_dtype", "out_strided", "lse_shape", "lse_dtype"])
def test_attn_fwd_refuses_mismatched_outputs(bad):
    q, k, v = _qkv()
    sentinel = {}
    for name, t in bad.items():
        bad[name] = t.to("cuda").fill_(7)
        sentinel[name] = bad[name].clone()
    with pytest.raises(ValueError):
        binding.attn_fwd(q, k, v, causal=True, **bad)
    torch.cuda.synchronize()
    for name, t in bad.items():
        assert torch.equal(t, sentinel[name]), f"{name} was written"


def test_outputs_on_the_host_are_refused():
    q, k, v = _qkv()
    with pytest.raises(ValueError):
        binding.attn_fwd(q, k, v, out=torch.empty((B, H, NQ, D), dtype=torch.bfloat16))


def test_decode_refuses_host_workspace_and_wrong_outputs():
    q, k, v = make_qkv(B, H, 1, 5000, D, seed=405, device="cuda")
    with pytest.raises(ValueError):
        binding.attn_fwd_decode(q, k, v, workspace=torch.empty(1 << 20, dtype=torch.uint8))
    with pytest.raises(ValueError):
        binding.attn_fwd_decode(q, k, v, out=torch.empty((B, H, 2, D), dtype=torch.bfloat16,
                                                         device="cuda"))


def test_backward_refuses_mismatched_gradient_buffers():
    q, k, v = _qkv()
    o, lse = binding.attn_fwd(q, k, v, causal=True)
    dout = torch.randn_like(q)
    with pytest.raises(ValueError):
        binding.attn_bwd(q, k, v, o, lse, dout, causal=True, dk=torch.empty_like(q))
    with pytest.raises(ValueError):
        binding.attn_bwd(q, k, v, o, lse, dout, causal=True, dq=torch.empty_like(q).float())
    with pytest.raises(ValueError):
        binding.attn_bwd(q, k, v, o, lse.cpu(), dout, causal=True)


def test_ragged_refuses_host_lengths():
    q, k, v = _qkv()
    with pytest.raises(ValueError):
        binding.attn_fwd_ragged(q, k, v, seqlens_k=torch.full((B,), NK, dtype=torch.int32))


def test_merge_refuses_mismatched_outputs():
    o_parts = torch.zeros((2, B, H, NQ, D), dtype=torch.bfloat16, device="cuda")
    lse_parts = torch.zeros((2, B, H, NQ), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        binding.attn_merge(o_parts, lse_parts, lse=torch.empty((B, H, NQ, 1), device="cuda"))


def test_host_path_refuses_wrong_host_dtype():
    q, k, v = (t.cpu() for t in _qkv())
    o = torch.empty((B, H, NQ, D), dtype=torch.float32)  # should be bf16
    lse = torch.empty((B, H, NQ), dtype=torch.float32)
    dq, dk, dv = (torch.empty_like(t, device="cuda") for t in (q, k, v))
    with pytest.raises(ValueError):
        binding.attn_fwd_from_host(q, k, v, o, lse, dq, dk, dv, torch.empty_like(dq),
                                   torch.empty((B, H, NQ), device="cuda"))


def test_host_path_refuses_pageable_host_memory():
    # pageable buffers would turn the pipelined copies synchronous
    q, k, v = (t.cpu() for t in _qkv())
    o = torch.empty((B, H, NQ, D), dtype=torch.bfloat16)
    lse = torch.empty((B, H, NQ), dtype=torch.float32)
    dq, dk, dv = (torch.empty_like(t, device="cuda") for t in (q, k, v))
    with pytest.raises(ValueError, match="pinned"):
        binding.attn_fwd_from_host(q, k, v, o, lse, dq, dk, dv, torch.empty_like(dq),
                                   torch.empty((B, H, NQ), device="cuda"))
