"""The failure path on the GPU, without a fault: a kernel waits on a barrier
that nothing ever arrives on; the bounded wait gives up, the device error
word reports it (ATTN_ERR_TIMEOUT) and is cleared by the read, and the
context keeps working."""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import bf16_bits, make_qkv

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_reports_and_recovers():
    lib = binding.load()
    assert binding.device_error() == 0
    t0 = time.monotonic()
    st = lib.attn_selftest_timeout(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    assert binding.device_error() == 5  # ATTN_ERR_TIMEOUT, after the 2 s limit
    assert 1.5 <= time.monotonic() - t0 <= 60.0
    assert binding.device_error() == 0  # cleared by the read
    # the context is still usable: an attention call afterwards is correct
    q, k, v = make_qkv(1, 2, 200, 200, 64, seed=97, device="cuda")
    o, lse = binding.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=True)
    assert np.abs(o.float().cpu().numpy() - ro).max() <= 2e-2
    assert np.abs(lse.cpu().numpy() - rl).max() <= 2e-3
    assert binding.device_error() == 0
