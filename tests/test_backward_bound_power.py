"""The tight bound of `test_backward_emulated_gpu.py` notices the mistakes it is
meant to (CPU only): the emulated backward with a planted mistake -- one key
wrongly visible to one late query row, or D dropped from dS for one row -- is
compared with the correct emulation under that bound and must fail it.  The
forward statistics come from the fp64 oracle, as in the GPU test."""
import numpy as np
import torch

import oracle
from attention_flashattention_fwd_gb300.inputs import bf16_bits, make_qkv
from tests.test_backward_emulated_gpu import REL, RMS, _bf16, _emulate


def _fails_bound(got, ref):
    rms = float(np.sqrt(np.mean(ref * ref)))
    return (np.abs(got - ref) - REL * np.abs(ref)).max() > RMS * rms


def _case(B=1, H=1, N=300, d=64, causal=True, seed=191):
    q, k, v = make_qkv(B, H, N, N, d, seed=seed)
    dout = torch.randn(q.shape, generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16)
    scale = d ** -0.5
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=causal,
                              scale=scale)
    o = torch.from_numpy(ro).to(torch.bfloat16).double().numpy()
    lse = torch.from_numpy(rl).to(torch.float32).double().numpy()
    f64 = [t.double().numpy() for t in (q, k, v, dout)]
    return f64, o, lse, scale


def test_bound_holds_for_the_correct_emulation_against_itself_rounded_differently():
    # sanity: the emulation with fp32 inputs to the final rounding stays in the bound
    (q, k, v, dout), o, lse, scale = _case()
    ref = _emulate(q, k, v, dout, o, lse, True, scale)
    again = _emulate(q, k, v, dout, o, lse.astype(np.float32).astype(np.float64), True, scale)
    for a, b in zip(again, ref):
        assert not _fails_bound(a, b)


def test_bound_catches_one_key_unmasked_for_a_late_row():
    (q, k, v, dout), o, lse, scale = _case()
    ref = _emulate(q, k, v, dout, o, lse, True, scale)
    i = 290  # query row 290 also sees key 291 (its future)
    s = np.einsum("bhid,bhjd->bhij", q, k)
    mask = np.arange(300)[None, :] > np.arange(300)[:, None]
    mask[i, i + 1] = False
    s = np.where(mask, -np.inf, s)
    p = _bf16(np.exp(scale * s - lse[..., None]))
    dp = np.einsum("bhid,bhjd->bhij", dout, v)
    D = np.sum(dout * o, axis=-1)
    ds = _bf16(p * (dp - D[..., None]))
    dq = _bf16(scale * np.einsum("bhij,bhjd->bhid", ds, k))
    dk = _bf16(scale * np.einsum("bhij,bhid->bhjd", ds, q))
    dv = _bf16(np.einsum("bhij,bhid->bhjd", p, dout))
    assert any(_fails_bound(g, r) for g, r in zip((dq, dk, dv), ref))


def test_bound_catches_D_dropped_for_one_row():
    (q, k, v, dout), o, lse, scale = _case(causal=False, seed=193)
    ref = _emulate(q, k, v, dout, o, lse, False, scale)
    s = np.einsum("bhid,bhjd->bhij", q, k)
    p = _bf16(np.exp(scale * s - lse[..., None]))
    dp = np.einsum("bhid,bhjd->bhij", dout, v)
    D = np.sum(dout * o, axis=-1)
    D[..., 150] = 0.0
    ds = _bf16(p * (dp - D[..., None]))
    dq = _bf16(scale * np.einsum("bhij,bhjd->bhid", ds, k))
    assert _fails_bound(dq, ref[0])
