"""The CUDA backward against a host emulation of its own rounding steps, with a
tight per-element bound.

`test_backward_gpu.py` compares attn_bwd with the exact fp64 gradients under a
bound derived from the roundings the kernel makes (P and dS rounded to bf16
before the dV, dK and dQ products; D from the bf16 forward output); that bound
must allow the legitimate rounding error of every element, which is large
next to, e.g., one key wrongly masked for a late query row (weight about 1/i).
Here the reference makes the same roundings at the same points, in fp64:

    P   = bf16(exp(scale s - lse))         dP = dO V^T
    D   = rowsum(dO * O)                   dS = bf16(P (dP - D))
    dV  = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K,  each rounded to bf16

with O and lse taken from the fp64 oracle (rounded to bf16 and fp32) and passed
to the kernel as well, so both sides start from the same forward statistics.
What remains between the two is fp32 against fp64 arithmetic inside the
kernel (scores, exponentials, sums: relative 2^-20 or less), which moves a
rounded P or dS by one bf16 unit only when it lies next to a rounding boundary,
and the last unit of the final bf16 rounding.  Two values rounded to bf16 from
pre-rounding values a and b differ by at most |a - b| plus one unit, and a unit
is at most 2^-7 of the value, so per element
    |got - emu| <= 2^-7 |emu| + delta,    delta = |a - b| <= 2^-7 rms(emu),
where delta collects the flipped P / dS units (each 2^-8 of one term of a sum of
many) and fp32 summation; the largest delta measured over these cases is
0.0034 rms (2^-8.2).  The exact-gradient test allows 2^-3 rms beyond its
rounding term; this one allows 16x less.  A key wrongly masked for query row i
changes dQ_i by about scale |dS_ij| |k_j| with |dS_ij| ~ 1/i, several percent of
rms(dQ) for these sizes.  The emulation is the tests' own numpy; it shares
nothing with the CUDA path.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import bf16_bits, make_qkv

pytestmark = pytest.mark.gpu

REL, RMS = 2.0 ** -7, 2.0 ** -7


def _bf16(x):
    """Round float64 values to bf16 (round to nearest even), as float64."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float64).numpy()


def _emulate(q, k, v, dout, o, lse, causal, scale):
    """fp64 backward with the kernel's bf16 roundings; all arrays float64."""
    s = np.einsum("bhid,bhjd->bhij", q, k)
    Nq, Nk = q.shape[2], k.shape[2]
    if causal:
        mask = np.arange(Nk)[None, :] > np.arange(Nq)[:, None] + (Nk - Nq)
        s = np.where(mask, -np.inf, s)
    p = _bf16(np.exp(scale * s - lse[..., None]))
    dp = np.einsum("bhid,bhjd->bhij", dout, v)
    D = np.sum(dout * o, axis=-1)
    ds = _bf16(p * (dp - D[..., None]))
    dv = np.einsum("bhij,bhid->bhjd", p, dout)
    dk = scale * np.einsum("bhij,bhid->bhjd", ds, q)
    dq = scale * np.einsum("bhij,bhjd->bhid", ds, k)
    return _bf16(dq), _bf16(dk), _bf16(dv)


SHAPES = [
    # B, H, Nq, Nk, d, causal
    (1, 2, 256, 256, 64, True),
    (1, 2, 300, 300, 128, True),     # ragged last tile
    (2, 2, 384, 384, 128, False),
    (1, 2, 200, 513, 128, True),     # causal chunk against a longer key sequence
    (1, 1, 77, 77, 128, True),
    (1, 3, 200, 513, 64, False),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", SHAPES,
                         ids=[f"b{B}h{H}q{Nq}k{Nk}d{d}{'c' if c else ''}"
                              for B, H, Nq, Nk, d, c in SHAPES])
def test_backward_matches_emulated_rounding(B, H, Nq, Nk, d, causal):
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed=171 + Nq + Nk + d, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(172 + Nq)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
    scale = d ** -0.5
    # the forward statistics from the oracle, in the dtypes the kernel takes
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=causal,
                              scale=scale)
    o = torch.from_numpy(ro).to(torch.bfloat16).cuda()
    lse = torch.from_numpy(rl).to(torch.float32).cuda()
    dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, dout, causal=causal, scale=scale)
    torch.cuda.synchronize()
    f64 = [t.double().cpu().numpy() for t in (q, k, v, dout, o)]
    emu = _emulate(*f64, lse.double().cpu().numpy(), causal, scale)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), emu):
        got = got.double().cpu().numpy()
        assert np.all(np.isfinite(got)), name
        rms = float(np.sqrt(np.mean(ref * ref)))
        e = np.abs(got - ref)
        excess = (e - REL * np.abs(ref)).max() / rms
        msg = f"{name}: max {e.max():.3g}, beyond 2^-7|ref| {excess:.3g} rms, rms {rms:.3g}"
        print(msg)
        assert excess <= RMS, msg
    assert binding.device_error() == 0
