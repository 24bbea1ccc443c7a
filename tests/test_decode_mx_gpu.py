"""attn_fwd_decode_mx (MXFP8 keys and values: E4M3 codes, one E8M0 scale per
32 consecutive elements of a row) against the fp64 oracle, which decodes the
codes by the OCP MX definition and runs the naive attention on them.

Tolerance: the kernel widens every code exactly and scales by exact powers of
two, so it computes the attention of the same dequantised keys and values as
the oracle, in fp32 with a bf16 output: the bf16 study tolerances apply (O
within 2e-2 max-abs and 1e-3 mean-abs, lse within 2e-3).
"""
import numpy as np
import pytest
import torch

import oracle
from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import (WORKLOADS, bf16_bits, make_qkv_mx,
                                                       make_workload_mx)

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 2e-3

pytestmark = pytest.mark.gpu


def _check(o, lse, ro, rl, what):
    o = np.asarray(o, np.float64)
    lse = np.asarray(lse, np.float64)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{what}: non-finite output"
    e, el = np.abs(o - ro), np.abs(lse - rl)
    msg = f"{what}: O max {e.max():.3g} mean {e.mean():.3g}, lse max {el.max():.3g}"
    assert e.max() <= O_MAX and e.mean() <= O_MEAN and el.max() <= LSE_MAX, msg


def _np(t):
    return t.cpu().numpy()


SHAPES = [
    # B, H, Nk, d
    (1, 1, 1, 64),
    (1, 1, 37, 128),
    (1, 1, 511, 128),
    (1, 1, 513, 64),
    (2, 3, 3000, 64),
    (2, 4, 8192, 128),    # 16 splits per head
    (1, 1, 20000, 128),
    (16, 32, 1024, 128),  # one split per head on a 152-SM GPU
]


@pytest.mark.parametrize("B,H,Nk,d", SHAPES, ids=[f"b{B}h{H}k{Nk}d{d}" for B, H, Nk, d in SHAPES])
def test_decode_mx_matches_oracle(B, H, Nk, d):
    q, k8, ks, v8, vs = make_qkv_mx(B, H, Nk, d, seed=61 + Nk + d, device="cuda")
    o, lse = binding.attn_fwd_decode_mx(q, k8, ks, v8, vs)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_mx(bf16_bits(q), _np(k8), _np(ks), _np(v8), _np(vs))
    _check(_np(o.float()), _np(lse), ro, rl, f"decode mx {(B, H, Nk, d)}")


def test_decode_mx_wide_scales_and_extreme_codes():
    """Scales over a wide range (2^-20 .. 2^10 per block), the largest E4M3
    codes (+-448) and zeros in the same rows."""
    B, H, Nk, d = 2, 2, 700, 128
    q, k8, ks, v8, vs = make_qkv_mx(B, H, Nk, d, seed=62, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(63)
    ks = torch.randint(107, 122, ks.shape, generator=g, device="cuda").to(torch.uint8)
    vs = torch.randint(117, 137, vs.shape, generator=g, device="cuda").to(torch.uint8)
    k8 = k8.clone()
    v8 = v8.clone()
    k8[:, :, ::7, :5] = 0x7E   # +448
    k8[:, :, 3::11, 9:20] = 0xFE  # -448
    v8[:, :, ::5, 40:48] = 0x00  # zeros
    v8[:, :, 1::9, 100:] = 0x7E
    o, lse = binding.attn_fwd_decode_mx(q, k8, ks, v8, vs, scale=0.05)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_mx(bf16_bits(q), _np(k8), _np(ks), _np(v8), _np(vs), scale=0.05)
    # values up to 448 * 2^10: compare relative to the output's scale
    s = max(1.0, float(np.abs(ro).max()))
    _check(_np(o.float()) / s, _np(lse), ro / s, rl, "wide scales")


def test_decode_mx_workload_sampled_heads():
    """The decode workload's shape (B=64, H=32, Nk=8192, d=128) with MXFP8 K and
    V; 128 sampled heads against the oracle."""
    w = WORKLOADS["decode_b64h32nk8192d128"]
    q, k8, ks, v8, vs = make_workload_mx(w, device="cuda")
    o, lse = binding.attn_fwd_decode_mx(q, k8, ks, v8, vs, scale=w.scale)
    torch.cuda.synchronize()
    BH = w.B * w.H
    sel = np.sort(np.random.default_rng(64).choice(BH, 128, replace=False))
    sel[0], sel[-1] = 0, BH - 1
    idx = torch.as_tensor(sel, device="cuda")

    def pick(t, n):
        return t.reshape(BH, n, -1).index_select(0, idx).reshape(1, len(sel), n, -1)

    ro, rl = oracle.attention_mx(bf16_bits(pick(q, 1)), _np(pick(k8, w.Nk)), _np(pick(ks, w.Nk)),
                                 _np(pick(v8, w.Nk)), _np(pick(vs, w.Nk)), scale=w.scale)
    og = o.reshape(BH, w.d).index_select(0, idx).float().cpu().numpy().reshape(ro.shape)
    lg = lse.reshape(BH).index_select(0, idx).cpu().numpy().reshape(rl.shape)
    _check(og, lg, ro, rl, w.name + " (MXFP8 K, V)")
    assert binding.device_error() == 0


def test_decode_mx_accepts_torch_float8_dtypes():
    B, H, Nk, d = 1, 2, 600, 64
    q, k8, ks, v8, vs = make_qkv_mx(B, H, Nk, d, seed=65, device="cuda")
    o1, l1 = binding.attn_fwd_decode_mx(q, k8, ks, v8, vs)
    o2, l2 = binding.attn_fwd_decode_mx(q, k8.view(torch.float8_e4m3fn),
                                        ks.view(torch.float8_e8m0fnu),
                                        v8.view(torch.float8_e4m3fn), vs.view(torch.float8_e8m0fnu))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
