"""A seeded sweep of prefill shapes against the fp64 oracle: many head counts,
query and key lengths (ragged tiles, fewer keys than a tile, causal with fewer
queries than keys) and both head sizes, every row checked.  Head counts reach
past the SM count so that some non-causal launches run their last wave as
single query tiles."""
import numpy as np
import pytest
import torch

import oracle
from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import bf16_bits, make_qkv

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 2e-3


def _shapes(n=36, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = int(rng.choice([64, 128]))
        causal = bool(rng.integers(0, 2))
        BH = int(rng.choice([1, 2, 3, 7, 40, 77, 79, 150, 153, 160]))
        Nq = int(rng.integers(1, 700))
        Nk = int(rng.integers(1, 700))
        if causal and Nq > Nk:
            Nq, Nk = Nk, Nq
        if BH * Nq * Nk > 2.5e7:  # keeps the oracle at a fraction of a second
            continue
        B = 1 if BH in (1, 7, 77, 79, 153) else 2 if BH % 2 == 0 else 3
        H = BH // B
        if B * H != BH:
            B, H = 1, BH
        out.append((B, H, Nq, Nk, d, causal))
    return out


SHAPES = _shapes()


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", SHAPES,
                         ids=[f"b{B}h{H}q{Nq}k{Nk}d{d}{'c' if c else ''}"
                              for B, H, Nq, Nk, d, c in SHAPES])
def test_prefill_shape_sweep(B, H, Nq, Nk, d, causal):
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed=5000 + Nq * 7 + Nk + d, device="cuda:0")
    o, lse = binding.attn_fwd(q, k, v, causal=causal)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=causal)
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    e, el = np.abs(o - ro), np.abs(lse - rl)
    assert e.max() <= O_MAX and e.mean() <= O_MEAN and el.max() <= LSE_MAX, (
        f"O max {e.max():.3g} mean {e.mean():.3g}, lse max {el.max():.3g}")
