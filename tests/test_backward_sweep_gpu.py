"""A seeded sweep of backward shapes against the fp64 oracle's gradients: head
counts up to past the SM count, ragged query and key tiles, fewer keys than a
tile, causal chunks with fewer queries than keys, both head sizes.  The
tolerance and its derivation are those of ``tests/test_backward_gpu.py``."""
import numpy as np
import pytest

import oracle
from attention_flashattention_fwd_gb300.inputs import bf16_bits

from .test_backward_gpu import _assert_grad_close, _run

pytestmark = pytest.mark.gpu


def _shapes(n=20, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = int(rng.choice([64, 128]))
        causal = bool(rng.integers(0, 2))
        BH = int(rng.choice([1, 2, 3, 6, 40, 153, 160]))
        Nq = int(rng.integers(1, 520))
        Nk = int(rng.integers(1, 520))
        if causal and Nq > Nk:
            Nq, Nk = Nk, Nq
        if BH * Nq * Nk > 8e6:  # keeps the fp64 gradients at a few seconds
            continue
        B = 2 if BH % 2 == 0 and BH > 1 else 1
        out.append((B, BH // B, Nq, Nk, d, causal))
    return out


SHAPES = _shapes()


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", SHAPES,
                         ids=[f"b{B}h{H}q{Nq}k{Nk}d{d}{'c' if c else ''}"
                              for B, H, Nq, Nk, d, c in SHAPES])
def test_backward_shape_sweep(B, H, Nq, Nk, d, causal):
    (q, k, v, dout), (dq, dk, dv) = _run(B, H, Nq, Nk, d, causal, seed=7000 + 3 * Nq + Nk + d)
    rq, rk, rv = oracle.attention_bwd(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(dout),
                                      causal=causal)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _assert_grad_close(got.float().cpu().numpy(), ref, f"{(B, H, Nq, Nk, d, causal)} {name}")
