"""Seeded shape sweeps of the other entry points against the fp64 oracle:

* attn_fwd_fp8 (E4M3 operands; key counts a multiple of 16), with the FP8
  tolerance derived in ``tests/test_fp8_gpu.py``;
* attn_fwd_decode, every (b, h) row;
* attn_fwd_ragged, random per-sequence lengths in a padded batch, padding
  filled so a leak is loud (NaN queries, large keys and values) and output
  rows past each sequence's length checked untouched;
* attn_merge over a random number of uneven key shards.

Shapes and lengths come from fixed seeds, so a failure names a reproducible
case.  Forward tolerances: O max-abs 2e-2 and mean-abs 1e-3, lse 2e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import bf16_bits, make_qkv, make_qkv_fp8

from .test_fp8_gpu import _full

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 2e-3


def _close(o, lse, ro, rl, what):
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{what}: non-finite"
    e, el = np.abs(o - ro), np.abs(lse - rl)
    assert e.max() <= O_MAX and e.mean() <= O_MEAN and el.max() <= LSE_MAX, (
        f"{what}: O max {e.max():.3g} mean {e.mean():.3g} lse {el.max():.3g}")


def _fp8_shapes(n=12, seed=8):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        causal = bool(rng.integers(0, 2))
        B, H = int(rng.integers(1, 3)), int(rng.choice([1, 2, 5, 77]))
        Nk = 16 * int(rng.integers(1, 45))
        Nq = int(rng.integers(1, 700))
        if causal and Nq > Nk:
            Nq = Nk - int(rng.integers(0, Nk))
        if B * H * Nq * Nk > 1.5e7:
            continue
        out.append((B, H, Nq, Nk, causal))
    return out


FP8_SHAPES = _fp8_shapes()


@pytest.mark.parametrize("B,H,Nq,Nk,causal", FP8_SHAPES,
                         ids=[f"b{B}h{H}q{Nq}k{Nk}{'c' if c else ''}" for B, H, Nq, Nk, c in FP8_SHAPES])
def test_fp8_shape_sweep(B, H, Nq, Nk, causal):
    q8, k8, vt8, ds = make_qkv_fp8(B, H, Nq, Nk, 128, seed=8100 + Nq + 3 * Nk, device="cuda")
    _full(q8, k8, vt8, ds, causal, what=f"fp8 {(B, H, Nq, Nk, causal)}")


def _decode_shapes(n=10, seed=9):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        B, H = int(rng.integers(1, 9)), int(rng.choice([1, 3, 8, 32]))
        Nk = int(rng.choice([int(rng.integers(1, 300)), int(rng.integers(300, 12000))]))
        out.append((B, H, Nk, int(rng.choice([64, 128]))))
    return out


DECODE_SHAPES = _decode_shapes()


@pytest.mark.parametrize("B,H,Nk,d", DECODE_SHAPES,
                         ids=[f"b{B}h{H}k{Nk}d{d}" for B, H, Nk, d in DECODE_SHAPES])
def test_decode_shape_sweep(B, H, Nk, d):
    q, k, v = make_qkv(B, H, 1, Nk, d, seed=9100 + Nk + d, device="cuda")
    o, lse = binding.attn_fwd_decode(q, k, v)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v))
    _close(o, lse, ro, rl, f"decode {(B, H, Nk, d)}")


RAGGED_SEEDS = list(range(6))


@pytest.mark.parametrize("seed", RAGGED_SEEDS)
def test_ragged_prefill_sweep(seed):
    rng = np.random.default_rng(1000 + seed)
    B, H = int(rng.integers(2, 6)), int(rng.integers(1, 4))
    d = int(rng.choice([64, 128]))
    causal = bool(seed % 2)
    Nq, Nk = int(rng.integers(130, 520)), int(rng.integers(130, 520))
    if causal:
        Nq = min(Nq, Nk)
    lk = [int(rng.integers(1, Nk + 1)) for _ in range(B)]
    lq = [int(rng.integers(1, (min(Nq, n) if causal else Nq) + 1)) for n in lk]
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed=1100 + seed, device="cuda")
    for b in range(B):
        q[b, :, lq[b]:] = float("nan")
        k[b, :, lk[b]:] = 3.0e4
        v[b, :, lk[b]:] = 3.0e4
    sq = torch.tensor(lq, dtype=torch.int32, device="cuda")
    sk = torch.tensor(lk, dtype=torch.int32, device="cuda")
    o = torch.full_like(q, 3.0)
    lse = torch.full((B, H, Nq), 7.0, dtype=torch.float32, device="cuda")
    binding.attn_fwd_ragged(q, k, v, sq, sk, causal=causal, out=o, lse=lse)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    for b in range(B):
        qs = q[b:b + 1, :, :lq[b]].contiguous()
        ks = k[b:b + 1, :, :lk[b]].contiguous()
        vs = v[b:b + 1, :, :lk[b]].contiguous()
        ro, rl = oracle.attention(bf16_bits(qs), bf16_bits(ks), bf16_bits(vs), causal=causal)
        _close(o[b:b + 1, :, :lq[b]], lse[b:b + 1, :, :lq[b]], ro, rl,
               f"ragged seed {seed} seq {b} (lq {lq[b]}, lk {lk[b]})")
        assert (o[b, :, lq[b]:] == 3.0).all() and (lse[b, :, lq[b]:] == 7.0).all()


MERGE_SEEDS = list(range(6))


@pytest.mark.parametrize("seed", MERGE_SEEDS)
def test_merge_sweep(seed):
    rng = np.random.default_rng(2000 + seed)
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 5))
    d = int(rng.choice([64, 128]))
    Nq = int(rng.choice([1, int(rng.integers(2, 400))]))
    parts = int(rng.integers(1, 8))
    split = [int(rng.integers(1, 400)) for _ in range(parts)]
    Nk = sum(split)
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed=2100 + seed, device="cuda")
    # each shard's outputs in their own (aligned) buffers, then stacked: a
    # slice of one [S, B, H, Nq] lse tensor need not start on 16 bytes
    outs = []
    k0 = 0
    for n in split:
        ks = k[:, :, k0:k0 + n].contiguous()
        vs = v[:, :, k0:k0 + n].contiguous()
        outs.append(binding.attn_fwd(q, ks, vs))
        k0 += n
    o_parts = torch.stack([o for o, _ in outs])
    lse_parts = torch.stack([lp for _, lp in outs])
    o, lse = binding.attn_merge(o_parts, lse_parts)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v))
    _close(o, lse, ro, rl, f"merge seed {seed} split {split}")
