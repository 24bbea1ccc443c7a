"""Ragged batches (sequences of different lengths in one padded batch):
attn_fwd_ragged and attn_fwd_decode_ragged against the fp64 oracle run on
each sequence's own rows.  Padding is filled so that any leak is loud: large
finite keys and values past seqlens_k (the prefill kernel reads them in
whole tiles and must give them weight 0), NaN queries past seqlens_q (rows
are independent) and NaN keys and values past seqlens_k in decode (never
read there).  Output rows past seqlens_q must be left untouched."""
import numpy as np
import pytest
import torch

import oracle
from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import bf16_bits, make_qkv

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 2e-3


def _close(o, lse, ro, rl, what):
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{what}: non-finite"
    e, el = np.abs(o - ro), np.abs(lse - rl)
    assert e.max() <= O_MAX and e.mean() <= O_MEAN and el.max() <= LSE_MAX, (
        f"{what}: O max {e.max():.3g} mean {e.mean():.3g} lse {el.max():.3g}")


def _pad(t, lens, value):
    for b, n in enumerate(lens):
        t[b, :, n:] = value


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_prefill_matches_oracle_per_sequence(causal, d):
    B, H, N = 3, 2, 600
    lq = [600, 130, 257]
    lk = [600, 300, 257]
    q, k, v = make_qkv(B, H, N, N, d, seed=81 + d, device="cuda")
    _pad(q, lq, float("nan"))
    _pad(k, lk, 3.0e4)
    _pad(v, lk, 3.0e4)
    sq = torch.tensor(lq, dtype=torch.int32, device="cuda")
    sk = torch.tensor(lk, dtype=torch.int32, device="cuda")
    o = torch.full_like(q, 3.0)
    lse = torch.full((B, H, N), 7.0, dtype=torch.float32, device="cuda")
    binding.attn_fwd_ragged(q, k, v, sq, sk, causal=causal, out=o, lse=lse)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    for b in range(B):
        qs, ks, vs = (t[b:b + 1, :, :n] for t, n in ((q, lq[b]), (k, lk[b]), (v, lk[b])))
        ro, rl = oracle.attention(bf16_bits(qs.contiguous()), bf16_bits(ks.contiguous()),
                                  bf16_bits(vs.contiguous()), causal=causal)
        _close(o[b:b + 1, :, :lq[b]], lse[b:b + 1, :, :lq[b]], ro, rl, f"seq {b}")
        assert (o[b, :, lq[b]:] == 3.0).all() and (lse[b, :, lq[b]:] == 7.0).all()


def test_ragged_without_lengths_is_attn_fwd():
    q, k, v = make_qkv(2, 2, 300, 300, 128, seed=85, device="cuda")
    a = binding.attn_fwd(q, k, v, causal=True)
    b = binding.attn_fwd_ragged(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_ragged_decode_matches_oracle_per_sequence():
    B, H, Nk, d = 4, 8, 5000, 128
    lk = [5000, 1, 777, 4096]
    q, k, v = make_qkv(B, H, 1, Nk, d, seed=87, device="cuda")
    _pad(k, lk, float("nan"))
    _pad(v, lk, float("nan"))
    sk = torch.tensor(lk, dtype=torch.int32, device="cuda")
    o, lse = binding.attn_fwd_decode_ragged(q, k, v, sk)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    for b in range(B):
        ro, rl = oracle.attention(bf16_bits(q[b:b + 1].contiguous()),
                                  bf16_bits(k[b:b + 1, :, :lk[b]].contiguous()),
                                  bf16_bits(v[b:b + 1, :, :lk[b]].contiguous()))
        _close(o[b:b + 1], lse[b:b + 1], ro, rl, f"decode seq {b}")


def test_out_of_range_lengths_are_reported_and_skipped():
    B, H, N, d = 3, 2, 256, 64
    q, k, v = make_qkv(B, H, N, N, d, seed=89, device="cuda")
    lq = [256, 0, 200]            # sequence 1 has no queries: out of range
    lk = [256, 100, 512]          # sequence 2 claims more keys than the tensor holds
    sq = torch.tensor(lq, dtype=torch.int32, device="cuda")
    sk = torch.tensor(lk, dtype=torch.int32, device="cuda")
    o = torch.full_like(q, 3.0)
    lse = torch.full((B, H, N), 7.0, dtype=torch.float32, device="cuda")
    binding.attn_fwd_ragged(q, k, v, sq, sk, out=o, lse=lse)
    torch.cuda.synchronize()
    assert binding.device_error() == 1  # ATTN_ERR_INVALID_ARG
    assert (o[1:] == 3.0).all() and (lse[1:] == 7.0).all()  # skipped sequences untouched
    ro, rl = oracle.attention(bf16_bits(q[:1]), bf16_bits(k[:1]), bf16_bits(v[:1]))
    _close(o[:1], lse[:1], ro, rl, "valid sequence")
    # decode: the out-of-range sequence gets o = 0, lse = -inf
    qd = q[:, :, :1].contiguous()
    od, ld = binding.attn_fwd_decode_ragged(qd, k, v, torch.tensor([256, 0, 9999], dtype=torch.int32,
                                                                     device="cuda"))
    torch.cuda.synchronize()
    assert binding.device_error() == 1
    assert (od[1:].float() == 0).all() and torch.isinf(ld[1:]).all()
    assert binding.device_error() == 0  # the word was cleared
