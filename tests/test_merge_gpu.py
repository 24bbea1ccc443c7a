"""attn_merge (the exchange step of key-sharded attention) against the fp64
oracle: the keys of each head are split into uneven shards, each shard goes
through the prefill or decode kernel, and the merged result must match
attention over all keys within the forward's tolerances."""
import numpy as np
import pytest
import torch

import oracle
from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import bf16_bits, make_qkv

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 2e-3


def _check(o, lse, ro, rl, what):
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    e, el = np.abs(o - ro), np.abs(lse - rl)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    assert e.max() <= O_MAX and e.mean() <= O_MEAN and el.max() <= LSE_MAX, (
        f"{what}: O max {e.max():.3g} mean {e.mean():.3g} lse {el.max():.3g}")


@pytest.mark.parametrize("B,H,Nq,split,d", [
    (1, 2, 300, (128, 300, 77), 128),
    (2, 3, 1, (700, 1000, 300, 48), 128),     # decode-shaped shards
    (1, 4, 256, (512, 512), 64),
    (1, 1, 77, (5,), 64),                     # one part: the identity
    (1, 2, 190, (200, 100, 300, 50, 129, 77), 128),  # more than 4 parts: batched online form
    (2, 1, 64, (64, 64, 64, 64, 64), 64),
])
def test_sharded_attention_merges_to_full(B, H, Nq, split, d):
    Nk = sum(split)
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed=61 + Nk, device="cuda")
    o_parts, lse_parts = [], []
    k0 = 0
    for n in split:
        ks, vs = k[:, :, k0:k0 + n].contiguous(), v[:, :, k0:k0 + n].contiguous()
        o_s, l_s = binding.attention(q, ks, vs)
        o_parts.append(o_s)
        lse_parts.append(l_s)
        k0 += n
    o, lse = binding.attn_merge(torch.stack(o_parts), torch.stack(lse_parts))
    torch.cuda.synchronize()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v))
    _check(o, lse, ro, rl, f"{(B, H, Nq, split, d)}")


def test_empty_parts_have_no_weight():
    q, k, v = make_qkv(1, 2, 128, 256, 128, seed=67, device="cuda")
    o1, l1 = binding.attn_fwd(q, k, v)
    junk = torch.full_like(o1, 7.0)
    ninf = torch.full_like(l1, float("-inf"))
    o, lse = binding.attn_merge(torch.stack([junk, o1, junk]), torch.stack([ninf, l1, ninf]))
    torch.cuda.synchronize()
    assert torch.equal(lse, l1)
    assert (o.float() - o1.float()).abs().max().item() <= 2 ** -8 * o1.float().abs().max().item()
    # more than 4 parts (the batched form): empty parts before and after the live one
    o, lse = binding.attn_merge(torch.stack([junk, junk, junk, junk, o1, junk]),
                                torch.stack([ninf, ninf, ninf, ninf, l1, ninf]))
    torch.cuda.synchronize()
    assert torch.equal(lse, l1)
    assert (o.float() - o1.float()).abs().max().item() <= 2 ** -8 * o1.float().abs().max().item()
    # every part empty: o = 0, lse = -inf (both forms)
    for n in (2, 5):
        o, lse = binding.attn_merge(torch.stack([junk] * n), torch.stack([ninf] * n))
        torch.cuda.synchronize()
        assert (o.float() == 0).all() and torch.isinf(lse).all() and (lse < 0).all()


def test_merge_of_the_bench_shards_closed_form():
    """The bench's merge call at full size (four shards of the B2 H16 N4096 d128
    shape, every o_s the same o and lse_s = lse - s): the merged row is the same
    convex combination of identical rows, o, and the merged logsumexp is
    lse + ln(1 + e^-1 + e^-2 + e^-3)."""
    from attention_flashattention_fwd_gb300.inputs import WORKLOADS, make_workload
    w = WORKLOADS["b2h16n4096d128_causal"]
    q, k, v = make_workload(w, device="cuda")
    o, lse = binding.attn_fwd(q, k, v, causal=True, scale=w.scale)
    o_parts = torch.stack([o] * 4).contiguous()
    l_parts = torch.stack([lse - float(s) for s in range(4)]).contiguous()
    om, lm = binding.attn_merge(o_parts, l_parts)
    torch.cuda.synchronize()
    shift = float(np.log(sum(np.exp(-s) for s in range(4))))
    eo = (om.float() - o.float()).abs().max().item()
    el = (lm - (lse + shift)).abs().max().item()
    assert eo <= 2.0 ** -8 * o.float().abs().max().item() and el <= 1e-5, (eo, el)
    assert binding.device_error() == 0


def test_merge_full_size_key_shards():
    """Four key shards of the non-causal B2 H16 N4096 d128 workload (1024 keys
    each), attended one by one and merged: against the fp64 oracle on sampled
    rows, and every row against one call over all keys."""
    from attention_flashattention_fwd_gb300.inputs import EXTRA_WORKLOADS, make_workload
    w = EXTRA_WORKLOADS["b2h16n4096d128"]
    q, k, v = make_workload(w, device="cuda")
    parts = [binding.attn_fwd(q, k[:, :, a:a + 1024].contiguous(), v[:, :, a:a + 1024].contiguous(),
                              scale=w.scale) for a in range(0, 4096, 1024)]
    om, lm = binding.attn_merge(torch.stack([p[0] for p in parts]),
                                torch.stack([p[1] for p in parts]))
    of, lf = binding.attn_fwd(q, k, v, scale=w.scale)
    torch.cuda.synchronize()
    assert (om.float() - of.float()).abs().max().item() <= 2e-2
    assert (lm - lf).abs().max().item() <= 2e-3
    rng = np.random.default_rng(5)
    BH = w.B * w.H
    rows = np.array([(int(rng.integers(BH)), int(rng.integers(w.Nq))) for _ in range(128)],
                    dtype=np.int64)
    ro, rl = oracle.attention_rows(bf16_bits(q), bf16_bits(k), bf16_bits(v), rows, causal=False,
                                   scale=w.scale)
    idx = torch.as_tensor(rows[:, 0] * w.Nq + rows[:, 1], device=om.device)
    og = om.reshape(BH * w.Nq, w.d).index_select(0, idx)
    lg = lm.reshape(BH * w.Nq).index_select(0, idx)
    _check(og, lg, ro, rl, "4 key shards of b2h16n4096d128")
    assert binding.device_error() == 0
