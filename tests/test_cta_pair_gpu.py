"""attn_fwd_cta_pair -- the prefill with CTA-pair (cta_group::2) products
(PDC Lecture 7 §7.13) -- against the fp64 oracle, and bit for bit against
attn_fwd: the pair kernel issues the same products in the same order, each
CTA's Tensor Memory accumulating its own 128 rows, so the outputs must be
identical, not only close."""
import pytest
import torch

import oracle
from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import (EXTRA_WORKLOADS, WORKLOADS, bf16_bits,
                                                       make_qkv, make_workload)
from tests.test_parity_gpu import _assert_close

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, H, Nq, Nk, causal: one quad, partial quads, Nq < 256 (no second pair
    # tile), Nq != Nk, ragged keys, the non-causal split of the last wave
    (1, 2, 512, 512, True),
    (2, 3, 1000, 1300, True),
    (1, 2, 300, 2000, False),
    (1, 1, 77, 77, True),
    (1, 3, 200, 513, False),
    (2, 2, 129, 129, True),
    (1, 4, 1536, 1536, False),
    (3, 16, 1024, 1024, False),   # 48 quads on 76 pairs: split tail items
]


@pytest.mark.parametrize("B,H,Nq,Nk,causal", SHAPES)
def test_cta_pair_matches_oracle_and_attn_fwd(B, H, Nq, Nk, causal):
    dev = torch.device("cuda:0")
    q, k, v = make_qkv(B, H, Nq, Nk, 128, seed=31 + Nq + Nk, device=dev)
    o2, l2 = binding.attn_fwd_cta_pair(q, k, v, causal=causal)
    o1, l1 = binding.attn_fwd(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o2, o1) and torch.equal(l2, l1), "not bit-identical to attn_fwd"
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=causal)
    _assert_close(o2.float().cpu().numpy(), l2.cpu().numpy(), ro, rl, f"pair {B,H,Nq,Nk,causal}")
    assert binding.device_error() == 0


@pytest.mark.parametrize("name", ["b2h16n4096d128_causal", "b2h16n4096d128"])
def test_cta_pair_full_workload_bit_identical(name):
    """The 4096-token workloads in full: bit-identical to attn_fwd, which the
    parity tests check against the oracle."""
    w = WORKLOADS.get(name) or EXTRA_WORKLOADS[name]
    q, k, v = make_workload(w, device=torch.device("cuda:0"))
    o2, l2 = binding.attn_fwd_cta_pair(q, k, v, causal=w.causal, scale=w.scale)
    o1, l1 = binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o2, o1) and torch.equal(l2, l1)
    assert binding.device_error() == 0
