"""The CTA-pair product (PDC Lecture 7 §7.13, CTA pair / MMA.2SM) on the GPU:
one thread of the even CTA of a two-CTA cluster issues tcgen05.mma.cta_group::2
with M = 256, each CTA holding 128 rows of A and half of B's rows in its shared
memory and receiving its 128 rows of D in its Tensor Memory.  The product is
checked against a host matrix product, and the issue-rate measurement of both
forms against what the tensor core can do at most."""
import pytest
import torch

from attention_flashattention_fwd_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", [0, 1])
def test_pair_product_matches_host_matmul(seed):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(256, 64, generator=g).to(torch.bfloat16)
    b = torch.randn(128, 64, generator=g).to(torch.bfloat16)
    d = binding.attn_pair_product(a.cuda(), b.cuda()).cpu().double()
    ref = a.double() @ b.double().T            # bf16 inputs are exact in fp64
    # fp32 accumulation of 64 exact products: |error| <= 64 u sum |a_k b_k|
    bound = 64 * 2.0 ** -24 * (a.double().abs() @ b.double().abs().T) + 1e-30
    assert torch.isfinite(d).all()
    assert ((d - ref).abs() <= bound).all(), (d - ref).abs().max().item()
    assert binding.device_error() == 0


def test_pair_product_rows_and_columns_land_where_stated():
    """A one-hot A and a B of distinct row tags: D[i, j] = B[j, i % 64] picks
    out every row of A from the CTA that holds it and every row of B from the
    CTA that holds it."""
    a = torch.zeros(256, 64)
    a[torch.arange(256), torch.arange(256) % 64] = 1.0
    # B[j, k] = (1 + j/128) 2^(k - 32): 8192 distinct values, each exact in bf16
    b = (1.0 + torch.arange(128).view(128, 1) / 128.0) * torch.pow(
        2.0, torch.arange(64).view(1, 64) - 32.0)
    a, b = a.to(torch.bfloat16), b.to(torch.bfloat16)
    assert b.float().unique().numel() == 128 * 64
    d = binding.attn_pair_product(a.cuda(), b.cuda()).cpu()
    ref = (a.float() @ b.float().T)
    assert torch.equal(d, ref)
    assert binding.device_error() == 0


@pytest.mark.parametrize("form", [1, 2])
@pytest.mark.parametrize("issuer", [0, 1])
@pytest.mark.parametrize("busy,waits", [(0, 0), (1, 1)])
def test_mma_rate_is_bounded_by_the_tensor_core(form, issuer, busy, waits):
    """Each product keeps every SM's tensor core busy for 64 cycles, so an
    issuer cannot finish `steps` groups of 8 in fewer than steps x 8 x 64
    cycles; far more than that would mean a hung pipeline."""
    steps = 512
    r = binding.bench_mma_rate(form, issuer=issuer, busy=busy, waits=waits, steps=steps, reps=2)
    floor = steps * 8 * 64
    assert r["sms"] >= 2 and r["sms"] % 2 == 0
    assert 0.95 * floor <= r["cycles"] <= 20 * floor, r
    assert r["ms"] > 0
    assert binding.device_error() == 0
