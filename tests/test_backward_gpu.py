"""The CUDA backward (attn_bwd) against the fp64 oracle's gradients, through
the C ABI.

The forward's own outputs (o, lse from attn_fwd) feed the backward, as a
training step would use them; dO is a seeded standard-normal bf16 tensor.
The oracle differentiates exact attention of the same bf16 inputs.

Tolerance (derived from the arithmetic; the pages give none for gradients).
Three sources of error:
  * output rounding: dQ, dK and dV are rounded to bf16, relative error
    <= 2^-9 of the element itself.  Gradients are heavy-tailed (under a causal
    mask query 0 sees only key 0, so dV_0 = dO_0 is many times the typical
    element), so this part is bounded per element: 2^-8 |ref|;
  * accumulation: P and dS are rounded to bf16 (relative <= 2^-9) before the
    dV, dK and dQ products, which sum many such terms with independent signs;
  * cancellation in dP_ij - D_i: D_i = rowsum(dO_i * O_i) comes from the bf16
    forward output, so it carries an error of about 2^-9 |dO_i| |O_i|, while
    for a sharp softmax (one dominant key) dP_ij - D_i is a small difference
    of two such quantities.  The notes' D formula has this property whatever
    the kernel does with it.
The last two are bounded on the tensor's scale rms(ref): whatever the output
rounding does not explain stays below 2^-3 rms(ref) on every element
(measured: at most 0.06 rms(ref) over the cases here, the sharp-softmax case
included) and the mean error below 2^-7 rms(ref) (measured: <= 0.0023).  A
dropped term, a wrong sign, a transposed operand or a mask shifted by one key
produces errors of the order of rms(ref) itself.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import WORKLOADS, bf16_bits, make_qkv, make_workload

pytestmark = pytest.mark.gpu

ELEM_REL, MAX_RMS, MEAN_RMS = 2.0 ** -8, 2.0 ** -3, 2.0 ** -7


def _dev():
    return torch.device("cuda:0")


def _dout(shape, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)


def _assert_grad_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite"
    rms = float(np.sqrt(np.mean(ref * ref)))
    e = np.abs(got - ref)
    excess = e - ELEM_REL * np.abs(ref)  # what the output rounding does not explain
    msg = (f"{what}: max {e.max():.3g} (beyond rounding {excess.max():.3g}) "
           f"mean {e.mean():.3g} rms(ref) {rms:.3g}")
    print(msg)
    assert excess.max() <= MAX_RMS * rms and e.mean() <= MEAN_RMS * rms, msg
    return excess.max() / rms, e.mean() / rms


def _run(B, H, Nq, Nk, d, causal, seed, scale=None):
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed=seed, device=_dev())
    dout = _dout((B, H, Nq, d), seed + 1)
    o, lse = binding.attn_fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, dout, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return (q, k, v, dout), (dq, dk, dv)


BWD_SHAPES = [
    # B, H, Nq, Nk, d, causal
    (1, 1, 128, 128, 64, False),
    (1, 2, 256, 256, 128, False),
    (2, 2, 384, 384, 128, True),
    (1, 2, 300, 300, 64, True),      # ragged last tile
    (1, 1, 77, 77, 128, True),       # less than one tile
    (1, 3, 200, 513, 128, False),    # Nq != Nk, ragged keys
    (1, 2, 200, 513, 128, True),     # causal chunk: queries are the newest 200 tokens
    (1, 1, 1000, 1000, 128, True),
    (2, 1, 640, 640, 64, True),
    (1, 1, 5, 3, 64, False),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", BWD_SHAPES,
                         ids=[f"b{B}h{H}q{Nq}k{Nk}d{d}{'c' if c else ''}"
                              for B, H, Nq, Nk, d, c in BWD_SHAPES])
def test_backward_matches_oracle(B, H, Nq, Nk, d, causal):
    (q, k, v, dout), (dq, dk, dv) = _run(B, H, Nq, Nk, d, causal, seed=101 + Nq + Nk + d)
    rq, rk, rv = oracle.attention_bwd(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(dout),
                                      causal=causal)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _assert_grad_close(got.float().cpu().numpy(), ref, f"{(B, H, Nq, Nk, d, causal)} {name}")


def test_backward_scale_argument():
    (q, k, v, dout), (dq, dk, dv) = _run(1, 2, 256, 256, 128, True, seed=131, scale=0.3)
    rq, rk, rv = oracle.attention_bwd(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(dout),
                                      causal=True, scale=0.3)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _assert_grad_close(got.float().cpu().numpy(), ref, f"scale=0.3 {name}")


def test_backward_headline_shape_sampled():
    """The 2 x 16 x 4096 x 4096 causal workload at d = 128: dQ on sampled
    rows, dK and dV on sampled keys of two heads (the oracle recomputes every
    row's statistics of those heads)."""
    w = WORKLOADS["b2h16n4096d128_causal"]
    q, k, v = make_workload(w, device=_dev())
    dout = _dout(q.shape, 2024)
    o, lse = binding.attn_fwd(q, k, v, causal=True, scale=w.scale)
    dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, dout, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    BH = w.B * w.H
    rng = np.random.default_rng(77)
    rows = np.array([(int(rng.integers(BH)), i) for i in
                     [0, 1, 127, 128, 4095] + list(rng.integers(0, w.Nq, 120))], dtype=np.int64)
    keys = np.array([(bh, j) for bh in (0, BH - 1) for j in
                     [0, 127, 128, 4095] + list(rng.integers(0, w.Nk, 28))], dtype=np.int64)
    bits = [bf16_bits(t) for t in (q, k, v, dout)]
    rq, _ = oracle.attention_bwd_dq_rows(*bits, rows, causal=True, scale=w.scale)
    rk, rv = oracle.attention_bwd_dkdv_keys(*bits, keys, causal=True, scale=w.scale)
    gq = dq.reshape(BH, w.Nq, w.d)[rows[:, 0], rows[:, 1]].float().cpu().numpy()
    gk = dk.reshape(BH, w.Nk, w.d)[keys[:, 0], keys[:, 1]].float().cpu().numpy()
    gv = dv.reshape(BH, w.Nk, w.d)[keys[:, 0], keys[:, 1]].float().cpu().numpy()
    _assert_grad_close(gq, rq, "headline dq rows")
    _assert_grad_close(gk, rk, "headline dk keys")
    _assert_grad_close(gv, rv, "headline dv keys")


def test_backward_sum_rules_on_gpu():
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i per head (softmax rows sum
    to one), checked on the kernel's own output at a size no oracle runs."""
    (q, k, v, dout), (dq, dk, dv) = _run(1, 4, 2048, 2048, 128, True, seed=141)
    sk = dk.float().sum(dim=2)
    sv = dv.float().sum(dim=2) - dout.float().sum(dim=2)
    scale_k = dk.float().abs().sum(dim=2)
    scale_v = dv.float().abs().sum(dim=2)
    assert (sk.abs() <= 2e-2 * scale_k + 1e-3).all()
    assert (sv.abs() <= 2e-2 * scale_v + 1e-3).all()
    assert binding.device_error() == 0


def test_backward_rejects_small_workspace():
    q, k, v = make_qkv(1, 1, 128, 128, 64, seed=5, device=_dev())
    o, lse = binding.attn_fwd(q, k, v)
    ws = torch.empty(binding.bwd_workspace_bytes(1, 1, 128, 128, 64) - 16, dtype=torch.uint8,
                     device="cuda")
    with pytest.raises(binding.GbattnError):
        binding.attn_bwd(q, k, v, o, lse, o, workspace=ws)


def test_backward_d64_2048_tokens_full():
    (q, k, v, dout), (dq, dk, dv) = _run(1, 2, 2048, 2048, 64, True, seed=151)
    rq, rk, rv = oracle.attention_bwd(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(dout),
                                      causal=True)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _assert_grad_close(got.float().cpu().numpy(), ref, f"d64 2048 {name}")
