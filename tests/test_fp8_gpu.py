"""The FP8 (E4M3) forward against the fp64 oracle on the same E4M3 operands.

Both sides read the same E4M3 codes and descales, so the operands are exact
and what differs is the kernel's arithmetic:
  (1) P rounded to E4M3 before the P V product.  The kernel's p are relative
      to a reference maximum m_ref at or below the row's true maximum m
      (p_kernel = p_true 2^(m - m_ref) >= p_true, l_kernel >= l_true >= 1).
      Round to nearest moves a normal p (>= 2^-6) by at most 2^-4 of itself
      and a smaller one by at most 2^-10 (p below 2^-10 flushes to 0);
  (2) fp32 scores and accumulators (exact E4M3 products);
  (3) the bf16 output, half an ulp = 2^-9 of |O|.
The row sum l is taken from the unrounded p, so per element
    |O_kernel - O| <= 2^-4 A + 2^-9 |O| + r,
A = softmax(S) |V| (the oracle's attention of the same scores on |V|) and r
the sum over the keys below 2^-6 in the kernel's frame -- a subset of J, the
keys with p_true < 2^-6 -- of roundings of at most 2^-10 |v_j| / l_true each,
independent, signed by v_j.  The tests bound r by six standard deviations of
that sum, 6 * 2^-10 sqrt(sum_{j in J} v_j^2) / l_true, with the scores, J and
l_true computed here in fp64 from the dequantised operands, plus 2^-14 max|V|
for fp32 rounding.  The mean error is held to 2^-6 of the mean of A.  lse uses
the unrounded row sum: the bf16 path's 2e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import WORKLOADS, make_qkv_fp8, make_workload_fp8

LSE_MAX = 2e-3

pytestmark = pytest.mark.gpu


def _dev():
    return torch.device("cuda:0")


def _np(t):
    return t.cpu().numpy()


def _small_p_term(q, k, v, rows, causal, scale):
    """6 * 2^-10 sqrt(sum_{j in J} v_j^2) / l_true + 2^-14 max|V| for each listed
    row ([n, 2] of (bh, i)) of float64 operands q [BH,Nq,d], k, v [BH,Nk,d]."""
    Nq, Nk = q.shape[1], k.shape[1]
    out = np.empty((len(rows), v.shape[2]))
    for t, (bh, i) in enumerate(rows):
        sc = scale * (k[bh] @ q[bh, i])
        if causal:
            sc[i + (Nk - Nq) + 1:] = -np.inf
        p = np.exp(sc - sc.max())
        small = p < 2.0 ** -6
        out[t] = 6 * 2.0 ** -10 * np.sqrt((v[bh][small] ** 2).sum(axis=0)) / p.sum()
    return out + 2.0 ** -14 * np.abs(v).max()


def _check(o, lse, ro, rl, ra, rr, what):
    """o, lse: the kernel's; ro, rl: the oracle's; ra: the oracle's A; rr: the
    small-p term (all of o's shape)."""
    o = np.asarray(o, np.float64)
    lse = np.asarray(lse, np.float64)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{what}: non-finite output"
    e = np.abs(o - ro)
    tol = 2.0 ** -4 * ra + 2.0 ** -9 * np.abs(ro) + rr
    el = np.abs(lse - rl)
    ratio = (e / tol).max()
    msg = (f"{what}: O max {e.max():.3g} (max err/tol {ratio:.3g}) mean {e.mean():.3g} "
           f"(A mean {ra.mean():.3g}), lse max {el.max():.3g}")
    assert ratio <= 1.0 and e.mean() <= 2.0 ** -6 * ra.mean() + 1e-4 and el.max() <= LSE_MAX, msg
    return e.max(), e.mean(), el.max()


def _abs_codes(c):
    """E4M3 codes of |x|: the sign bit cleared."""
    return np.bitwise_and(c, np.uint8(0x7F))


def _full(q8, k8, vt8, ds, causal, scale=None, what=""):
    o, lse = binding.attn_fwd_fp8(q8, k8, vt8, *ds, causal=causal, scale=scale)
    torch.cuda.synchronize()
    a = dict(causal=causal, scale=scale, descale_q=ds[0], descale_k=ds[1], descale_v=ds[2])
    qn, kn, vn = _np(q8), _np(k8), _np(vt8)
    ro, rl = oracle.attention_fp8(qn, kn, vn, **a)
    ra, _ = oracle.attention_fp8(qn, kn, _abs_codes(vn), **a)
    B, H, Nq, d = qn.shape
    qd, kd, vd = (x.reshape(B * H, -1, d) for x in oracle.fp8_operands(qn, kn, vn, *ds))
    rows = np.array([(bh, i) for bh in range(B * H) for i in range(Nq)])
    rr = _small_p_term(qd, kd, vd, rows, causal, scale if scale is not None else d ** -0.5)
    return _check(_np(o.float()), _np(lse), ro, rl, ra, rr.reshape(ro.shape), what)


SHAPES = [
    # B, H, Nq, Nk, causal  (d = 128; Nk a multiple of 16)
    (1, 1, 128, 128, False),
    (1, 2, 256, 256, True),
    (2, 2, 384, 384, True),
    (1, 2, 300, 304, False),     # ragged query and key tiles
    (1, 1, 80, 80, True),        # less than one tile
    (1, 3, 200, 512, False),     # Nq != Nk
    (1, 2, 200, 528, True),      # causal chunk: the newest 200 of 528 tokens
    (1, 1, 1, 16, False),        # one query, the fewest keys
    (1, 1, 5, 16, True),
    (1, 1, 1008, 1008, True),    # many tiles, ragged, causal
    (1, 1, 1, 704, True),        # one causal query row sees every key
    (1, 77, 512, 512, False),    # 154 pairs on 152 SMs: the last wave as single tiles
    (1, 79, 300, 384, False),    # 158 pairs: 12 single tiles
    (2, 1, 640, 1280, False),
]


@pytest.mark.parametrize("B,H,Nq,Nk,causal", SHAPES,
                         ids=[f"b{B}h{H}q{Nq}k{Nk}{'c' if c else ''}" for B, H, Nq, Nk, c in SHAPES])
def test_fp8_matches_oracle(B, H, Nq, Nk, causal):
    q8, k8, vt8, ds = make_qkv_fp8(B, H, Nq, Nk, 128, seed=31 + Nq + Nk, device=_dev())
    _full(q8, k8, vt8, ds, causal, what=f"{(B, H, Nq, Nk, causal)}")


def test_fp8_scale_and_descales():
    """The score scale and each descale act as the oracle says: a doubled value
    descale doubles O, query/key descales are a score scale."""
    q8, k8, vt8, ds = make_qkv_fp8(1, 2, 256, 256, 128, seed=50, device=_dev())
    _full(q8, k8, vt8, (ds[0], ds[1], 2 * ds[2]), True, what="descale_v x2")
    _full(q8, k8, vt8, (4 * ds[0], 0.5 * ds[1], ds[2]), False, scale=0.05, what="scale 0.05")
    _full(q8, k8, vt8, (1.0, 1.0, 1.0), False, scale=1e-3, what="unit descales")


def test_fp8_wide_logits():
    """sigma 1.7 queries and keys: large row maxima and moves of the reference."""
    q8, k8, vt8, ds = make_qkv_fp8(1, 2, 512, 512, 128, seed=51, device=_dev(), sigma_qk=1.7)
    _full(q8, k8, vt8, ds, True, what="wide logits")


def test_fp8_extreme_codes():
    """Every query and key code at +-448 (the largest E4M3 magnitude) and a
    one-hot dominant key: saturated operands, scores far beyond one tile's
    first maximum."""
    B, H, N = 1, 1, 256
    dev = _dev()
    q8 = torch.full((B, H, N, 128), 0x7E, dtype=torch.uint8, device=dev)
    k8 = torch.full((B, H, N, 128), 0x00, dtype=torch.uint8, device=dev)
    k8[:, :, 200, :] = 0x7E                       # +448: key 200 dominates every row that sees it
    k8[:, :, 7, ::2] = 0xFE                       # -448 on half of key 7's columns
    g = torch.Generator(device=dev).manual_seed(52)
    v = torch.randn((B, H, N, 128), generator=g, device=dev)
    vt8 = torch.clamp(v * 40, -448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    vt8 = vt8.transpose(2, 3).contiguous()
    _full(q8, k8, vt8, (2.0 ** -6, 2.0 ** -6, 1 / 40), False, what="saturated non-causal")
    _full(q8, k8, vt8, (2.0 ** -6, 2.0 ** -6, 1 / 40), True, what="saturated causal")


def _sampled(w, rows_per_head=48, heads=4, seed=None):
    """Sampled rows of a full-size workload: the kernel on the whole problem,
    the oracle on the sampled rows of a few heads (decoded head by head)."""
    dev = _dev()
    q8, k8, vt8, ds = make_workload_fp8(w, device=dev, seed=seed)
    o, lse = binding.attn_fwd_fp8(q8, k8, vt8, *ds, causal=w.causal)
    torch.cuda.synchronize()
    BH = w.B * w.H
    rng = np.random.default_rng(7)
    hs = np.unique(np.concatenate([[0, BH - 1], rng.choice(BH, heads - 2, replace=False)]))
    of = o.reshape(BH, w.Nq, w.d)
    lf = lse.reshape(BH, w.Nq)
    q8f, k8f, vt8f = (t.reshape(BH, *t.shape[2:]) for t in (q8, k8, vt8))
    for h in hs:
        sl = slice(int(h), int(h) + 1)
        qn, kn, vn = (_np(t[sl]).reshape(1, 1, *t.shape[1:]) for t in (q8f, k8f, vt8f))
        edge = [0, 1, 127, 128, 255, 256, w.Nq - 129, w.Nq - 128, w.Nq - 1]
        ii = np.unique(np.concatenate([edge, rng.choice(w.Nq, rows_per_head, replace=False)]))
        rows = np.stack([np.zeros_like(ii), ii], axis=1)
        qd, kd, vd = oracle.fp8_operands(qn, kn, vn, *ds)
        _, _, va = oracle.fp8_operands(qn, kn, _abs_codes(vn), *ds)
        ro, rl = oracle.attention_rows(qd, kd, vd, rows, causal=w.causal, scale=w.scale)
        ra, _ = oracle.attention_rows(qd, kd, va, rows, causal=w.causal, scale=w.scale)
        rr = _small_p_term(qd[0], kd[0], vd[0], rows, w.causal, w.scale)
        idx = torch.as_tensor(ii, device=dev)
        _check(_np(of[int(h)].index_select(0, idx).float()), _np(lf[int(h)].index_select(0, idx)),
               ro, rl, ra, rr, f"{w.name} head {h}")


def test_fp8_headline_workload_sampled():
    _sampled(WORKLOADS["b2h16n4096d128_causal"])


def test_fp8_long_workload_sampled():
    _sampled(WORKLOADS["b1h32n16384d128_causal"], rows_per_head=24, heads=3)


def test_fp8_rejects_unsupported_sizes():
    dev = _dev()
    q8 = torch.zeros((1, 1, 64, 128), dtype=torch.uint8, device=dev)
    k8 = torch.zeros((1, 1, 40, 128), dtype=torch.uint8, device=dev)
    vt8 = torch.zeros((1, 1, 128, 40), dtype=torch.uint8, device=dev)
    with pytest.raises(binding.GbattnError):
        binding.attn_fwd_fp8(q8, k8, vt8)   # Nk = 40 is not a multiple of 16
    assert binding.device_error() == 0
