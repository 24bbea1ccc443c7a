"""The CUDA path against the fp64 oracle, element by element, through the C ABI.

Tolerances are the ones the study states for bf16 inputs and outputs:
O within 2e-2 max-abs and 1e-3 mean-abs of the fp64 result, lse within 2e-3.
Inputs come from the seeded generator; large workloads are checked on sampled
rows (rows are independent, so a sampled row is checked exactly).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_flashattention_fwd_gb300 import binding
from attention_flashattention_fwd_gb300.inputs import WORKLOADS, bf16_bits, make_qkv, make_workload
from tests.conftest import nan_full

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 2e-3

pytestmark = pytest.mark.gpu


def _dev():
    return torch.device("cuda:0")


def _assert_close(o, lse, ro, rl, what=""):
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{what}: non-finite output"
    e = np.abs(o - ro)
    el = np.abs(lse - rl)
    msg = f"{what}: O max {e.max():.3g} mean {e.mean():.3g}, lse max {el.max():.3g}"
    assert e.max() <= O_MAX and e.mean() <= O_MEAN and el.max() <= LSE_MAX, msg
    return e.max(), e.mean(), el.max()


def _full_check(q, k, v, causal, scale=None, what=""):
    o, lse = binding.attn_fwd(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=causal,
                              scale=scale)
    return _assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, what)


# --------------------------------------------------------------- prefill shapes

PREFILL_SHAPES = [
    # B, H, Nq, Nk, d, causal
    (1, 1, 128, 128, 64, False),    # the tiny workload's shape
    (1, 2, 256, 256, 64, False),
    (1, 2, 256, 256, 128, False),
    (2, 2, 384, 384, 128, True),
    (1, 2, 300, 300, 64, True),     # ragged last tile
    (1, 1, 77, 77, 128, True),      # less than one tile
    (1, 1, 77, 77, 64, False),
    (1, 3, 200, 513, 128, False),   # Nq != Nk, ragged keys
    (1, 1, 128, 50, 64, False),     # fewer keys than a tile
    (1, 1, 5, 3, 128, False),
    (1, 1, 1, 1, 64, False),        # one query, one key
    (1, 1, 1, 700, 128, False),     # a single query row through the prefill kernel
    (1, 1, 1000, 1000, 128, True),  # many tiles, ragged, causal
    (2, 1, 640, 640, 64, True),
    (1, 1, 1280, 1280, 128, False),
    # causal with Nq < Nk: the queries are the newest Nq tokens (query i sees
    # keys j <= i + Nk - Nq); offsets that are and are not multiples of a tile
    (1, 2, 200, 513, 128, True),
    (2, 2, 128, 1024, 64, True),
    (1, 3, 384, 1000, 128, True),
    (1, 1, 77, 78, 64, True),
    (1, 2, 300, 4096, 128, True),
    (1, 1, 1, 700, 128, True),      # one causal query row sees every key
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", PREFILL_SHAPES,
                         ids=[f"b{B}h{H}q{Nq}k{Nk}d{d}{'c' if c else ''}"
                              for B, H, Nq, Nk, d, c in PREFILL_SHAPES])
def test_prefill_matches_oracle(B, H, Nq, Nk, d, causal):
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed=11 + Nq + Nk + d, device=_dev())
    _full_check(q, k, v, causal, what=f"{(B, H, Nq, Nk, d, causal)}")


# Non-causal work whose query-tile pairs would leave the last wave of the
# persistent grid part-full runs that tail as single 128-row tiles.  On a
# 152-SM GB300: 158 pairs -> 152 pairs + 12 single tiles (of which the last
# head's upper halves, rows 384..511 of 300, are empty), 154 pairs -> 152
# pairs + 4 single tiles, 160 pairs -> 152 + 16.  Every row is checked.
@pytest.mark.parametrize("B,H,Nq,Nk,d", [
    (1, 79, 300, 300, 64),
    (1, 80, 260, 260, 64),
    (1, 79, 384, 640, 128),    # Nq != Nk
    (1, 77, 512, 512, 128),
    (1, 77, 512, 512, 64),
    (1, 79, 1000, 1000, 128),  # ragged last key tile
    (1, 77, 300, 1024, 128),   # the tail tiles hold rows past Nq
])
def test_last_wave_single_tiles_match_oracle(B, H, Nq, Nk, d):
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed=23 + Nq + Nk + d, device=_dev())
    _full_check(q, k, v, False, what=f"{(B, H, Nq, Nk, d)} split tail")


# A causal launch of at most one wave of query-tile pairs runs every pair as
# two single tiles, heaviest first.  On a 152-SM GB300: 19 heads of 2048 rows
# are 152 pairs (split into 304 tiles, two rounds), 20 heads 160 pairs (kept
# whole); rows 384..511 of 300 are an empty half; Nq < Nk moves the diagonal.
# Every row is checked.
@pytest.mark.parametrize("B,H,Nq,Nk,d", [
    (1, 19, 2048, 2048, 128),
    (1, 20, 2048, 2048, 128),
    (1, 4, 300, 300, 128),
    (2, 3, 1000, 1500, 64),
    (1, 2, 640, 4096, 128),
])
def test_one_wave_causal_single_tiles_match_oracle(B, H, Nq, Nk, d):
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed=31 + Nq + Nk + d, device=_dev())
    _full_check(q, k, v, True, what=f"{(B, H, Nq, Nk, d)} causal single tiles")


def test_one_wave_causal_16384_token_head_sampled():
    # 64 pairs as 128 single tiles; the last tiles see every key
    _sampled_custom(1, 1, 16384, 16384, 128, True, seed=3004,
                    extra_rows=[0, 127, 128, 255, 8191, 16255, 16256, 16383])


def test_chunked_prefill_equals_prefill_at_once():
    """A 1000-token causal prefill run as three query chunks, each against the
    keys and values of every token up to its end (the KV cache so far), gives
    the rows of the run at once; both are checked against the oracle."""
    B, H, N, d = 1, 2, 1000, 128
    q, k, v = make_qkv(B, H, N, N, d, seed=23, device=_dev())
    o, lse = binding.attn_fwd(q, k, v, causal=True)
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=True)
    start = 0
    for end in (256, 601, 1000):
        oc, lc = binding.attn_fwd(q[:, :, start:end].contiguous(), k[:, :, :end].contiguous(),
                                  v[:, :, :end].contiguous(), causal=True)
        torch.cuda.synchronize()
        _assert_close(oc.float().cpu().numpy(), lc.cpu().numpy(), ro[:, :, start:end],
                      rl[:, :, start:end], f"chunk [{start}, {end})")
        # the two runs round differently only through tile boundaries
        assert (oc.float() - o[:, :, start:end].float()).abs().max().item() <= 2 * O_MAX
        start = end


def test_causal_single_query_dispatches_to_decode():
    q, k, v = make_qkv(2, 3, 1, 1500, 128, seed=24, device=_dev())
    o, lse = binding.attention(q, k, v, causal=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=True)
    _assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, "causal decode")


def test_prefill_scale_argument():
    q, k, v = make_qkv(1, 2, 256, 256, 128, seed=21, device=_dev())
    _full_check(q, k, v, True, scale=0.3, what="scale=0.3")
    _full_check(q, k, v, False, scale=0.02, what="scale=0.02")


def test_prefill_wide_logits():
    # sigma 3 logits: large row maxima, many rescales of the running max
    q, k, v = make_qkv(1, 2, 512, 512, 128, seed=22, device=_dev(), sigma_qk=1.7)
    _full_check(q, k, v, True, what="wide logits causal")
    _full_check(q, k, v, False, what="wide logits")


def test_tiny_workload():
    w = WORKLOADS["tiny_b1h1n128d64"]
    q, k, v = make_workload(w, device=_dev())
    _full_check(q, k, v, w.causal, scale=w.scale, what=w.name)


def test_b4h8n1024d64_workload_all_rows():
    w = WORKLOADS["b4h8n1024d64"]
    q, k, v = make_workload(w, device=_dev())
    _full_check(q, k, v, w.causal, scale=w.scale, what=w.name)


def _sampled_rows(w, rng, full_heads, n_random, extra_rows):
    BH = w.B * w.H
    rows = []
    for bh in full_heads:
        rows += [(bh, i) for i in range(w.Nq)]
    for i in extra_rows:
        rows.append((rng.integers(BH), i))
    rows += [(rng.integers(BH), rng.integers(w.Nq)) for _ in range(n_random)]
    return np.array(rows, dtype=np.int64)


def _rows_check(w, full_heads, n_random, extra_rows):
    q, k, v = make_workload(w, device=_dev())
    o, lse = binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1234)
    rows = _sampled_rows(w, rng, full_heads, n_random, extra_rows)
    ro, rl = oracle.attention_rows(bf16_bits(q), bf16_bits(k), bf16_bits(v), rows,
                                   causal=w.causal, scale=w.scale)
    BH = w.B * w.H
    idx = torch.as_tensor(rows[:, 0] * w.Nq + rows[:, 1], device=o.device)
    og = o.reshape(BH * w.Nq, w.d).index_select(0, idx).float().cpu().numpy()
    lg = lse.reshape(BH * w.Nq).index_select(0, idx).cpu().numpy()
    return _assert_close(og, lg, ro, rl, w.name)


def test_b2h16n4096d128_causal_sampled():
    w = WORKLOADS["b2h16n4096d128_causal"]
    _rows_check(w, full_heads=[0, w.B * w.H - 1], n_random=256,
                extra_rows=[0, 127, 128, 255, 256, 4095])


def test_b2h16n4096d128_noncausal_sampled():
    from attention_flashattention_fwd_gb300.inputs import EXTRA_WORKLOADS
    w = EXTRA_WORKLOADS["b2h16n4096d128"]
    _rows_check(w, full_heads=[5], n_random=256, extra_rows=[0, 127, 128, 4095])


def test_b1h32n16384d128_causal_sampled():
    w = WORKLOADS["b1h32n16384d128_causal"]
    # one full head (all 16384 rows, ~70 GFLOP in the fp64 oracle) plus samples
    _rows_check(w, full_heads=[w.B * w.H - 1], n_random=384,
                extra_rows=[0, 1, 127, 128, 255, 256, 8191, 8192, 16383] + list(range(0, 512, 7)))


# ---------------------------------------------------------------- decode

DECODE_SHAPES = [
    # B, H, Nk, d
    (1, 1, 1, 64),
    (1, 1, 511, 128),
    (1, 1, 513, 128),
    (2, 3, 3000, 64),
    (2, 4, 8192, 128),
    (1, 1, 20000, 128),
    (3, 5, 777, 64),
    (16, 32, 1024, 128),
]


@pytest.mark.parametrize("B,H,Nk,d", DECODE_SHAPES,
                         ids=[f"b{B}h{H}k{Nk}d{d}" for B, H, Nk, d in DECODE_SHAPES])
def test_decode_matches_oracle(B, H, Nk, d):
    q, k, v = make_qkv(B, H, 1, Nk, d, seed=31 + Nk + d, device=_dev())
    o, lse = binding.attn_fwd_decode(q, k, v)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v))
    _assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, f"decode {B, H, Nk, d}")


def test_decode_workload_sampled_heads():
    w = WORKLOADS["decode_b64h32nk8192d128"]
    q, k, v = make_workload(w, device=_dev())
    need = binding.decode_workspace_bytes(w.B, w.H, w.Nk, w.d)
    ws = torch.empty(need, dtype=torch.uint8, device=_dev())
    o, lse = binding.attn_fwd_decode(q, k, v, scale=w.scale, workspace=ws)
    torch.cuda.synchronize()
    BH = w.B * w.H
    sel = np.sort(np.random.default_rng(99).choice(BH, 256, replace=False))
    sel[0], sel[-1] = 0, BH - 1
    idx = torch.as_tensor(sel, device=_dev())
    qs = q.reshape(BH, 1, 1, w.d).index_select(0, idx).reshape(1, len(sel), 1, w.d)
    ks = k.reshape(BH, w.Nk, w.d).index_select(0, idx).reshape(1, len(sel), w.Nk, w.d)
    vs = v.reshape(BH, w.Nk, w.d).index_select(0, idx).reshape(1, len(sel), w.Nk, w.d)
    ro, rl = oracle.attention(bf16_bits(qs), bf16_bits(ks), bf16_bits(vs), scale=w.scale)
    og = o.reshape(BH, w.d).index_select(0, idx).float().cpu().numpy().reshape(ro.shape)
    lg = lse.reshape(BH).index_select(0, idx).cpu().numpy().reshape(rl.shape)
    _assert_close(og, lg, ro, rl, w.name)


def test_decode_equals_prefill_path():
    q, k, v = make_qkv(2, 4, 1, 2500, 128, seed=41, device=_dev())
    o1, l1 = binding.attn_fwd_decode(q, k, v)
    o2, l2 = binding.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= O_MAX
    assert (l1 - l2).abs().max().item() <= LSE_MAX


def test_decode_rejects_small_workspace():
    q, k, v = make_qkv(1, 1, 1, 8192, 128, seed=42, device=_dev())
    need = binding.decode_workspace_bytes(1, 1, 8192, 128)
    assert need > 0
    ws = torch.empty(need - 16, dtype=torch.uint8, device=_dev())
    with pytest.raises(binding.GbattnError) as ei:
        binding.attn_fwd_decode(q, k, v, workspace=ws)
    assert ei.value.status == 1


# ------------------------------------------------- invariants through the kernels

def test_q_zero_gives_mean_of_visible_values():
    B, H, N, d = 1, 2, 300, 128
    _, k, v = make_qkv(B, H, N, N, d, seed=51, device=_dev())
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device=_dev())
    vd = v.double().cpu()
    o, lse = binding.attn_fwd(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert (o.double().cpu() - vd.mean(dim=2, keepdim=True)).abs().max().item() <= O_MAX
    assert (lse.double().cpu() - math.log(N)).abs().max().item() <= LSE_MAX
    o, lse = binding.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    prefix = vd.cumsum(dim=2) / torch.arange(1, N + 1, dtype=torch.float64)[None, None, :, None]
    assert (o.double().cpu() - prefix).abs().max().item() <= O_MAX
    ln = torch.log(torch.arange(1, N + 1, dtype=torch.float64))[None, None]
    assert (lse.double().cpu() - ln).abs().max().item() <= LSE_MAX
    # decode: the column mean of V
    od, ld = binding.attn_fwd_decode(q[:, :, :1].contiguous(), k, v)
    torch.cuda.synchronize()
    assert (od.double().cpu() - vd.mean(dim=2, keepdim=True)).abs().max().item() <= O_MAX
    assert (ld.double().cpu() - math.log(N)).abs().max().item() <= LSE_MAX


def test_causal_row0_is_v0():
    q, k, v = make_qkv(2, 3, 256, 256, 64, seed=52, device=_dev())
    o, lse = binding.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o[:, :, 0], v[:, :, 0])
    ref = (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1) / 8.0
    assert (lse[:, :, 0].double() - ref).abs().max().item() <= LSE_MAX


def test_dominant_logit_selects_its_value_row():
    B, H, N, d = 1, 2, 384, 128
    q, k, v = make_qkv(B, H, N, N, d, seed=53, device=_dev())
    q = (q.float() * 0.05).to(torch.bfloat16)
    k = (k.float() * 0.05).to(torch.bfloat16)
    jstar, i = 200, 300
    qi = q[:, :, i].double()
    k[:, :, jstar] = (60.0 * qi / (qi * qi).sum(-1, keepdim=True)).to(torch.bfloat16)
    o, lse = binding.attn_fwd(q, k, v, causal=False, scale=1.0)
    torch.cuda.synchronize()
    assert (o[:, :, i].float() - v[:, :, jstar].float()).abs().max().item() <= O_MAX
    logit = (q[:, :, i].double() * k[:, :, jstar].double()).sum(-1)
    assert (lse[:, :, i].double() - logit).abs().max().item() <= 5e-2


def test_value_affine_map():
    q, k, v = make_qkv(1, 2, 256, 256, 128, seed=54, device=_dev())
    v2 = (v.float() * 0.5 + 0.25).to(torch.bfloat16)  # exact in bf16 for |v| < 2^7
    o1, l1 = binding.attn_fwd(q, k, v, causal=True)
    o2, l2 = binding.attn_fwd(q, k, v2, causal=True)
    torch.cuda.synchronize()
    assert (o2.float() - (o1.float() * 0.5 + 0.25)).abs().max().item() <= O_MAX
    assert torch.equal(l1, l2)


def test_deterministic_and_stream_aware():
    q, k, v = make_qkv(2, 4, 640, 640, 128, seed=55, device=_dev())
    o1, l1 = binding.attn_fwd(q, k, v, causal=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, l2 = binding.attn_fwd(q, k, v, causal=True, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("B,H,N,d", [(1, 4, 512, 128), (1, 3, 300, 64), (1, 1, 200, 128),
                                     (1, 5, 200, 64), (1, 7, 130, 128),
                                     (2, 5, 256, 128)])
def test_from_host_end_to_end(B, H, N, d):
    # the heads cross the host link in up to five chunks (sizes falling off) on three streams
    q, k, v = make_qkv(B, H, N, N, d, seed=56 + H, device="cpu")
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = nan_full((B, H, N, d), torch.bfloat16, pin=True)
    lh = nan_full((B, H, N), torch.float32, pin=True)
    dq, dk, dv = (nan_full(t.shape, t.dtype, _dev()) for t in (q, k, v))
    do_ = nan_full((B, H, N, d), torch.bfloat16, _dev())
    dl = nan_full((B, H, N), torch.float32, _dev())
    s = torch.cuda.Stream()
    binding.attn_fwd_from_host(qh, kh, vh, oh, lh, dq, dk, dv, do_, dl, causal=True, stream=s)
    s.synchronize()  # the caller's stream alone covers the whole call
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=True)
    _assert_close(oh.float().numpy(), lh.numpy(), ro, rl, "from_host")


def test_no_device_error_reported():
    assert binding.device_error() == 0


@pytest.mark.parametrize("name", ["b2h16n4096d128_causal", "b4h8n1024d64"])
def test_repeated_launches_are_bitwise_stable(name):
    # 30 launches of one workload must give identical bits: an ordering race
    # between the tensor-core products and the softmax would show up here
    w = WORKLOADS[name]
    q, k, v = make_workload(w, device=_dev())
    o0, l0 = binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
    o, lse = torch.empty_like(o0), torch.empty_like(l0)
    for _ in range(30):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)
        torch.cuda.synchronize()
        assert torch.equal(o, o0) and torch.equal(lse, l0)


# ------------------------------------------------------------ large and wide shapes

def _sampled_custom(B, H, Nq, Nk, d, causal, seed, extra_rows, n_random=96, scale=None):
    from attention_flashattention_fwd_gb300.inputs import Workload
    w = Workload(f"b{B}h{H}q{Nq}k{Nk}d{d}", B, H, Nq, Nk, d, causal, seed=seed)
    return _rows_check(w, full_heads=[], n_random=n_random, extra_rows=extra_rows)


def test_65536_token_causal_head_sampled():
    # positions near 2^16: query and key offsets, TMA coordinates and row offsets
    _sampled_custom(1, 1, 65536, 65536, 128, True, seed=3001,
                    extra_rows=[0, 1, 127, 128, 32767, 32768, 65407, 65408, 65535])


def test_32768_tokens_d64_noncausal_sampled():
    _sampled_custom(1, 2, 32768, 32768, 64, False, seed=3002, extra_rows=[0, 16383, 32767])


def test_many_small_heads_sampled():
    # 1024 (b, h) pairs of 256 tokens: many work items per CTA
    _sampled_custom(16, 64, 256, 256, 64, True, seed=3003, extra_rows=[0, 255], n_random=256)


def test_decode_8192_heads_sampled():
    B, H, Nk, d = 256, 32, 1024, 64
    q, k, v = make_qkv(B, H, 1, Nk, d, seed=3004, device=_dev())
    o, lse = binding.attn_fwd_decode(q, k, v)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3005)
    heads = np.unique(np.concatenate([[0, B * H - 1], rng.integers(0, B * H, 120)]))
    rows = np.stack([heads, np.zeros_like(heads)], axis=1)
    ro, rl = oracle.attention_rows(bf16_bits(q), bf16_bits(k), bf16_bits(v), rows)
    og = o.reshape(B * H, d)[torch.as_tensor(heads, device=o.device)].float().cpu().numpy()
    lg = lse.reshape(B * H)[torch.as_tensor(heads, device=o.device)].cpu().numpy()
    _assert_close(og, lg, ro, rl, "decode 8192 heads")


@pytest.mark.parametrize("name", ["b2h16n4096d128_causal", "b2h16n4096d128",
                                  "b1h32n16384d128_causal"])
def test_full_workload_every_row_against_fp32_recompute(name):
    """Every row of every head of the full-size workloads, against an fp32
    recomputation of the definition on the GPU (torch products, head by head:
    S = scale Q K^T with the causal mask, lse = log sum exp S, O = softmax(S) V)
    -- a check independent of the library beside the fp64 oracle's full head and
    sampled rows above.  The outputs start as NaN, so a tile no work item wrote
    fails here wherever it is."""
    from attention_flashattention_fwd_gb300.inputs import EXTRA_WORKLOADS
    w = WORKLOADS.get(name) or EXTRA_WORKLOADS[name]
    q, k, v = make_workload(w, device=_dev())
    o, lse = binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    BH = w.B * w.H
    qf, kf, vf = (t.reshape(BH, -1, w.d) for t in (q, k, v))
    of, lf = o.reshape(BH, w.Nq, w.d), lse.reshape(BH, w.Nq)
    mask = None
    if w.causal:
        i = torch.arange(w.Nq, device=_dev()).view(-1, 1)
        j = torch.arange(w.Nk, device=_dev()).view(1, -1)
        mask = j > i + (w.Nk - w.Nq)
    worst_o = worst_l = 0.0
    sum_o = 0.0
    for h in range(BH):
        s = (qf[h].float() @ kf[h].float().T) * w.scale
        if mask is not None:
            s.masked_fill_(mask, float("-inf"))
        rl = torch.logsumexp(s, dim=1)
        ro = torch.softmax(s, dim=1) @ vf[h].float()
        e = (of[h].float() - ro).abs()
        worst_o = max(worst_o, e.max().item())
        sum_o += e.mean().item()
        worst_l = max(worst_l, (lf[h] - rl).abs().max().item())
        del s, ro, rl, e
    assert worst_o <= O_MAX and sum_o / BH <= O_MEAN and worst_l <= LSE_MAX, \
        (name, worst_o, sum_o / BH, worst_l)
    assert binding.device_error() == 0


def test_causal_head_groups_uneven_last_group_and_chunk():
    """Causal work whose K and V exceed L2 several times over is dealt in head
    groups (32 MB of K and V per head here: groups of 3, 3, 3 and 1 heads), with
    a causal query chunk shorter than the keys (Nq < Nk): sampled rows of every
    head against the oracle, first and last rows of each pair of query tiles
    included, and every output written (NaN-filled before the call)."""
    from attention_flashattention_fwd_gb300.inputs import Workload
    w = Workload("b1h10q2048k65536d128_causal", 1, 10, 2048, 65536, 128, True, seed=2100)
    q, k, v = make_workload(w, device=_dev())
    o, lse = binding.attn_fwd(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(77)
    rows = [(h, i) for h in range(10) for i in (0, 255, 256, 511, 1792, 2047)]
    rows += [(int(rng.integers(10)), int(rng.integers(2048))) for _ in range(60)]
    rows = np.array(rows, dtype=np.int64)
    ro, rl = oracle.attention_rows(bf16_bits(q), bf16_bits(k), bf16_bits(v), rows, causal=True,
                                   scale=w.scale)
    idx = torch.as_tensor(rows[:, 0] * w.Nq + rows[:, 1], device=o.device)
    og = o.reshape(10 * w.Nq, w.d).index_select(0, idx).float().cpu().numpy()
    lg = lse.reshape(10 * w.Nq).index_select(0, idx).cpu().numpy()
    _assert_close(og, lg, ro, rl, w.name)
    assert binding.device_error() == 0


def test_from_host_long_workload_bit_identical():
    """The bench's end-to-end call at full size: the long workload (B1 H32 N16384
    d128 causal) from pinned host buffers through attn_fwd_from_host (five head
    chunks on three streams) gives the same bits as attn_fwd on the device copy
    (every row's products run in the same order whichever heads share a launch),
    which the tests above check against the oracle and an fp32 recomputation."""
    w = WORKLOADS["b1h32n16384d128_causal"]
    q, k, v = make_workload(w, device=_dev())
    o1, l1 = binding.attn_fwd(q, k, v, causal=True, scale=w.scale)
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    oh = nan_full(o1.shape, torch.bfloat16, pin=True)
    lh = nan_full(l1.shape, torch.float32, pin=True)
    dq, dk, dv = (nan_full(t.shape, t.dtype, _dev()) for t in (q, k, v))
    do_ = nan_full(o1.shape, torch.bfloat16, _dev())
    dl = nan_full(l1.shape, torch.float32, _dev())
    s = torch.cuda.Stream()
    binding.attn_fwd_from_host(qh, kh, vh, oh, lh, dq, dk, dv, do_, dl, causal=True,
                               scale=w.scale, stream=s)
    s.synchronize()
    assert torch.equal(oh, o1.cpu()) and torch.equal(lh, l1.cpu())
    assert binding.device_error() == 0
