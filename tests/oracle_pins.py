"""Checks that pin the fp64 oracle to facts fixed outside the oracle itself.

Each function raises AssertionError when the oracle disagrees with what the
lecture pages print or with what the mathematics of attention fixes.  They are
collected by ``test_oracle_pins.py`` and re-run against deliberately broken
copies of the oracle by ``test_oracle_mutants.py`` (every plausible mistake has
to fail at least one of them).
"""
import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# -- values printed by the pages ---------------------------------------------

def pin_exercise8_online_softmax(orc):
    """CS336 L5 exercise 8: online softmax of [1, 3 | 2, 5] in two blocks."""
    g = _golden("cs336_l5_exercise8.json")
    m, l = orc.online_softmax_blocks(g["x"], g["block_ends"])
    for b, exp in enumerate(g["after_block"]):
        assert m[b] == exp["m"], (b, m[b], exp["m"])
    tol0 = 0.5 * 10 ** -g["after_block"][0]["printed_decimals"]
    assert abs(l[0] - g["after_block"][0]["l"]) <= tol0, l[0]
    # the page sums three terms it rounded to 4 decimals: allow 3 half-units
    tol1 = 1.5 * 10 ** -g["after_block"][1]["printed_decimals"]
    assert abs(l[1] - g["after_block"][1]["l"]) <= tol1, l[1]
    t = g["second_update_terms"]
    half = 0.5 * 10 ** -t["printed_decimals"]
    assert abs(l[0] * math.exp(m[0] - m[1]) - t["old_l_rescaled"]) <= half
    # the same m, l through the two-block merge rule
    mm, ll, _ = orc.softmax_merge(m[0], l[0], np.zeros(1), 5.0, math.exp(2 - 5) + 1.0,
                                  np.zeros(1))
    assert mm == 5.0 and abs(ll - l[1]) <= 1e-15
    # the probability of the last element, through full attention: with q = e0,
    # k_j = x_j e0, scale 1 and V = I the output row is the softmax row itself
    x = np.array(g["x"])
    n = len(x)
    q = np.zeros((1, 1, 1, n)); q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, 1, n, n)); k[0, 0, :, 0] = x
    v = np.eye(n)[None, None]
    o, lse = orc.attention(q, k, v, causal=False, scale=1.0)
    p_last = g["softmax_of_last"]
    assert abs(o[0, 0, 0, -1] - p_last["value"]) <= 0.5 * 10 ** -p_last["printed_decimals"]
    assert abs(o[0, 0, 0, -1] - math.exp(x[-1] - m[1]) / l[1]) <= 1e-15
    # L = m + log l with the page's final (m, l)
    assert abs(lse[0, 0, 0] - (m[1] + math.log(l[1]))) <= 1e-14


# -- closed forms and invariants ---------------------------------------------

def pin_rows_sum_to_one(orc):
    """With V = I (d = Nk) the output row is the probability row: rows sum to 1,
    entries are >= 0, and causal rows are exactly 0 beyond the diagonal."""
    n = 37
    q = _rand((2, 3, n, n), 1)
    k = _rand((2, 3, n, n), 2)
    v = np.broadcast_to(np.eye(n), (2, 3, n, n)).copy()
    for causal in (False, True):
        p, _ = orc.attention(q, k, v, causal=causal, scale=0.3)
        assert np.all(p >= 0)
        assert np.max(np.abs(p.sum(-1) - 1.0)) <= 1e-14
        if causal:
            upper = np.triu(np.ones((n, n), bool), 1)
            assert np.all(p[..., upper] == 0.0)
            assert np.all(p[..., ~upper] > 0.0)


def pin_q_zero(orc):
    """Q = 0: every visible logit is 0, so O_i is the mean of the visible V rows
    and lse_i = ln(number of visible keys)."""
    B, H, n, d = 2, 2, 29, 8
    q = np.zeros((B, H, n, d))
    k = _rand((B, H, n, d), 3)
    v = _rand((B, H, n, d), 4)
    o, lse = orc.attention(q, k, v, causal=False)
    assert np.max(np.abs(o - v.mean(axis=2, keepdims=True))) <= 1e-14
    assert np.max(np.abs(lse - math.log(n))) <= 1e-14
    o, lse = orc.attention(q, k, v, causal=True)
    prefix = np.cumsum(v, axis=2) / np.arange(1, n + 1)[None, None, :, None]
    assert np.max(np.abs(o - prefix)) <= 1e-14
    assert np.max(np.abs(lse - np.log(np.arange(1, n + 1))[None, None])) <= 1e-14


def pin_one_hot_dominant(orc):
    """A key whose logit beats every other by >= 50 takes all the weight:
    O_i = V_{j*} to within e^-50."""
    B, H, n, d = 1, 2, 40, 16
    q = _rand((B, H, n, d), 5) * 0.1
    k = _rand((B, H, n, d), 6) * 0.1
    v = _rand((B, H, n, d), 7)
    jstar, i = 17, 30
    # key j* points along q_i with q_i . k_j* = 80, far above every other logit
    k[:, :, jstar, :] = 80.0 * q[:, :, i, :] / np.sum(q[:, :, i, :] ** 2, axis=-1, keepdims=True)
    o, lse = orc.attention(q, k, v, causal=False, scale=1.0)
    others = np.einsum("bhc,bhjc->bhj", q[:, :, i, :], np.delete(k, jstar, axis=2))
    assert np.max(others) < 80.0 - 50.0
    bound = n * math.exp(-50) * np.max(np.abs(v)) * 2
    assert np.max(np.abs(o[:, :, i, :] - v[:, :, jstar, :])) <= bound
    assert np.max(np.abs(lse[:, :, i] - 80.0)) <= 1e-12


def pin_causal_row0(orc):
    """Causal row 0 sees only key 0: O_0 = V_0 and lse_0 = scale q_0 . k_0."""
    B, H, n, d = 2, 3, 19, 12
    q, k, v = _rand((B, H, n, d), 8), _rand((B, H, n, d), 9), _rand((B, H, n, d), 10)
    o, lse = orc.attention(q, k, v, causal=True, scale=0.25)
    assert np.array_equal(o[:, :, 0, :], v[:, :, 0, :])
    ref = 0.25 * np.einsum("bhc,bhc->bh", q[:, :, 0, :], k[:, :, 0, :])
    assert np.max(np.abs(lse[:, :, 0] - ref)) <= 1e-14


def pin_v_affine(orc):
    """Rows of P sum to 1, so O(a V + b) = a O(V) + b, and lse does not change."""
    B, H, n, d = 1, 2, 33, 8
    q, k, v = _rand((B, H, n, d), 11), _rand((B, H, n, d), 12), _rand((B, H, n, d), 13)
    for causal in (False, True):
        o1, l1 = orc.attention(q, k, v, causal=causal)
        o2, l2 = orc.attention(q, k, -1.5 * v + 0.75, causal=causal)
        assert np.max(np.abs(o2 - (-1.5 * o1 + 0.75))) <= 1e-13
        assert np.array_equal(l1, l2)


def pin_key_permutation(orc):
    """Non-causal attention is a set function of the (key, value) pairs."""
    B, H, n, d = 2, 2, 31, 8
    q, k, v = _rand((B, H, n, d), 14), _rand((B, H, n, d), 15), _rand((B, H, n, d), 16)
    perm = np.random.default_rng(17).permutation(n)
    o1, l1 = orc.attention(q, k, v)
    o2, l2 = orc.attention(q, k[:, :, perm], v[:, :, perm])
    assert np.max(np.abs(o1 - o2)) <= 1e-14
    assert np.max(np.abs(l1 - l2)) <= 1e-14


def pin_scale_is_applied(orc):
    """S = scale Q K^T: scaling Q by c with scale s equals scale c*s."""
    B, H, n, d = 1, 1, 21, 8
    q, k, v = _rand((B, H, n, d), 18), _rand((B, H, n, d), 19), _rand((B, H, n, d), 20)
    o1, l1 = orc.attention(q * 4.0, k, v, scale=0.125)
    o2, l2 = orc.attention(q, k, v, scale=0.5)
    assert np.max(np.abs(o1 - o2)) <= 1e-14 and np.max(np.abs(l1 - l2)) <= 1e-13
    # and the default is 1 / sqrt(d)
    o3, l3 = orc.attention(q, k, v)
    o4, l4 = orc.attention(q, k, v, scale=1.0 / math.sqrt(d))
    assert np.array_equal(o3, o4) and np.array_equal(l3, l4)


# -- blocked / online forms against the unblocked definition ------------------

def pin_blocked_equals_unblocked(orc):
    """The tiled forward (CS336 L5 8.3) equals naive attention for any block
    sizes, dividing N or not (CS336 L5 exercise 10a)."""
    B, H, n, d = 1, 2, 45, 8
    q, k, v = _rand((B, H, n, d), 21), _rand((B, H, n, d), 22), _rand((B, H, n, d), 23)
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, causal=causal)
        for br, bc in ((1, 1), (7, 5), (16, 16), (45, 45), (64, 3), (8, 64)):
            ob, lb = orc.attention_blocked(q, k, v, causal=causal, block_q=br, block_k=bc)
            assert np.max(np.abs(ob - o)) <= 1e-13, (causal, br, bc)
            assert np.max(np.abs(lb - lse)) <= 1e-13, (causal, br, bc)
    # fewer queries than keys (a chunk at the end of the sequence)
    qc = q[:, :, 26:]
    for causal in (False, True):
        o, lse = orc.attention(qc, k, v, causal=causal)
        for br, bc in ((1, 1), (7, 5), (16, 16), (4, 19)):
            ob, lb = orc.attention_blocked(qc, k, v, causal=causal, block_q=br, block_k=bc)
            assert np.max(np.abs(ob - o)) <= 1e-13, (causal, br, bc)
            assert np.max(np.abs(lb - lse)) <= 1e-13, (causal, br, bc)


def pin_merge_rule(orc):
    """CS149 L9 concept 9: attention over keys [0, s) and [s, n) separately,
    merged with m = max(m1, m2), l = e^{m1-m} l1 + e^{m2-m} l2, equals attention
    over all keys (the split-K decode combine)."""
    n, d = 50, 8
    q, k, v = _rand((1, 1, 3, d), 24), _rand((1, 1, n, d), 25), _rand((1, 1, n, d), 26)
    o, lse = orc.attention(q, k, v, scale=0.7)
    for s in (1, 13, 25, 49):
        o1, l1 = orc.attention(q, k[:, :, :s], v[:, :, :s], scale=0.7)
        o2, l2 = orc.attention(q, k[:, :, s:], v[:, :, s:], scale=0.7)
        for i in range(3):
            # a block's (m, l) is any pair with m + ln l = its lse; take m = lse, l = 1
            m, l, om = orc.softmax_merge(l1[0, 0, i], 1.0, o1[0, 0, i], l2[0, 0, i], 1.0,
                                         o2[0, 0, i])
            assert abs(m + math.log(l) - lse[0, 0, i]) <= 1e-13
            assert np.max(np.abs(om - o[0, 0, i])) <= 1e-14


# -- independent implementations -----------------------------------------------

def pin_bruteforce_fsum(orc):
    """Tiny shapes against a second implementation in pure Python with
    exactly-rounded sums (math.fsum)."""
    rng = np.random.default_rng(27)
    for (n, m, d, causal) in ((1, 1, 1, False), (3, 5, 2, False), (6, 6, 3, True), (8, 8, 4, True),
                              (3, 7, 2, True), (1, 4, 3, True)):
        q = rng.standard_normal((1, 1, n, d))
        k = rng.standard_normal((1, 1, m, d))
        v = rng.standard_normal((1, 1, m, d))
        scale = 0.9
        o, lse = orc.attention(q, k, v, causal=causal, scale=scale)
        for i in range(n):
            logits = [scale * math.fsum(q[0, 0, i, c] * k[0, 0, j, c] for c in range(d))
                      for j in range(m) if not (causal and j > i + (m - n))]
            mx = max(logits)
            w = [math.exp(s - mx) for s in logits]
            tot = math.fsum(w)
            assert abs(lse[0, 0, i] - (mx + math.log(tot))) <= 1e-13
            for c in range(d):
                ref = math.fsum(w[j] * v[0, 0, j, c] for j in range(len(w))) / tot
                assert abs(o[0, 0, i, c] - ref) <= 1e-14


def pin_causal_chunk_is_suffix(orc):
    """A KV cache that grows during inference (PDC L4 section 4.9): attending
    with the last Nq queries of a sequence against all of its Nk keys gives
    exactly the last Nq rows of causal attention over the whole sequence,
    whatever the split (prefill in chunks = prefill at once; Nq = 1 is a decode
    step, which sees every key)."""
    B, H, n, d = 2, 2, 29, 8
    q, k, v = _rand((B, H, n, d), 33), _rand((B, H, n, d), 34), _rand((B, H, n, d), 35)
    o, lse = orc.attention(q, k, v, causal=True, scale=0.6)
    for nq in (1, 5, 13, 28):
        oc, lc = orc.attention(q[:, :, n - nq:], k, v, causal=True, scale=0.6)
        assert np.array_equal(oc, o[:, :, n - nq:]), nq
        assert np.array_equal(lc, lse[:, :, n - nq:]), nq
    # the last row sees every key: a one-query causal call is the non-causal one
    od, ld = orc.attention(q[:, :, n - 1:], k, v, causal=False, scale=0.6)
    assert np.array_equal(od, o[:, :, n - 1:]) and np.array_equal(ld, lse[:, :, n - 1:])


def pin_torch_crosscheck(orc):
    """The pages' own checks (CS336 L5 8.2/8.3 demos): agreement with
    torch.softmax(S) @ V and F.scaled_dot_product_attention in float64."""
    import torch
    import torch.nn.functional as F
    B, H, n, d = 2, 3, 24, 16
    g = torch.Generator().manual_seed(28)
    q, k, v = (torch.randn(B, H, n, d, generator=g, dtype=torch.float64) for _ in range(3))
    for causal in (False, True):
        o, lse = orc.attention(q.numpy(), k.numpy(), v.numpy(), causal=causal)
        ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal)
        s = (q @ k.transpose(-1, -2)) / math.sqrt(d)
        if causal:
            s = s.masked_fill(torch.triu(torch.ones(n, n, dtype=torch.bool), 1), float("-inf"))
        ref2 = torch.softmax(s, dim=-1) @ v
        assert np.max(np.abs(o - ref.numpy())) <= 1e-12
        assert np.max(np.abs(o - ref2.numpy())) <= 1e-12
        assert np.max(np.abs(lse - torch.logsumexp(s, dim=-1).numpy())) <= 1e-12


def pin_bf16_widening(orc):
    """bf16 bit patterns are widened exactly: the uint16 path equals the float64
    path on the same values (values from torch's own bf16 -> float64)."""
    import torch
    g = torch.Generator().manual_seed(29)
    q, k, v = (torch.randn(1, 2, 9, 8, generator=g).to(torch.bfloat16) for _ in range(3))
    bits = [t.view(torch.int16).numpy().view(np.uint16) for t in (q, k, v)]
    wide = [t.to(torch.float64).numpy() for t in (q, k, v)]
    o1, l1 = orc.attention(*bits, causal=True)
    o2, l2 = orc.attention(*wide, causal=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_rows_equal_full(orc):
    """The sampled-row entry point returns exactly the full computation's rows."""
    B, H, n, d = 2, 2, 17, 8
    q, k, v = _rand((B, H, n, d), 30), _rand((B, H, n, d), 31), _rand((B, H, n, d), 32)
    o, lse = orc.attention(q, k, v, causal=True)
    rows = np.array([[0, 0], [3, 16], [1, 5], [2, 9]])
    orow, lrow = orc.attention_rows(q, k, v, rows, causal=True)
    for t, (bh, i) in enumerate(rows):
        assert np.array_equal(orow[t], o.reshape(B * H, n, d)[bh, i])
        assert lrow[t] == lse.reshape(B * H, n)[bh, i]


# -- backward (CS336 L5 section 8.4) ------------------------------------------

def _bwd_case(seed, B=1, H=2, nq=9, nk=13, d=6):
    return (_rand((B, H, nq, d), seed), _rand((B, H, nk, d), seed + 1),
            _rand((B, H, nk, d), seed + 2), _rand((B, H, nq, d), seed + 3))


def pin_bwd_finite_differences(orc):
    """The gradients are those of L = sum(O * dO) with O from the (separately
    pinned) forward: central differences on single entries of Q, K and V."""
    q, k, v, do = _bwd_case(40)
    h = 1e-5
    for causal in (False, True):
        dq, dk, dv = orc.attention_bwd(q, k, v, do, causal=causal, scale=0.45)

        def loss(qq, kk, vv):
            o, _ = orc.attention(qq, kk, vv, causal=causal, scale=0.45)
            return float(np.sum(o * do))

        rng = np.random.default_rng(41)
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for _ in range(6):
                idx = tuple(int(rng.integers(n)) for n in x.shape)
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
                args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
                fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
                assert abs(fd - g[idx]) <= 1e-7 * max(1.0, abs(fd)), (name, causal, idx, fd, g[idx])


def pin_bwd_torch_autograd(orc):
    """CS336 L5 section 8.4, demo 3: agreement with torch autograd in float64
    (the page reports differences of order 1e-15)."""
    import torch
    q, k, v, do = _bwd_case(44, B=2, H=2, nq=10, nk=17, d=8)
    for causal in (False, True):
        dq, dk, dv = orc.attention_bwd(q, k, v, do, causal=causal, scale=0.3)
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        s = (tq @ tk.transpose(-1, -2)) * 0.3
        if causal:  # the newest 10 of 17 tokens: query i sees keys j <= i + 7
            vis = torch.ones(10, 17, dtype=torch.bool).tril(7)
            s = s.masked_fill(~vis, float("-inf"))
        (torch.softmax(s, dim=-1) @ tv).backward(torch.tensor(do))
        for got, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
            assert np.max(np.abs(got - ref.numpy())) <= 1e-13, causal


def pin_bwd_exercise9_identity(orc):
    """CS336 L5 exercise 9: D_i = sum_j P_ij dP_ij equals sum_k dO_ik O_ik."""
    q, k, v, do = _bwd_case(48, nq=11, nk=11)
    for causal in (False, True):
        o, _ = orc.attention(q, k, v, causal=causal)
        rows = np.array([[bh, i] for bh in range(2) for i in range(11)])
        _, D = orc.attention_bwd_dq_rows(q, k, v, do, rows, causal=causal)
        ref = np.sum(do * o, axis=-1).reshape(-1)
        assert np.max(np.abs(D - ref)) <= 1e-13, causal


def pin_bwd_invariants(orc):
    """Softmax rows sum to one, so sum_j dS_ij = 0: the key gradients of a head
    sum to zero, the value gradients sum to the sum of dO, and with all keys
    equal the query gradient vanishes."""
    q, k, v, do = _bwd_case(52)
    for causal in (False, True):
        dq, dk, dv = orc.attention_bwd(q, k, v, do, causal=causal)
        assert np.max(np.abs(dk.sum(axis=2))) <= 1e-12, causal
        assert np.max(np.abs(dv.sum(axis=2) - do.sum(axis=2))) <= 1e-12, causal
        keq = np.broadcast_to(k[:, :, :1], k.shape).copy()
        dq0, _, _ = orc.attention_bwd(q, keq, v, do, causal=causal)
        assert np.max(np.abs(dq0)) <= 1e-12, causal


def pin_bwd_rows_and_keys_equal_full(orc):
    """The sampled entry points give the full backward's rows and keys."""
    q, k, v, do = _bwd_case(56, B=2, H=1, nq=8, nk=12)
    for causal in (False, True):
        dq, dk, dv = orc.attention_bwd(q, k, v, do, causal=causal)
        rows = np.array([[0, 0], [1, 7], [0, 3]])
        dqr, _ = orc.attention_bwd_dq_rows(q, k, v, do, rows, causal=causal)
        keys = np.array([[1, 0], [0, 11], [1, 5], [0, 4]])
        dkk, dvk = orc.attention_bwd_dkdv_keys(q, k, v, do, keys, causal=causal)
        for t, (bh, i) in enumerate(rows):
            assert np.max(np.abs(dqr[t] - dq.reshape(2, 8, -1)[bh, i])) <= 1e-13
        for t, (bh, j) in enumerate(keys):
            assert np.max(np.abs(dkk[t] - dk.reshape(2, 12, -1)[bh, j])) <= 1e-13
            assert np.max(np.abs(dvk[t] - dv.reshape(2, 12, -1)[bh, j])) <= 1e-13


# ---- FP8 (E4M3) operands ----------------------------------------------------

def _fp8_codes(shape, seed, sigma=1.0):
    """uint8 E4M3 codes of seeded normal values (torch's float8 rounding)."""
    import torch
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g) * sigma
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pin_e4m3_spec_values(orc):
    """Codes whose values the E4M3 definition fixes: zeros, the smallest and
    largest subnormal (2^-9, 7 * 2^-9), the smallest normal 2^-6, 0.5, 1, 1.5, 2,
    the largest finite value 448, the sign bit and the two NaN codes."""
    codes = np.array([0x00, 0x80, 0x01, 0x07, 0x08, 0x30, 0x38, 0x3C, 0x40, 0x7E, 0xB8, 0xFE,
                      0x7F, 0xFF], np.uint8)
    want = [0.0, -0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 0.5, 1.0, 1.5, 2.0, 448.0, -1.0,
            -448.0]
    got = orc.decode_e4m3(codes)
    assert np.array_equal(got[:12], np.array(want))
    assert np.signbit(got[1]) and np.all(np.isnan(got[12:]))


def pin_e4m3_torch(orc):
    """Every one of the 256 codes decodes to torch's float8_e4m3fn value, and the
    descale multiplies it."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for ds in (1.0, 0.3125, 7.0):
        got = orc.decode_e4m3(codes, ds)
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], ref[~nan] * ds)


def pin_fp8_attention_dequantised(orc):
    """FP8 attention equals fp64 attention of the operands torch dequantises,
    with V supplied transposed ([B,H,d,Nk]) and one descale per tensor."""
    import torch
    B, H, nq, nk, d = 1, 2, 7, 11, 16
    q8, k8 = _fp8_codes((B, H, nq, d), 40), _fp8_codes((B, H, nk, d), 41)
    vt8 = _fp8_codes((B, H, d, nk), 42)
    dq, dk, dv = 0.375, 1.75, 0.0625

    def deq(c, ds):
        return torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).to(torch.float64) * ds

    q, k = deq(q8, dq).numpy(), deq(k8, dk).numpy()
    v = deq(vt8, dv).transpose(2, 3).contiguous().numpy()
    for causal in (False, True):
        o1, l1 = orc.attention_fp8(q8, k8, vt8, causal=causal, scale=0.3, descale_q=dq,
                                   descale_k=dk, descale_v=dv)
        o2, l2 = orc.attention(q, k, v, causal=causal, scale=0.3)
        assert np.max(np.abs(o1 - o2)) <= 1e-14 and np.max(np.abs(l1 - l2)) <= 1e-14


def pin_fp8_descales(orc):
    """The value descale multiplies O and leaves lse alone; the query and key
    descales act as one factor on the scores (a change of scale)."""
    B, H, nq, nk, d = 1, 1, 5, 9, 8
    q8, k8, vt8 = _fp8_codes((B, H, nq, d), 43), _fp8_codes((B, H, nk, d), 44), \
        _fp8_codes((B, H, d, nk), 45)
    o1, l1 = orc.attention_fp8(q8, k8, vt8, scale=0.5)
    o2, l2 = orc.attention_fp8(q8, k8, vt8, scale=0.5, descale_v=3.0)
    assert np.max(np.abs(o2 - 3.0 * o1)) <= 1e-13 and np.array_equal(l1, l2)
    o3, l3 = orc.attention_fp8(q8, k8, vt8, scale=0.5, descale_q=2.0, descale_k=0.25)
    o4, l4 = orc.attention_fp8(q8, k8, vt8, scale=0.25)
    assert np.max(np.abs(o3 - o4)) <= 1e-13 and np.max(np.abs(l3 - l4)) <= 1e-13


# -- MX (microscaling) FP8 keys and values ----------------------------------

def pin_e8m0_spec_values(orc):
    """OCP MX v1.0 E8M0: value 2^(code - 127); 0xFF is NaN (decoded on E4M3
    elements equal to 1.0, code 0x38)."""
    codes = np.full((1, 7 * 32), 0x38, np.uint8)
    scales = np.array([[0, 1, 126, 127, 128, 254, 255]], np.uint8)
    got = orc.decode_mx(codes, scales).reshape(7, 32)
    want = [2.0 ** -127, 2.0 ** -126, 0.5, 1.0, 2.0, 2.0 ** 127]
    assert np.array_equal(got[:6], np.repeat(np.array(want)[:, None], 32, axis=1))
    assert np.all(np.isnan(got[6]))


def pin_e8m0_torch(orc):
    """Every E8M0 code decodes to torch's float8_e8m0fnu value."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = orc.decode_mx(np.full((256, 32), 0x38, np.uint8), codes[:, None])[:, 0]
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], ref[~nan])


def _mx_codes(rows, d, seed):
    """Seeded E4M3 element codes and E8M0 scale codes (scales 2^-6 .. 2^5)."""
    rng = np.random.default_rng(seed)
    codes = _fp8_codes((rows, d), seed)
    scales = rng.integers(121, 133, size=(rows, d // 32)).astype(np.uint8)
    return codes, scales


def pin_mx_block_layout(orc):
    """Element c of a row takes the scale of its block c // 32 of that row: the
    decode equals torch's E4M3 value times torch's E8M0 value of that block."""
    import torch
    codes, scales = _mx_codes(5, 128, 50)
    e = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    x = torch.from_numpy(scales.copy()).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    want = e * np.repeat(x, 32, axis=1)
    got = orc.decode_mx(codes, scales)
    assert np.array_equal(got, want)


def pin_mx_attention_dequantised(orc):
    """MX attention equals fp64 attention of the keys and values dequantised
    block by block (numpy composition of the E4M3 and E8M0 decodes)."""
    B, H, nk, d = 1, 3, 45, 64
    rng = np.random.default_rng(51)
    q = rng.standard_normal((B, H, 1, d))
    k8, ks = _mx_codes(B * H * nk, d, 52)
    v8, vs = _mx_codes(B * H * nk, d, 53)
    k = (orc.decode_e4m3(k8) * np.repeat(2.0 ** (ks.astype(np.float64) - 127), 32, axis=1))
    v = (orc.decode_e4m3(v8) * np.repeat(2.0 ** (vs.astype(np.float64) - 127), 32, axis=1))
    shp, sshp = (B, H, nk, d), (B, H, nk, d // 32)
    o1, l1 = orc.attention_mx(q, k8.reshape(shp), ks.reshape(sshp), v8.reshape(shp),
                              vs.reshape(sshp), scale=0.2)
    o2, l2 = orc.attention(q, k.reshape(shp), v.reshape(shp), scale=0.2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # a bf16 query (bit patterns) is widened exactly, as attention() widens it
    import torch
    qb = torch.from_numpy(q).to(torch.bfloat16)
    bits = qb.view(torch.int16).numpy().view(np.uint16)
    o3, l3 = orc.attention_mx(bits, k8.reshape(shp), ks.reshape(sshp), v8.reshape(shp),
                              vs.reshape(sshp), scale=0.2)
    o4, l4 = orc.attention(qb.to(torch.float64).numpy(), k.reshape(shp), v.reshape(shp), scale=0.2)
    assert np.array_equal(o3, o4) and np.array_equal(l3, l4)


ALL_PINS = [
    pin_exercise8_online_softmax,
    pin_rows_sum_to_one,
    pin_q_zero,
    pin_one_hot_dominant,
    pin_causal_row0,
    pin_v_affine,
    pin_key_permutation,
    pin_scale_is_applied,
    pin_blocked_equals_unblocked,
    pin_merge_rule,
    pin_bruteforce_fsum,
    pin_causal_chunk_is_suffix,
    pin_torch_crosscheck,
    pin_bf16_widening,
    pin_rows_equal_full,
    pin_bwd_finite_differences,
    pin_bwd_torch_autograd,
    pin_bwd_exercise9_identity,
    pin_bwd_invariants,
    pin_bwd_rows_and_keys_equal_full,
    pin_e4m3_spec_values,
    pin_e4m3_torch,
    pin_fp8_attention_dequantised,
    pin_fp8_descales,
    pin_e8m0_spec_values,
    pin_e8m0_torch,
    pin_mx_block_layout,
    pin_mx_attention_dequantised,
]
