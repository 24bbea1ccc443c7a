"""The debug build (libgbattn_debug.so, GBATTN_DEBUG): every kernel checks the
index of each direct global-memory access against its buffer and reports an
out-of-range one (ATTN_ERR_OUT_OF_RANGE) instead of making the access.  With
no memory checker on this machine's GPUs, it is the library's stand-in.

In a fresh process with GBATTN_DEBUG=1 every entry point runs on small shapes
(both head sizes, causal and not, ragged, FP8, bf16 and MXFP8 decode, split
and single-split decode, the no-allocation decode, merge, backward) with
NaN-filled outputs; each result is checked against the fp64 oracle and the
device error word must stay clear: no false alarm from the checks, and the
debug kernels compute what the release ones do.  Then the bounds self-test
(a kernel whose check fails on purpose, making no access) must be reported
once and cleared.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent(r"""
    import ctypes, numpy as np, torch
    import oracle
    from attention_flashattention_fwd_gb300 import binding
    from attention_flashattention_fwd_gb300.inputs import (bf16_bits, make_qkv, make_qkv_fp8,
                                                           make_qkv_mx)
    lib = binding.load()
    assert binding.LIB_PATH.endswith("libgbattn_debug.so") and lib.attn_debug_build() == 1
    dev = torch.device("cuda:0")

    def nan(shape, dtype):
        return torch.full(shape, float("nan"), dtype=dtype, device=dev)

    def close(o, lse, ro, rl, what, omax=2e-2):
        e = np.abs(o.float().cpu().numpy() - ro)
        el = np.abs(lse.cpu().numpy() - rl)
        assert np.isfinite(e).all() and e.max() <= omax and el.max() <= 2e-3, (what, e.max(), el.max())

    for (B, H, Nq, Nk, d, c) in [(1, 2, 300, 300, 64, True), (1, 2, 200, 513, 128, True),
                                 (2, 1, 256, 384, 128, False), (1, 77, 512, 512, 128, False)]:
        q, k, v = make_qkv(B, H, Nq, Nk, d, seed=5 + Nq, device=dev)
        o, lse = nan((B, H, Nq, d), torch.bfloat16), nan((B, H, Nq), torch.float32)
        binding.attn_fwd(q, k, v, causal=c, out=o, lse=lse)
        ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=c)
        close(o, lse, ro, rl, ("fwd", B, H, Nq, Nk, d, c))

    # the CTA-pair forward: bit-identical to attn_fwd; the pair product
    for (B, H, Nq, Nk, c) in [(1, 2, 1000, 1300, True), (2, 3, 300, 513, False)]:
        q, k, v = make_qkv(B, H, Nq, Nk, 128, seed=7 + Nq, device=dev)
        o2, l2 = nan((B, H, Nq, 128), torch.bfloat16), nan((B, H, Nq), torch.float32)
        binding.attn_fwd_cta_pair(q, k, v, causal=c, out=o2, lse=l2)
        o1, l1 = binding.attn_fwd(q, k, v, causal=c)
        assert torch.equal(o1, o2) and torch.equal(l1, l2), ("pair", B, H, Nq, Nk, c)
    a = torch.randn(256, 64, device=dev).to(torch.bfloat16)
    bm = torch.randn(128, 64, device=dev).to(torch.bfloat16)
    d = binding.attn_pair_product(a, bm).double().cpu()
    ref = a.double().cpu() @ bm.double().cpu().T
    assert (d - ref).abs().max().item() <= 1e-3 * max(1.0, ref.abs().max().item())

    # ragged: sequence lengths; rows past them stay untouched
    B, H, Nq, Nk, d = 2, 2, 256, 300, 128
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed=9, device=dev)
    sq = torch.tensor([200, 256], dtype=torch.int32, device=dev)
    sk = torch.tensor([250, 300], dtype=torch.int32, device=dev)
    o, lse = binding.attn_fwd_ragged(q, k, v, seqlens_q=sq, seqlens_k=sk, causal=True)
    for b, (nq, nk) in enumerate(((200, 250), (256, 300))):
        ro, rl = oracle.attention(bf16_bits(q[b:b + 1, :, :nq]), bf16_bits(k[b:b + 1, :, :nk]),
                                  bf16_bits(v[b:b + 1, :, :nk]), causal=True)
        close(o[b:b + 1, :, :nq], lse[b:b + 1, :, :nq], ro, rl, ("ragged", b))

    # FP8 forward
    q8, k8, vt8, ds = make_qkv_fp8(1, 2, 200, 208, 128, seed=12, device=dev)
    o, lse = binding.attn_fwd_fp8(q8, k8, vt8, *ds, causal=True)
    ro, rl = oracle.attention_fp8(*(t.cpu().numpy() for t in (q8, k8, vt8)), causal=True,
                                  descale_q=ds[0], descale_k=ds[1], descale_v=ds[2])
    close(o, lse, ro, rl, "fp8", omax=0.2)

    # decode: several splits, one split; MXFP8; ragged; no allocation
    for (B, H, Nk, d) in [(2, 3, 3000, 64), (16, 32, 700, 128)]:
        q, k, v = make_qkv(B, H, 1, Nk, d, seed=21 + Nk, device=dev)
        o, lse = binding.attn_fwd_decode(q, k, v)
        ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v))
        close(o, lse, ro, rl, ("decode", B, H, Nk, d))
        q, k8, ks, v8, vs = make_qkv_mx(B, H, Nk, d, seed=22 + Nk, device=dev)
        o, lse = binding.attn_fwd_decode_mx(q, k8, ks, v8, vs)
        ro, rl = oracle.attention_mx(bf16_bits(q), *(t.cpu().numpy() for t in (k8, ks, v8, vs)))
        close(o, lse, ro, rl, ("decode mx", B, H, Nk, d))
    q, k, v = make_qkv(2, 2, 1, 1500, 128, seed=31, device=dev)
    sk = torch.tensor([1000, 1500], dtype=torch.int32, device=dev)
    o, lse = binding.attn_fwd_decode_ragged(q, k, v, seqlens_k=sk)
    for b, nk in enumerate((1000, 1500)):
        ro, rl = oracle.attention(bf16_bits(q[b:b + 1]), bf16_bits(k[b:b + 1, :, :nk]),
                                  bf16_bits(v[b:b + 1, :, :nk]))
        close(o[b:b + 1], lse[b:b + 1], ro, rl, ("decode ragged", b))
    fn = lib.attn_fwd_decode_no_alloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, P, P, I, I, I, I, F, P]
    q, k, v = make_qkv(4, 8, 1, 2048, 128, seed=33, device=dev)
    o, lse = nan((4, 8, 1, 128), torch.bfloat16), nan((4, 8, 1), torch.float32)
    st = fn(P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), P(o.data_ptr()),
            P(lse.data_ptr()), 4, 8, 2048, 128, 128 ** -0.5,
            P(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v))
    close(o, lse, ro, rl, "decode no-alloc")

    # merge of three key shards, and the backward
    q, k, v = make_qkv(1, 2, 64, 300, 128, seed=41, device=dev)
    parts = [binding.attn_fwd(q, k[:, :, a:b].contiguous(), v[:, :, a:b].contiguous())
             for a, b in ((0, 100), (100, 220), (220, 300))]
    o, lse = binding.attn_merge(torch.stack([p[0] for p in parts]),
                                torch.stack([p[1] for p in parts]))
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v))
    close(o, lse, ro, rl, "merge")
    q, k, v = make_qkv(1, 2, 300, 300, 64, seed=51, device=dev)
    dout = torch.randn(q.shape, generator=torch.Generator(device=dev).manual_seed(52),
                       device=dev).to(torch.bfloat16)
    o, lse = binding.attn_fwd(q, k, v, causal=True)
    grads = binding.attn_bwd(q, k, v, o, lse, dout, causal=True)
    refs = oracle.attention_bwd(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(dout),
                                causal=True)
    for name, got, ref in zip(("dq", "dk", "dv"), grads, refs):
        got = got.float().cpu().numpy()
        rms = float(np.sqrt(np.mean(ref * ref)))
        assert (np.abs(got - ref) - 2.0 ** -8 * np.abs(ref)).max() <= 2.0 ** -3 * rms, name

    assert binding.device_error() == 0, "a debug kernel reported an out-of-range index"
    # the check itself reports, once, and the context stays usable
    assert lib.attn_selftest_bounds(ctypes.c_void_p(0)) == 0
    assert binding.device_error() == 6  # ATTN_ERR_OUT_OF_RANGE
    assert binding.device_error() == 0
    print("debug build ok")
""")


def test_debug_build_computes_the_same_and_reports_nothing():
    env = dict(os.environ, GBATTN_DEBUG="1")
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "debug build ok" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])
