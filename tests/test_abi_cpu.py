"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

from attention_flashattention_fwd_gb300 import binding, build_lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "gbattn.h")
OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[a-z_ ]+[ *]+\**(attn_[a-z0-9_]+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("attn_fwd", "attn_fwd_decode", "attn_fwd_decode_workspace_bytes",
              "attn_fwd_from_host", "attn_status_string", "attn_device_error", "attn_version"):
        assert n in names, names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libgbattn.so does not export {name}"


def test_version_and_status_strings(lib):
    assert lib.attn_version() >= 100
    for st in range(7):
        assert binding.status_string(st).startswith("ATTN_")
    assert binding.status_string(99) == "unknown status"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, Nq=128, Nk=128, d=64,
        causal=0, scale=0.125):
    P = ctypes.c_void_p
    return lib.attn_fwd(P(q), P(k), P(v), P(o), P(lse), B, H, Nq, Nk, d, causal, scale, P(0))


@pytest.mark.parametrize("kw,expect", [
    (dict(q=0), INVALID), (dict(k=0), INVALID), (dict(v=0), INVALID), (dict(o=0), INVALID),
    (dict(lse=0), INVALID), (dict(B=0), INVALID), (dict(H=-1), INVALID), (dict(Nq=0), INVALID),
    (dict(Nk=0), INVALID), (dict(scale=float("nan")), INVALID), (dict(scale=float("inf")), INVALID),
    (dict(scale=0.0), INVALID), (dict(scale=-1.0), INVALID), (dict(causal=2), INVALID),
    (dict(d=96), UNSUPPORTED), (dict(d=256), UNSUPPORTED), (dict(d=0), UNSUPPORTED),
    (dict(causal=1, Nq=256, Nk=128), UNSUPPORTED),  # rows with no visible key
    (dict(Nq=1 << 30, Nk=1 << 30), UNSUPPORTED),     # query positions beyond int32
    (dict(B=1 << 20, H=1 << 12), UNSUPPORTED),
    (dict(q=FAKE + 8), MISALIGNED), (dict(o=FAKE + 2), MISALIGNED), (dict(lse=FAKE + 4), MISALIGNED),
])
def test_attn_fwd_rejects_before_launch(lib, kw, expect):
    assert fwd(lib, **kw) == expect


def test_decode_workspace_bytes_is_host_arithmetic(lib):
    # room for the largest plan of any device: one split per 512 keys, d + 1
    # floats per (head, split); 2048 heads of 8192 keys -> 16 splits each
    assert lib.attn_fwd_decode_workspace_bytes(64, 32, 8192, 128) == 2048 * 16 * (128 + 1) * 4
    assert lib.attn_fwd_decode_workspace_bytes(1, 1, 8192, 128) == 16 * (128 + 1) * 4
    assert lib.attn_fwd_decode_workspace_bytes(1, 1, 8193, 64) == 17 * (64 + 1) * 4
    # at most 64 splits
    assert lib.attn_fwd_decode_workspace_bytes(2, 3, 1 << 20, 128) == 6 * 64 * (128 + 1) * 4
    # a single split needs no workspace
    assert lib.attn_fwd_decode_workspace_bytes(64, 32, 300, 64) == 0
    assert lib.attn_fwd_decode_workspace_bytes(1, 1, 0, 64) == 0
    assert lib.attn_fwd_decode_workspace_bytes(1, 1, 100, 96) == 0


def test_decode_rejects_before_launch(lib):
    P = ctypes.c_void_p
    need = lib.attn_fwd_decode_workspace_bytes(1, 1, 8192, 128)

    def dec(q=FAKE, ws=FAKE, ws_bytes=need, d=128, scale=0.1, Nk=8192):
        return lib.attn_fwd_decode(P(q), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 1, Nk, d, scale,
                                   P(ws), ws_bytes, P(0))

    assert dec(q=0) == INVALID
    assert dec(ws=0) == INVALID
    assert dec(ws_bytes=need - 1) == INVALID
    assert dec(scale=-1.0) == INVALID
    assert dec(d=80) == UNSUPPORTED
    assert dec(Nk=0) == INVALID
    assert dec(q=FAKE + 8) == MISALIGNED
    assert dec(ws=FAKE + 4) == MISALIGNED


def test_decode_mx_rejects_before_launch(lib):
    P = ctypes.c_void_p
    lib.attn_fwd_decode_mx.argtypes = [P] * 7 + [ctypes.c_int] * 4 + [ctypes.c_float, P,
                                                                      ctypes.c_size_t, P]
    lib.attn_fwd_decode_mx.restype = ctypes.c_int
    need = lib.attn_fwd_decode_workspace_bytes(1, 1, 8192, 128)

    def dec(ks=FAKE, vs=FAKE, k8=FAKE, d=128, Nk=8192, ws_bytes=need):
        return lib.attn_fwd_decode_mx(P(FAKE), P(k8), P(ks), P(FAKE), P(vs), P(FAKE), P(FAKE),
                                      1, 1, Nk, d, 0.1, P(FAKE), ws_bytes, P(0))

    assert dec(ks=0) == INVALID
    assert dec(vs=0) == INVALID
    assert dec(ws_bytes=need - 1) == INVALID
    assert dec(d=96) == UNSUPPORTED
    assert dec(k8=FAKE + 8) == MISALIGNED
    assert dec(ks=FAKE + 1, vs=FAKE + 3, k8=FAKE + 8) == MISALIGNED  # scales: any alignment


def test_from_host_rejects_before_launch(lib):
    P = ctypes.c_void_p
    args = [P(FAKE)] * 10
    args[7] = P(0)  # dv missing
    assert lib.attn_fwd_from_host(*args, 1, 1, 128, 128, 64, 0, 0.125, P(0)) == INVALID
    args = [P(FAKE)] * 10
    args[6] = P(FAKE + 8)  # dk misaligned
    assert lib.attn_fwd_from_host(*args, 1, 1, 128, 128, 64, 0, 0.125, P(0)) == MISALIGNED
    args = [P(FAKE)] * 10
    assert lib.attn_fwd_from_host(*args, 1, 1, 128, 128, 72, 0, 0.125, P(0)) == UNSUPPORTED


def test_bwd_workspace_bytes_is_host_arithmetic(lib):
    lib.attn_bwd_workspace_bytes.argtypes = [ctypes.c_int] * 5
    lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    # dQ accumulator (d floats) plus two floats per row, rows padded to 128
    assert lib.attn_bwd_workspace_bytes(2, 16, 4096, 4096, 128) == 32 * 4096 * 130 * 4
    assert lib.attn_bwd_workspace_bytes(1, 1, 77, 77, 64) == 128 * 66 * 4
    assert lib.attn_bwd_workspace_bytes(1, 1, 77, 77, 96) == 0
    assert lib.attn_bwd_workspace_bytes(1, 0, 77, 77, 64) == 0


def test_bwd_rejects_before_launch(lib):
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_bwd.argtypes = [P] * 9 + [I, I, I, I, I, I, F, P, S, P]
    lib.attn_bwd.restype = I
    need = 128 * 66 * 4

    def bwd(ptrs=None, Nq=128, Nk=128, d=64, causal=0, scale=0.125, ws=FAKE, ws_bytes=need):
        p = [FAKE] * 9 if ptrs is None else ptrs
        return lib.attn_bwd(*[P(x) for x in p], 1, 1, Nq, Nk, d, causal, scale, P(ws), ws_bytes,
                            P(0))

    for i in range(9):  # q, k, v, o, dout, lse, dq, dk, dv
        ptrs = [FAKE] * 9
        ptrs[i] = 0
        assert bwd(ptrs) == INVALID, i
        ptrs[i] = FAKE + 8
        assert bwd(ptrs) == MISALIGNED, i
    assert bwd(ws=0) == INVALID
    assert bwd(ws_bytes=need - 1) == INVALID
    assert bwd(ws=FAKE + 4) == MISALIGNED
    assert bwd(d=80) == UNSUPPORTED
    assert bwd(causal=1, Nq=256, Nk=128, ws_bytes=1 << 20) == UNSUPPORTED
    assert bwd(scale=float("nan")) == INVALID


def test_merge_rejects_before_launch(lib):
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.attn_merge.argtypes = [P, P, I, P, P, I, I, I, I, P]
    lib.attn_merge.restype = I

    def merge(op=FAKE, lp=FAKE, n=2, o=FAKE, lse=FAKE, B=1, H=1, Nq=4, d=64):
        return lib.attn_merge(P(op), P(lp), n, P(o), P(lse), B, H, Nq, d, P(0))

    assert merge(op=0) == INVALID and merge(lp=0) == INVALID and merge(o=0) == INVALID
    assert merge(lse=0) == INVALID and merge(n=0) == INVALID and merge(Nq=0) == INVALID
    assert merge(d=96) == UNSUPPORTED
    assert merge(op=FAKE + 8) == MISALIGNED and merge(lse=FAKE + 4) == MISALIGNED


def test_ragged_entry_points_reject_before_launch(lib):
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd_ragged.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, P]
    lib.attn_fwd_ragged.restype = I
    lib.attn_fwd_decode_ragged.argtypes = [P, P, P, P, P, P, I, I, I, I, F, P, S, P]
    lib.attn_fwd_decode_ragged.restype = I

    def rag(sq=FAKE, sk=FAKE, q=FAKE, d=64, causal=0, Nq=128, Nk=128):
        return lib.attn_fwd_ragged(P(q), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(sq), P(sk), 2, 1,
                                   Nq, Nk, d, causal, 0.125, P(0))

    assert rag(sq=FAKE + 2) == MISALIGNED and rag(sk=FAKE + 1) == MISALIGNED
    assert rag(q=0) == INVALID and rag(d=80) == UNSUPPORTED
    assert rag(causal=1, Nq=256, Nk=128) == UNSUPPORTED
    need = lib.attn_fwd_decode_workspace_bytes(1, 1, 8192, 128)
    assert lib.attn_fwd_decode_ragged(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE + 2), 1, 1,
                                      8192, 128, 0.1, P(FAKE), need, P(0)) == MISALIGNED
    assert lib.attn_fwd_decode_ragged(P(0), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 1,
                                      8192, 128, 0.1, P(FAKE), need, P(0)) == INVALID


def test_fp8_entry_point_rejects_before_launch(lib):
    P = ctypes.c_void_p

    def f8(q=FAKE, vt=FAKE, o=FAKE, d=128, Nq=128, Nk=128, causal=0, scale=0.1, dq=0.01,
           dk=0.01, dv=0.01):
        return lib.attn_fwd_fp8(P(q), P(FAKE), P(vt), P(o), P(FAKE), 1, 2, Nq, Nk, d, causal,
                                scale, dq, dk, dv, P(0))

    assert f8(q=0) == INVALID and f8(vt=0) == INVALID and f8(Nq=0) == INVALID
    assert f8(dq=0.0) == INVALID and f8(dk=-1.0) == INVALID and f8(dv=float("nan")) == INVALID
    assert f8(dv=float("inf")) == INVALID and f8(scale=0.0) == INVALID
    assert f8(scale=1e30, dq=1e10, dk=1e10) == INVALID    # folded score scale overflows fp32
    assert f8(d=64) == UNSUPPORTED and f8(d=96) == UNSUPPORTED
    assert f8(Nk=120) == UNSUPPORTED                        # V^T rows of 120 bytes
    assert f8(causal=1, Nq=256, Nk=128) == UNSUPPORTED
    assert f8(vt=FAKE + 8) == MISALIGNED and f8(o=FAKE + 2) == MISALIGNED


def test_release_and_debug_builds_identify_themselves(lib):
    """attn_debug_build tells the builds apart; the release build has no index
    checks, so its bounds self-test is refused before any CUDA call."""
    import ctypes as C
    import os
    from attention_flashattention_fwd_gb300 import build_lib
    lib.attn_debug_build.restype = C.c_int
    lib.attn_selftest_bounds.argtypes = [C.c_void_p]
    lib.attn_selftest_bounds.restype = C.c_int
    if not binding.LIB_PATH.endswith("_debug.so"):
        assert lib.attn_debug_build() == 0
        assert lib.attn_selftest_bounds(C.c_void_p(0)) == UNSUPPORTED
    build_lib.build(debug=True)
    dbg = C.CDLL(build_lib.LIB_DEBUG)
    dbg.attn_debug_build.restype = C.c_int
    assert dbg.attn_debug_build() == 1
    for name in declared_functions():
        assert hasattr(dbg, name), f"libgbattn_debug.so does not export {name}"


def test_pair_entry_points_reject_before_launch(lib):
    """The CTA-pair product and the issue-rate measurement check their
    arguments on the host before any CUDA call."""
    P = ctypes.c_void_p
    assert lib.attn_pair_product(P(0), P(FAKE), P(FAKE), P(0)) == INVALID
    assert lib.attn_pair_product(P(FAKE), P(FAKE), P(0), P(0)) == INVALID
    assert lib.attn_pair_product(P(FAKE + 4), P(FAKE), P(FAKE), P(0)) == MISALIGNED
    ms = ctypes.c_float()

    def rate(form=1, issuer=1, busy=0, waits=0, steps=16, reps=1, out=True):
        return lib.attn_bench_mma_rate(form, issuer, busy, waits, steps, reps,
                                       ctypes.byref(ms) if out else P(0), P(0), P(0), P(0))

    assert rate(form=0) == INVALID and rate(form=3) == INVALID
    assert rate(issuer=2) == INVALID and rate(issuer=-1) == INVALID
    assert rate(busy=2) == INVALID and rate(waits=-1) == INVALID
    assert rate(steps=0) == INVALID and rate(steps=(1 << 16) + 1) == INVALID
    assert rate(reps=0) == INVALID and rate(out=False) == INVALID


def test_cta_pair_entry_rejects_before_launch(lib):
    """attn_fwd_cta_pair validates like attn_fwd and takes d = 128 only."""
    P = ctypes.c_void_p

    def pair(q=FAKE, o=FAKE, d=128, Nq=128, Nk=128, causal=0, scale=0.1):
        return lib.attn_fwd_cta_pair(P(q), P(FAKE), P(FAKE), P(o), P(FAKE), 1, 2, Nq, Nk, d, causal,
                                     scale, P(0))

    assert pair(q=0) == INVALID and pair(Nq=0) == INVALID and pair(scale=0.0) == INVALID
    assert pair(d=64) == UNSUPPORTED and pair(d=96) == UNSUPPORTED
    assert pair(causal=1, Nq=256, Nk=128) == UNSUPPORTED
    assert pair(o=FAKE + 2) == MISALIGNED
