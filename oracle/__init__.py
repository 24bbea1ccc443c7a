"""fp64 CPU oracle for scaled-dot-product attention (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It is a thin ctypes wrapper around the
plain C implementation in ``attn_oracle.c`` (built by ``oracle/build.py``); it
shares nothing with the CUDA library.

Functions (each follows a passage of the lecture pages, cited in the C file):

* :func:`attention` -- naive attention, S = scale Q K^T, safe softmax, O = P V,
  lse = m + ln l (CS149 L9 concept 8; PDC L4 section 4.14; CS336 L5 8.1/8.3).
* :func:`attention_rows` -- the same on a list of (bh, i) rows.
* :func:`online_softmax_blocks` -- per-block online softmax (CS336 L5 8.2).
* :func:`softmax_merge` -- two-block merge rule (CS149 L9 concept 9).
* :func:`attention_blocked` -- tiled FlashAttention forward (CS336 L5 8.3).
* :func:`attention_bwd` -- gradients dQ, dK, dV for an upstream dO (CS336 L5
  8.4), with D_i taken from its definition sum_j P_ij dP_ij.
* :func:`attention_bwd_dq_rows`, :func:`attention_bwd_dkdv_keys` -- the same on
  listed query rows / key rows, for sampled checks of large problems.
* :func:`decode_e4m3` -- value of FP8 E4M3 codes times a per-tensor descale
  (CS336 L5 6.2; PDC L7 section 7.14).
* :func:`fp8_operands` / :func:`attention_fp8` -- attention of per-tensor
  scaled FP8 operands: decode, then the naive attention above.
* :func:`decode_mx` / :func:`attention_mx` -- MXFP8 (E4M3 elements, one E8M0
  scale per 32 consecutive elements of a row; PDC L7 section 7.14, OCP MX
  v1.0) keys and values: decode, then the naive attention above.

Inputs are numpy arrays, either float64 or bfloat16 bit patterns (uint16).
"""
import ctypes

import numpy as np

from . import build as _build

_lib = None


def _declare(lib):
    """Attach the C signatures to a loaded oracle library."""
    P = ctypes.c_void_p
    L = ctypes.c_long
    D = ctypes.c_double
    I = ctypes.c_int
    lib.oracle_attention.argtypes = [P, P, P, I, P, P, L, L, L, L, L, I, D]
    lib.oracle_attention.restype = I
    lib.oracle_attention_rows.argtypes = [P, P, P, I, P, L, P, P, L, L, L, L, L, I, D]
    lib.oracle_attention_rows.restype = I
    lib.oracle_online_softmax_blocks.argtypes = [P, L, P, L, P, P]
    lib.oracle_online_softmax_blocks.restype = I
    lib.oracle_softmax_merge.argtypes = [D, D, P, D, D, P, L, P, P, P]
    lib.oracle_softmax_merge.restype = None
    lib.oracle_attention_blocked.argtypes = [P, P, P, P, P, L, L, L, L, L, I, D, L, L]
    lib.oracle_attention_blocked.restype = I
    lib.oracle_attention_bwd.argtypes = [P, P, P, P, I, P, P, P, L, L, L, L, L, I, D]
    lib.oracle_attention_bwd.restype = I
    lib.oracle_attention_bwd_dq_rows.argtypes = [P, P, P, P, I, P, L, P, P, L, L, L, L, L, I, D]
    lib.oracle_attention_bwd_dq_rows.restype = I
    lib.oracle_attention_bwd_dkdv_keys.argtypes = [P, P, P, P, I, P, L, P, P, L, L, L, L, L, I, D]
    lib.oracle_attention_bwd_dkdv_keys.restype = I
    lib.oracle_decode_e4m3.argtypes = [P, P, L, D]
    lib.oracle_decode_e4m3.restype = None
    lib.oracle_decode_mx.argtypes = [P, P, P, L, L, L]
    lib.oracle_decode_mx.restype = I
    lib.oracle_widen_bf16.argtypes = [P, P, L]
    lib.oracle_widen_bf16.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = I
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _declare(ctypes.CDLL(_build.build()))
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _inputs(*xs):
    xs = tuple(np.ascontiguousarray(x) for x in xs)
    if all(x.dtype == np.uint16 for x in xs):
        return xs + (1,)
    return tuple(np.ascontiguousarray(x, dtype=np.float64) for x in xs) + (0,)


def attention(q, k, v, causal=False, scale=None):
    """Naive fp64 attention.  q: [B,H,Nq,d], k/v: [B,H,Nk,d] (float64 or
    bf16 bits as uint16).  Returns (o float64 [B,H,Nq,d], lse float64 [B,H,Nq])."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    q, k, v, is_bf16 = _inputs(q, k, v)
    o = np.empty((B, H, Nq, d), np.float64)
    lse = np.empty((B, H, Nq), np.float64)
    rc = _load().oracle_attention(_ptr(q), _ptr(k), _ptr(v), is_bf16, _ptr(o), _ptr(lse),
                                  B, H, Nq, Nk, d, int(bool(causal)), float(scale))
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    return o, lse


def attention_rows(q, k, v, rows, causal=False, scale=None):
    """Rows ``rows`` (int array [n, 2] of (bh, i)) of naive attention.
    Returns (o [n, d], lse [n])."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    q, k, v, is_bf16 = _inputs(q, k, v)
    rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 2)
    n = rows.shape[0]
    o = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    rc = _load().oracle_attention_rows(_ptr(q), _ptr(k), _ptr(v), is_bf16, _ptr(rows), n,
                                       _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                                       int(bool(causal)), float(scale))
    if rc != 0:
        raise ValueError("oracle_attention_rows rejected its arguments")
    return o, lse


def online_softmax_blocks(x, ends):
    """Running (m, l) after each block of x; ``ends`` are exclusive block ends."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    ends = np.ascontiguousarray(ends, dtype=np.int64)
    m = np.empty(len(ends), np.float64)
    l = np.empty(len(ends), np.float64)
    rc = _load().oracle_online_softmax_blocks(_ptr(x), x.size, _ptr(ends), ends.size,
                                              _ptr(m), _ptr(l))
    if rc != 0:
        raise ValueError("bad block list")
    return m, l


def softmax_merge(m1, l1, o1, m2, l2, o2):
    """Merge two blocks' (m, l, normalised o).  Returns (m, l, o)."""
    o1 = np.ascontiguousarray(o1, dtype=np.float64)
    o2 = np.ascontiguousarray(o2, dtype=np.float64)
    o = np.empty_like(o1)
    m = ctypes.c_double()
    l = ctypes.c_double()
    _load().oracle_softmax_merge(float(m1), float(l1), _ptr(o1), float(m2), float(l2),
                                 _ptr(o2), o1.size, ctypes.byref(m), ctypes.byref(l), _ptr(o))
    return m.value, l.value, o


def attention_blocked(q, k, v, causal=False, scale=None, block_q=128, block_k=128):
    """Tiled FlashAttention forward in fp64 (float64 inputs only)."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    q, k, v = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v))
    o = np.empty((B, H, Nq, d), np.float64)
    lse = np.empty((B, H, Nq), np.float64)
    rc = _load().oracle_attention_blocked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                          B, H, Nq, Nk, d, int(bool(causal)), float(scale),
                                          int(block_q), int(block_k))
    if rc != 0:
        raise ValueError("oracle_attention_blocked rejected its arguments")
    return o, lse


def threads_used() -> int:
    """Number of threads the oracle's row loops run on (1 without OpenMP)."""
    return int(_load().oracle_num_threads())


def attention_bwd(q, k, v, dout, causal=False, scale=None):
    """Gradients of naive attention for the upstream gradient ``dout``
    ([B,H,Nq,d]).  Returns (dq [B,H,Nq,d], dk, dv [B,H,Nk,d]) in float64."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    q, k, v, dout, is_bf16 = _inputs(q, k, v, dout)
    dq = np.empty((B, H, Nq, d), np.float64)
    dk = np.empty((B, H, Nk, d), np.float64)
    dv = np.empty((B, H, Nk, d), np.float64)
    rc = _load().oracle_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), is_bf16, _ptr(dq),
                                      _ptr(dk), _ptr(dv), B, H, Nq, Nk, d,
                                      int(bool(causal)), float(scale))
    if rc != 0:
        raise ValueError("oracle_attention_bwd rejected its arguments")
    return dq, dk, dv


def attention_bwd_dq_rows(q, k, v, dout, rows, causal=False, scale=None):
    """dQ on rows ``rows`` ([n, 2] of (bh, i)).  Returns (dq [n, d], D [n])
    with D_i = sum_j P_ij dP_ij."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    q, k, v, dout, is_bf16 = _inputs(q, k, v, dout)
    rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 2)
    n = rows.shape[0]
    dq = np.empty((n, d), np.float64)
    D = np.empty((n,), np.float64)
    rc = _load().oracle_attention_bwd_dq_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), is_bf16,
                                              _ptr(rows), n, _ptr(dq), _ptr(D), B, H, Nq, Nk, d,
                                              int(bool(causal)), float(scale))
    if rc != 0:
        raise ValueError("oracle_attention_bwd_dq_rows rejected its arguments")
    return dq, D


def attention_bwd_dkdv_keys(q, k, v, dout, keys, causal=False, scale=None):
    """dK and dV on key rows ``keys`` ([n, 2] of (bh, j)).  Returns (dk, dv),
    each [n, d]."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    q, k, v, dout, is_bf16 = _inputs(q, k, v, dout)
    keys = np.ascontiguousarray(keys, dtype=np.int64).reshape(-1, 2)
    n = keys.shape[0]
    dk = np.empty((n, d), np.float64)
    dv = np.empty((n, d), np.float64)
    rc = _load().oracle_attention_bwd_dkdv_keys(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), is_bf16,
                                                _ptr(keys), n, _ptr(dk), _ptr(dv), B, H, Nq, Nk,
                                                d, int(bool(causal)), float(scale))
    if rc != 0:
        raise ValueError("oracle_attention_bwd_dkdv_keys rejected its arguments")
    return dk, dv


def decode_e4m3(codes, descale=1.0):
    """float64 values descale * E4M3(codes) of a uint8 array (same shape)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, np.float64)
    _load().oracle_decode_e4m3(_ptr(codes), _ptr(out), codes.size, float(descale))
    return out


def fp8_operands(q8, k8, vt8, descale_q=1.0, descale_k=1.0, descale_v=1.0):
    """float64 Q, K, V of FP8 operands: q8 [B,H,Nq,d], k8 [B,H,Nk,d] and the
    value tensor given transposed, vt8 [B,H,d,Nk] (uint8 E4M3 codes).  V is
    returned in the [B,H,Nk,d] layout of :func:`attention`."""
    q = decode_e4m3(q8, descale_q)
    k = decode_e4m3(k8, descale_k)
    v = np.ascontiguousarray(np.swapaxes(decode_e4m3(vt8, descale_v), 2, 3))
    return q, k, v


def attention_fp8(q8, k8, vt8, causal=False, scale=None, descale_q=1.0, descale_k=1.0,
                  descale_v=1.0):
    """Attention of per-tensor scaled FP8 operands (see :func:`fp8_operands`):
    S = scale (descale_q Q8)(descale_k K8)^T, O = softmax(S) (descale_v V8).
    Returns (o [B,H,Nq,d], lse [B,H,Nq]) in float64."""
    q, k, v = fp8_operands(q8, k8, vt8, descale_q, descale_k, descale_v)
    return attention(q, k, v, causal=causal, scale=scale)


def decode_mx(codes, scales, block=32):
    """float64 values of MXFP8 data: codes uint8 [..., d] (E4M3), scales uint8
    [..., d / block] (E8M0), element c of a row scaled by its block's scale."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    d = codes.shape[-1]
    if d % block or scales.shape != codes.shape[:-1] + (d // block,):
        raise ValueError("scales must be [..., d / block]")
    out = np.empty(codes.shape, np.float64)
    rows = codes.size // d if d else 0
    if _load().oracle_decode_mx(_ptr(codes), _ptr(scales), _ptr(out), rows, d, block) != 0:
        raise ValueError("oracle_decode_mx rejected its arguments")
    return out


def attention_mx(q, k8, k_scale, v8, v_scale, causal=False, scale=None, block=32):
    """Attention with MXFP8 keys and values (see :func:`decode_mx`): q [B,H,Nq,d]
    (float64 or bf16 bits), k8 / v8 [B,H,Nk,d] E4M3 codes, k_scale / v_scale
    [B,H,Nk,d/32] E8M0 codes.  Returns (o, lse) in float64."""
    q = np.ascontiguousarray(q)
    if q.dtype == np.uint16:  # bf16 bits: widen exactly, like the other inputs
        qd = np.empty(q.shape, np.float64)
        _load().oracle_widen_bf16(_ptr(q), _ptr(qd), q.size)
        q = qd
    k = decode_mx(k8, k_scale, block)
    v = decode_mx(v8, v_scale, block)
    return attention(q, k, v, causal=causal, scale=scale)
