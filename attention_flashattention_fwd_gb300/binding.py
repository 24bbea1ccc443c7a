"""ctypes binding of ``libgbattn.so`` (the C ABI in ``include/gbattn.h``).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their pointers and the current CUDA stream are handed to the C
entry points of the same names, and a non-zero status is raised as
:class:`GbattnError`.  Every step of the computation runs in the CUDA kernels;
there is no fallback.  If the library has not been built, the first call
raises.
"""
import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# GBATTN_DEBUG=1 in the environment selects the debug build, whose kernels
# check every direct global-memory index (see include/gbattn.h)
LIB_PATH = os.path.join(_HERE, "libgbattn_debug.so" if os.environ.get("GBATTN_DEBUG") == "1"
                        else "libgbattn.so")

ATTN_OK = 0
_lib = None
_lib_lock = threading.Lock()


class GbattnError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def load():
    """Load the CUDA library (raises if it is missing).  Safe to call from
    several threads: the first caller configures it under a lock."""
    global _lib
    if _lib is not None:
        return _lib
    with _lib_lock:
        if _lib is None:
            _lib = _configure()
    return _lib


def _configure():
    """dlopen the library and declare every entry point's argument types."""
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; "
            f"g.build()\"` (or attention_flashattention_fwd_gb300/build_lib.py)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P]
    lib.attn_fwd.restype = I
    lib.attn_fwd_cta_pair.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P]
    lib.attn_fwd_cta_pair.restype = I
    lib.attn_fwd_fp8.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, F, F, F, P]
    lib.attn_fwd_fp8.restype = I
    lib.attn_fwd_decode_workspace_bytes.argtypes = [I, I, I, I]
    lib.attn_fwd_decode_workspace_bytes.restype = S
    lib.attn_fwd_decode.argtypes = [P, P, P, P, P, I, I, I, I, F, P, S, P]
    lib.attn_fwd_decode.restype = I
    lib.attn_fwd_from_host.argtypes = [P] * 10 + [I, I, I, I, I, I, F, P]
    lib.attn_fwd_from_host.restype = I
    lib.attn_bwd_workspace_bytes.argtypes = [I, I, I, I, I]
    lib.attn_bwd_workspace_bytes.restype = S
    lib.attn_bwd.argtypes = [P] * 9 + [I, I, I, I, I, I, F, P, S, P]
    lib.attn_bwd.restype = I
    lib.attn_fwd_ragged.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, P]
    lib.attn_fwd_ragged.restype = I
    lib.attn_fwd_decode_mx.argtypes = [P, P, P, P, P, P, P, I, I, I, I, F, P, S, P]
    lib.attn_fwd_decode_mx.restype = I
    lib.attn_fwd_decode_ragged.argtypes = [P, P, P, P, P, P, I, I, I, I, F, P, S, P]
    lib.attn_fwd_decode_ragged.restype = I
    lib.attn_merge.argtypes = [P, P, I, P, P, I, I, I, I, P]
    lib.attn_merge.restype = I
    lib.attn_status_string.argtypes = [I]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_device_error.argtypes = []
    lib.attn_device_error.restype = I
    lib.attn_selftest_timeout.argtypes = [P]
    lib.attn_selftest_timeout.restype = I
    lib.attn_version.argtypes = []
    lib.attn_version.restype = I
    lib.attn_selftest_bounds.argtypes = [P]
    lib.attn_selftest_bounds.restype = I
    lib.attn_debug_build.argtypes = []
    lib.attn_debug_build.restype = I
    lib.attn_pair_product.argtypes = [P, P, P, P]
    lib.attn_pair_product.restype = I
    lib.attn_bench_mma_rate.argtypes = [I, I, I, I, I, I, P, P, P, P]
    lib.attn_bench_mma_rate.restype = I
    return lib


def status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def _check(status, where):
    if status != ATTN_OK:
        raise GbattnError(status, where)


def _stream_ptr(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _out(t, shape, dtype, device, name):
    """An output buffer: a new one, or the caller's after checking that it is
    what the kernels will write (``shape`` elements of ``dtype`` at its
    address, on the inputs' device), since a mismatch would be written past."""
    shape = tuple(shape)
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    if (t.device != device or t.dtype != dtype or tuple(t.shape) != shape
            or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {shape} "
                         f"on {device}")
    return t


def _workspace(t, need, device):
    """A device workspace of at least ``need`` bytes (its size is checked by
    the C entry point): a new one, or the caller's on the right device."""
    if t is None:
        return torch.empty(need, dtype=torch.uint8, device=device) if need > 0 else None
    if t.device != device or not t.is_contiguous():
        raise ValueError(f"workspace must be a contiguous tensor on {device}")
    return t


def _on(device, stream):
    """The C entry points run on the current device: make the tensors' device
    current for the call, and refuse a stream of another device."""
    if stream is not None and stream.device != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return torch.cuda.device(device)


def _check_inputs(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k and v must be on the same device")
    B, H, Nq, d = q.shape
    if k.shape != (B, H, k.shape[2], d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, H, Nk, d] with q's B, H and d")
    return B, H, Nq, k.shape[2], d


def attention(q, k, v, causal=False, scale=None, stream=None):
    """O = softmax(scale Q K^T [+ causal mask]) V and the fp32 logsumexp,
    through ``attn_fwd_decode`` for a single query row and ``attn_fwd``
    otherwise.  A causal query block is the newest Nq tokens of the Nk-token
    sequence (query i sees keys j <= i + Nk - Nq), so one causal query row
    sees every key and is the decode step."""
    if q.dim() == 4 and q.shape[2] == 1:
        return attn_fwd_decode(q, k, v, scale=scale, stream=stream)
    return attn_fwd(q, k, v, causal=causal, scale=scale, stream=stream)


def attn_fwd(q, k, v, causal=False, scale=None, out=None, lse=None, stream=None):
    """The C entry point ``attn_fwd`` (prefill kernel) on torch tensors.

    q [B,H,Nq,d], k/v [B,H,Nk,d] bf16 CUDA tensors.  Returns
    (o bf16 [B,H,Nq,d], lse fp32 [B,H,Nq]).
    """
    B, H, Nq, Nk, d = _check_inputs(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = _out(out, (B, H, Nq, d), torch.bfloat16, q.device, "out")
    lse = _out(lse, (B, H, Nq), torch.float32, q.device, "lse")
    with _on(q.device, stream):
        st = load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nk, d,
                             int(bool(causal)), float(scale), _stream_ptr(stream))
    _check(st, "attn_fwd")
    return out, lse


def attn_fwd_cta_pair(q, k, v, causal=False, scale=None, out=None, lse=None, stream=None):
    """The C entry point ``attn_fwd_cta_pair``: attn_fwd with CTA-pair
    (cta_group::2) tensor-core products, d = 128; bit-identical output."""
    B, H, Nq, Nk, d = _check_inputs(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = _out(out, (B, H, Nq, d), torch.bfloat16, q.device, "out")
    lse = _out(lse, (B, H, Nq), torch.float32, q.device, "lse")
    with _on(q.device, stream):
        st = load().attn_fwd_cta_pair(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq,
                                      Nk, d, int(bool(causal)), float(scale), _stream_ptr(stream))
    _check(st, "attn_fwd_cta_pair")
    return out, lse


def attn_fwd_fp8(q8, k8, vt8, descale_q=1.0, descale_k=1.0, descale_v=1.0, causal=False,
                 scale=None, out=None, lse=None, stream=None):
    """The C entry point ``attn_fwd_fp8`` on torch tensors.

    q8 [B,H,Nq,d], k8 [B,H,Nk,d] and the transposed values vt8 [B,H,d,Nk]:
    contiguous CUDA tensors of E4M3 codes (torch.float8_e4m3fn or uint8).
    The operands are descale_* times the E4M3 values.  Returns
    (o bf16 [B,H,Nq,d], lse fp32 [B,H,Nq]).
    """
    for name, t in (("q8", q8), ("k8", k8), ("vt8", vt8)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
            raise ValueError(f"{name} must hold E4M3 codes (float8_e4m3fn or uint8)")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D tensor")
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    if k8.shape != (B, H, Nk, d) or vt8.shape != (B, H, d, Nk):
        raise ValueError("k8 must be [B, H, Nk, d] and vt8 [B, H, d, Nk] with q8's B, H and d")
    if k8.device != q8.device or vt8.device != q8.device:
        raise ValueError("q8, k8 and vt8 must be on the same device")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = _out(out, (B, H, Nq, d), torch.bfloat16, q8.device, "out")
    lse = _out(lse, (B, H, Nq), torch.float32, q8.device, "lse")
    with _on(q8.device, stream):
        st = load().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(vt8), _ptr(out), _ptr(lse), B, H, Nq,
                                 Nk, d, int(bool(causal)), float(scale), float(descale_q),
                                 float(descale_k), float(descale_v), _stream_ptr(stream))
    _check(st, "attn_fwd_fp8")
    return out, lse


def decode_workspace_bytes(B, H, Nk, d) -> int:
    return int(load().attn_fwd_decode_workspace_bytes(B, H, Nk, d))


def attn_fwd_decode(q, k, v, scale=None, out=None, lse=None, workspace=None, stream=None):
    """Single-query attention forward (q [B,H,1,d]) split over the keys.
    ``workspace`` (a CUDA uint8 tensor) is allocated here when not given."""
    B, H, Nq, Nk, d = _check_inputs(q, k, v)
    if Nq != 1:
        raise ValueError("attn_fwd_decode takes a single query row (Nq = 1)")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = _out(out, (B, H, 1, d), torch.bfloat16, q.device, "out")
    lse = _out(lse, (B, H, 1), torch.float32, q.device, "lse")
    workspace = _workspace(workspace, decode_workspace_bytes(B, H, Nk, d), q.device)
    ws_ptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with _on(q.device, stream):
        st = load().attn_fwd_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nk,
                                    d, float(scale), ws_ptr, ws_bytes, _stream_ptr(stream))
    _check(st, "attn_fwd_decode")
    return out, lse


def attn_fwd_decode_mx(q, k8, k_scale, v8, v_scale, scale=None, out=None, lse=None,
                       workspace=None, stream=None):
    """The C entry point ``attn_fwd_decode_mx``: single-query attention with
    MXFP8 keys and values.  q bf16 [B,H,1,d]; k8, v8 E4M3 codes [B,H,Nk,d]
    (torch.float8_e4m3fn or uint8); k_scale, v_scale E8M0 codes [B,H,Nk,d/32]
    (torch.float8_e8m0fnu or uint8).  Returns (o bf16 [B,H,1,d], lse fp32
    [B,H,1])."""
    if not q.is_cuda or q.dtype != torch.bfloat16 or q.dim() != 4 or not q.is_contiguous():
        raise ValueError("q must be a contiguous bf16 CUDA tensor [B, H, 1, d]")
    B, H, Nq, d = q.shape
    if Nq != 1:
        raise ValueError("attn_fwd_decode_mx takes a single query row (Nq = 1)")
    Nk = k8.shape[2] if k8.dim() == 4 else -1
    for name, t, shape, dts in (
            ("k8", k8, (B, H, Nk, d), (torch.uint8, torch.float8_e4m3fn)),
            ("v8", v8, (B, H, Nk, d), (torch.uint8, torch.float8_e4m3fn)),
            ("k_scale", k_scale, (B, H, Nk, d // 32), (torch.uint8, torch.float8_e8m0fnu)),
            ("v_scale", v_scale, (B, H, Nk, d // 32), (torch.uint8, torch.float8_e8m0fnu))):
        if (t.device != q.device or t.dtype not in dts or tuple(t.shape) != shape
                or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous {dts[0]} tensor of shape {shape} "
                             f"on {q.device}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = _out(out, (B, H, 1, d), torch.bfloat16, q.device, "out")
    lse = _out(lse, (B, H, 1), torch.float32, q.device, "lse")
    workspace = _workspace(workspace, decode_workspace_bytes(B, H, Nk, d), q.device)
    ws_ptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with _on(q.device, stream):
        st = load().attn_fwd_decode_mx(_ptr(q), _ptr(k8), _ptr(k_scale), _ptr(v8),
                                       _ptr(v_scale), _ptr(out), _ptr(lse), B, H, Nk, d,
                                       float(scale), ws_ptr, ws_bytes, _stream_ptr(stream))
    _check(st, "attn_fwd_decode_mx")
    return out, lse


def attn_fwd_from_host(q, k, v, o, lse, dq, dk, dv, do_, dlse, causal=False, scale=None,
                       stream=None):
    """End-to-end attn_fwd on pinned HOST tensors (q, k, v in; o, lse out)
    through the caller's device buffers dq, dk, dv, do_, dlse.  Asynchronous
    on ``stream``: synchronise before reading o and lse.  Host tensors that
    are not pinned are refused."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B, H, Nq, d] and k, v [B, H, Nk, d]")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    bf, f32 = torch.bfloat16, torch.float32
    for name, t, shape, dt in (("q", q, (B, H, Nq, d), bf), ("k", k, (B, H, Nk, d), bf),
                               ("v", v, (B, H, Nk, d), bf), ("o", o, (B, H, Nq, d), bf),
                               ("lse", lse, (B, H, Nq), f32)):
        if t.is_cuda or not t.is_contiguous() or t.dtype != dt or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be a contiguous {dt} host tensor of shape {shape}")
        # pageable memory would make every copy synchronous and serialise the
        # chunked pipeline whose overlap of copies and kernels is the point
        if not t.is_pinned():
            raise ValueError(f"{name} must be in pinned (page-locked) host memory "
                             f"(tensor.pin_memory())")
    dev = dq.device if dq is not None else torch.device("cuda", torch.cuda.current_device())
    if dev.type != "cuda":
        raise ValueError("dq, dk, dv, do_, dlse must be CUDA tensors")
    dq = _out(dq, (B, H, Nq, d), bf, dev, "dq")
    dk = _out(dk, (B, H, Nk, d), bf, dev, "dk")
    dv = _out(dv, (B, H, Nk, d), bf, dev, "dv")
    do_ = _out(do_, (B, H, Nq, d), bf, dev, "do_")
    dlse = _out(dlse, (B, H, Nq), f32, dev, "dlse")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with _on(dev, stream):
        st = load().attn_fwd_from_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dq),
                                       _ptr(dk), _ptr(dv), _ptr(do_), _ptr(dlse), B, H, Nq, Nk,
                                       d, int(bool(causal)), float(scale), _stream_ptr(stream))
    _check(st, "attn_fwd_from_host")
    return o, lse


def _seqlens_ptr(t, B, name, device):
    if t is None:
        return ctypes.c_void_p(0)
    if (t.device != device or t.dtype != torch.int32 or t.shape != (B,)
            or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous int32 tensor of shape [B] on {device}")
    return _ptr(t)


def attn_fwd_ragged(q, k, v, seqlens_q=None, seqlens_k=None, causal=False, scale=None,
                    out=None, lse=None, stream=None):
    """``attn_fwd_ragged``: sequence b uses its first seqlens_q[b] queries and
    seqlens_k[b] keys of the padded tensors (int32 CUDA tensors [B] or None).
    Rows past seqlens_q[b] of the outputs are not written."""
    B, H, Nq, Nk, d = _check_inputs(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = _out(out, (B, H, Nq, d), torch.bfloat16, q.device, "out")
    lse = _out(lse, (B, H, Nq), torch.float32, q.device, "lse")
    sq = _seqlens_ptr(seqlens_q, B, "seqlens_q", q.device)
    sk = _seqlens_ptr(seqlens_k, B, "seqlens_k", q.device)
    with _on(q.device, stream):
        st = load().attn_fwd_ragged(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), sq, sk, B,
                                    H, Nq, Nk, d, int(bool(causal)), float(scale),
                                    _stream_ptr(stream))
    _check(st, "attn_fwd_ragged")
    return out, lse


def attn_fwd_decode_ragged(q, k, v, seqlens_k=None, scale=None, out=None, lse=None,
                           workspace=None, stream=None):
    """``attn_fwd_decode_ragged``: one query per (b, h) over the first
    seqlens_k[b] keys of the padded k and v."""
    B, H, Nq, Nk, d = _check_inputs(q, k, v)
    if Nq != 1:
        raise ValueError("attn_fwd_decode_ragged takes a single query row (Nq = 1)")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = _out(out, (B, H, 1, d), torch.bfloat16, q.device, "out")
    lse = _out(lse, (B, H, 1), torch.float32, q.device, "lse")
    workspace = _workspace(workspace, decode_workspace_bytes(B, H, Nk, d), q.device)
    ws_ptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    sk = _seqlens_ptr(seqlens_k, B, "seqlens_k", q.device)
    with _on(q.device, stream):
        st = load().attn_fwd_decode_ragged(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), sk,
                                           B, H, Nk, d, float(scale), ws_ptr, ws_bytes,
                                           _stream_ptr(stream))
    _check(st, "attn_fwd_decode_ragged")
    return out, lse


def attn_merge(o_parts, lse_parts, out=None, lse=None, stream=None):
    """The C entry point ``attn_merge``: attention over all keys from the
    results over disjoint key sets.  o_parts bf16 [S, B, H, Nq, d] and
    lse_parts fp32 [S, B, H, Nq], CUDA, contiguous.  Returns (o, lse)."""
    if o_parts.dim() != 5 or lse_parts.shape != o_parts.shape[:4]:
        raise ValueError("o_parts must be [S, B, H, Nq, d] and lse_parts [S, B, H, Nq]")
    for name, t, dt in (("o_parts", o_parts, torch.bfloat16), ("lse_parts", lse_parts, torch.float32)):
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dt} CUDA tensor")
    if lse_parts.device != o_parts.device:
        raise ValueError("o_parts and lse_parts must be on the same device")
    S, B, H, Nq, d = o_parts.shape
    out = _out(out, (B, H, Nq, d), torch.bfloat16, o_parts.device, "out")
    lse = _out(lse, (B, H, Nq), torch.float32, o_parts.device, "lse")
    with _on(o_parts.device, stream):
        st = load().attn_merge(_ptr(o_parts), _ptr(lse_parts), S, _ptr(out), _ptr(lse), B, H,
                               Nq, d, _stream_ptr(stream))
    _check(st, "attn_merge")
    return out, lse


def bwd_workspace_bytes(B, H, Nq, Nk, d) -> int:
    return int(load().attn_bwd_workspace_bytes(B, H, Nq, Nk, d))


def attn_bwd(q, k, v, o, lse, dout, causal=False, scale=None, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """The C entry point ``attn_bwd``: gradients (dq, dk, dv) of attn_fwd for
    the upstream gradient ``dout``, given the forward's inputs and its
    outputs ``o`` and ``lse``.  ``workspace`` (a CUDA uint8 tensor) is
    allocated here when not given."""
    B, H, Nq, Nk, d = _check_inputs(q, k, v)
    for name, t, dt in (("o", o, torch.bfloat16), ("dout", dout, torch.bfloat16),
                        ("lse", lse, torch.float32)):
        if t.device != q.device or t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dt} tensor on {q.device}")
    if o.shape != q.shape or dout.shape != q.shape or lse.shape != (B, H, Nq):
        raise ValueError("o and dout must be [B, H, Nq, d] and lse [B, H, Nq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = _out(dq, q.shape, torch.bfloat16, q.device, "dq")
    dk = _out(dk, k.shape, torch.bfloat16, q.device, "dk")
    dv = _out(dv, v.shape, torch.bfloat16, q.device, "dv")
    workspace = _workspace(workspace, bwd_workspace_bytes(B, H, Nq, Nk, d), q.device)
    with _on(q.device, stream):
        st = load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                             _ptr(dq), _ptr(dk), _ptr(dv), B, H, Nq, Nk, d, int(bool(causal)),
                             float(scale), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check(st, "attn_bwd")
    return dq, dk, dv


def device_error() -> int:
    """Synchronise and read/clear the kernels' device error word (0 = none)."""
    return int(load().attn_device_error())


def attn_pair_product(a, b, d=None, stream=None):
    """D = A Bᵀ through the CTA-pair product (``attn_pair_product``): a is a
    256 x 64 and b a 128 x 64 bfloat16 CUDA tensor; returns the 256 x 128
    float32 D.  Blocks until the product is done."""
    for name, t, shape in (("a", a, (256, 64)), ("b", b, (128, 64))):
        if not t.is_cuda or t.dtype != torch.bfloat16 or tuple(t.shape) != shape \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor of shape {shape}")
    if b.device != a.device:
        raise ValueError("a and b must be on the same device")
    with _on(a.device, stream):
        d = _out(d, (256, 128), torch.float32, a.device, "d")
        _check(load().attn_pair_product(_ptr(a), _ptr(b), _ptr(d), _stream_ptr(stream)),
               "attn_pair_product")
    return d


def bench_mma_rate(form, issuer=1, busy=0, waits=0, steps=4096, reps=5, device=None,
                   stream=None):
    """Time one issuer's products (``attn_bench_mma_rate``): form 1 is the
    single-CTA 128 x 128 x 16 product, form 2 the CTA-pair 256 x 128 x 16 one;
    issuer 0 a lone lane, 1 a converged warp with an elected issuing lane.
    Returns {"ms": mean launch time, "cycles": mean issuer cycles, "sms": SMs
    used}."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    ms, cyc, sms = ctypes.c_float(), ctypes.c_double(), ctypes.c_int()
    with _on(dev, stream):
        _check(load().attn_bench_mma_rate(int(form), int(issuer), int(busy), int(waits), int(steps),
                                          int(reps),
                                          ctypes.byref(ms), ctypes.byref(cyc), ctypes.byref(sms),
                                          _stream_ptr(stream)),
               "attn_bench_mma_rate")
    return {"ms": ms.value, "cycles": cyc.value, "sms": sms.value}
