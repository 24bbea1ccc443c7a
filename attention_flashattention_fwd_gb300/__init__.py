"""Fused scaled-dot-product attention forward for one GB300 GPU (sm_103a).

O = softmax(scale * Q K^T [+ causal mask]) V and the fp32 logsumexp per row,
computed tile by tile with the online softmax so that the score matrix never
reaches HBM, and its backward pass (dQ, dK, dV recomputing P from the
logsumexp).  The compute runs in the CUDA library ``libgbattn.so`` behind a
C ABI (declared in ``include/gbattn.h``); :mod:`.binding` only marshals
torch tensors into that ABI.
"""
from .inputs import WORKLOADS, Workload, make_qkv, make_workload  # noqa: F401


def __getattr__(name):
    # The binding is imported on first use so that the input generator works on
    # machines without the built library; every compute entry point raises if
    # the CUDA library is missing.
    if name in ("attention", "attn_fwd", "attn_fwd_decode", "attn_fwd_from_host", "attn_bwd"):
        import importlib
        return getattr(importlib.import_module(__name__ + ".binding"), name)
    raise AttributeError(name)
