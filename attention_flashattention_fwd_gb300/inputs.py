"""Seeded synthetic inputs for the attention forward workloads.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so the CUDA path and the fp64 oracle can both be fed
from it without sharing any of the method.

Every workload is iid Gaussian Q, K, V drawn in fp32 from a seeded
``torch.Generator`` (Q first, then K, then V), scaled by its standard
deviation and rounded to bfloat16.  The long-sequence workload draws Q and K
with standard deviation 1.5 (a wider logit spread); all others use 1.
"""
from dataclasses import dataclass
import math

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    sigma_qk: float = 1.0
    seed: int = 1000

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def decode(self) -> bool:
        return self.Nq == 1

    def flops(self) -> float:
        """4 B H Nq Nk d (two GEMMs), halved for the causal mask."""
        f = 4.0 * self.B * self.H * self.Nq * self.Nk * self.d
        return f / 2 if self.causal else f

    def algorithmic_bytes(self) -> int:
        """Bytes read and written once: Q, K, V, O in bf16 and lse in fp32."""
        bh = self.B * self.H
        return bh * (2 * self.Nq * self.d * 2 + 2 * self.Nk * self.d * 2 + 4 * self.Nq)


# The five workloads of the attention forward study, in order.
WORKLOADS = {
    "tiny_b1h1n128d64": Workload("tiny_b1h1n128d64", 1, 1, 128, 128, 64, False, seed=1000),
    "b4h8n1024d64": Workload("b4h8n1024d64", 4, 8, 1024, 1024, 64, False, seed=1001),
    "b2h16n4096d128_causal": Workload("b2h16n4096d128_causal", 2, 16, 4096, 4096, 128, True,
                                      seed=1002),
    "b1h32n16384d128_causal": Workload("b1h32n16384d128_causal", 1, 32, 16384, 16384, 128,
                                       True, sigma_qk=1.5, seed=1003),
    "decode_b64h32nk8192d128": Workload("decode_b64h32nk8192d128", 64, 32, 1, 8192, 128, False,
                                        seed=1004),
}

# The non-causal counterpart of the 4096-token workload (the study's throughput
# target covers causal and non-causal prefill at d = 128, N >= 4096).
EXTRA_WORKLOADS = {
    "b2h16n4096d128": Workload("b2h16n4096d128", 2, 16, 4096, 4096, 128, False, seed=1005),
}


def make_qkv(B, H, Nq, Nk, d, seed, device="cpu", sigma_qk=1.0, sigma_v=1.0):
    """Q [B,H,Nq,d], K and V [B,H,Nk,d], bf16, contiguous, on ``device``."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    q = torch.randn((B, H, Nq, d), generator=g, device=device, dtype=torch.float32)
    q = (q * sigma_qk).to(torch.bfloat16)
    k = torch.randn((B, H, Nk, d), generator=g, device=device, dtype=torch.float32)
    k = (k * sigma_qk).to(torch.bfloat16)
    v = torch.randn((B, H, Nk, d), generator=g, device=device, dtype=torch.float32)
    v = (v * sigma_v).to(torch.bfloat16)
    return q, k, v


def make_workload(w: Workload, device="cpu", seed=None):
    return make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, w.seed if seed is None else seed, device,
                    sigma_qk=w.sigma_qk)


E4M3_MAX = 448.0  # largest finite float8_e4m3fn value


def make_qkv_fp8(B, H, Nq, Nk, d, seed, device="cpu", sigma_qk=1.0, sigma_v=1.0):
    """FP8 (E4M3) operands with one descale per tensor, for ``attn_fwd_fp8``.

    The Gaussian draws of :func:`make_qkv` (same seed and order, fp32 before any
    rounding), each tensor divided by its descale amax / 448 (so its largest
    magnitude lands on the largest E4M3 value) and rounded by torch to
    float8_e4m3fn.  Returns (q8 [B,H,Nq,d], k8 [B,H,Nk,d], vt8 [B,H,d,Nk] -- the
    values transposed, keys innermost -- as uint8 codes, and the descales
    (dq, dk, dv) as Python floats holding fp32 values)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out, ds = [], []
    for shape, sigma in (((B, H, Nq, d), sigma_qk), ((B, H, Nk, d), sigma_qk),
                         ((B, H, Nk, d), sigma_v)):
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * sigma
        descale = torch.clamp(x.abs().max() / E4M3_MAX, min=2.0 ** -100).to(torch.float32)
        codes = torch.clamp(x / descale, -E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
        out.append(codes.view(torch.uint8))
        ds.append(float(descale))
    q8, k8, v8 = out
    return q8, k8, v8.transpose(2, 3).contiguous(), tuple(ds)


def make_workload_fp8(w: Workload, device="cpu", seed=None):
    return make_qkv_fp8(w.B, w.H, w.Nq, w.Nk, w.d, w.seed if seed is None else seed, device,
                        sigma_qk=w.sigma_qk)


def bf16_bits(t: torch.Tensor):
    """The raw 16-bit patterns of a bf16 tensor as a numpy uint16 array (CPU copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def mx_quantize(x: torch.Tensor, block: int = 32):
    """MXFP8 quantisation of the last dimension of an fp32 tensor, following the
    OCP Microscaling (MX) v1.0 conversion: each block of ``block`` consecutive
    elements shares the E8M0 scale 2^(floor(log2 amax) - 8) (8 = the largest
    E4M3 exponent), the elements divided by it are rounded to E4M3 by torch,
    saturating at +-448.  Returns (codes uint8 [..., d], scales uint8
    [..., d / block])."""
    shp = x.shape
    xb = x.reshape(*shp[:-1], shp[-1] // block, block).to(torch.float32)
    amax = xb.abs().amax(dim=-1)
    e = torch.floor(torch.log2(torch.where(amax > 0, amax, torch.ones_like(amax)))) - 8
    X = torch.clamp(e + 127, 0, 254)  # biased E8M0 exponent
    y = xb / torch.exp2(X - 127)[..., None]
    codes = torch.clamp(y, -E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.reshape(shp), X.to(torch.uint8)


def make_qkv_mx(B, H, Nk, d, seed, device="cpu", sigma_qk=1.0, sigma_v=1.0):
    """A decode step with MXFP8 keys and values: the Gaussian draws of
    :func:`make_qkv` for Nq = 1 (same seed and order), q rounded to bf16 and K, V
    quantised by :func:`mx_quantize`.  Returns (q bf16 [B,H,1,d], k8, k_scale,
    v8, v_scale) with codes uint8 [B,H,Nk,d] and scales uint8 [B,H,Nk,d/32]."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    q = (torch.randn((B, H, 1, d), generator=g, device=device, dtype=torch.float32)
         * sigma_qk).to(torch.bfloat16)
    k = torch.randn((B, H, Nk, d), generator=g, device=device, dtype=torch.float32) * sigma_qk
    v = torch.randn((B, H, Nk, d), generator=g, device=device, dtype=torch.float32) * sigma_v
    k8, ks = mx_quantize(k)
    del k
    v8, vs = mx_quantize(v)
    return q, k8.contiguous(), ks.contiguous(), v8.contiguous(), vs.contiguous()


def make_workload_mx(w: Workload, device="cpu", seed=None):
    return make_qkv_mx(w.B, w.H, w.Nk, w.d, w.seed if seed is None else seed, device,
                       sigma_qk=w.sigma_qk)
