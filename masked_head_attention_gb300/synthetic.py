"""Seeded synthetic inputs for masked multi-head attention.

This module only draws random numbers and rounds them to the storage dtype.
It holds none of the attention arithmetic, so the fp64 oracle and the CUDA
kernels can both be fed from it without sharing any of the method.

Workloads (shapes, value distributions and length mixes) follow the five
configurations the pages' measurements are quoted on; they are synthetic
stand-ins, generated on the host with a seeded torch CPU generator.
"""
import math
from dataclasses import dataclass, field
from typing import Optional, Tuple

import torch

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_KV_LEN = 2

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    """One attention problem; `kind` is "mha" (self-attention), "prenorm"
    (Pre-LN cross-attention), "prenorm_residual" (the same plus x) or
    "mha_bwd" (the backward of self-attention: q, k, v and dout)."""
    name: str
    kind: str
    dtype: str
    B: int
    H: int
    Lq: int
    Lk: int
    D: int
    mask: int
    qk_std: float = 1.0                       # std of the N(0, s^2) draw for Q and K (or x)
    v_std: float = 1.0
    len_range: Optional[Tuple[int, int]] = None   # inclusive uniform range of kv lengths
    eps: float = 1e-5
    gamma_mean: float = 1.0
    gamma_std: float = 0.1
    beta_std: float = 0.1
    note: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


# The five workloads.  Sizes and distributions are the measured configurations
# of the masked-MHA pages; kv lengths are drawn per batch from the seed.
WORKLOADS = {
    "c1_causal_f32": Workload(
        "c1_causal_f32", "mha", "f32", B=4, H=8, Lq=128, Lk=128, D=64, mask=MASK_CAUSAL,
        note="causal self-attention, fp32, Q/K/V iid N(0,1)"),
    "c2_padding_f32": Workload(
        "c2_padding_f32", "mha", "f32", B=16, H=8, Lq=512, Lk=512, D=64, mask=MASK_KV_LEN,
        len_range=(1, 512), note="padding-mask self-attention, fp32, lengths U{1..512}"),
    "c3_causal_bf16": Workload(
        "c3_causal_bf16", "mha", "bf16", B=1, H=32, Lq=2048, Lk=2048, D=128, mask=MASK_CAUSAL,
        qk_std=math.sqrt(2.5),
        note="causal self-attention, bf16; Q,K std sqrt(2.5) so logits have std 2.5 (span ~[-10,10])"),
    "c4_prenorm_bf16": Workload(
        "c4_prenorm_bf16", "prenorm", "bf16", B=32, H=16, Lq=2048, Lk=2048, D=64,
        mask=MASK_KV_LEN, len_range=(1024, 2048),
        note="Pre-LN cross-attention, bf16, d_model 1024, kv lengths U{1024..2048}"),
    "c4r_prenorm_residual_bf16": Workload(
        "c4r_prenorm_residual_bf16", "prenorm_residual", "bf16", B=32, H=16, Lq=2048, Lk=2048,
        D=64, mask=MASK_KV_LEN, len_range=(1024, 2048),
        note="Pre-LN cross-attention with the residual add (out = x + attention), shapes of c4"),
    "c5_long_causal_bf16": Workload(
        "c5_long_causal_bf16", "mha", "bf16", B=2, H=32, Lq=8192, Lk=8192, D=128,
        mask=MASK_CAUSAL, note="long causal self-attention, bf16, Q/K/V iid N(0,1)"),
    "c6_decode_bf16": Workload(
        "c6_decode_bf16", "mha", "bf16", B=8, H=32, Lq=1, Lk=8192, D=128, mask=MASK_KV_LEN,
        len_range=(4096, 8192),
        note="decode step: one new query row per (b, h) against a KV cache of U{4096..8192} "
             "valid keys, bf16"),
    "b2_padding_f32_bwd": Workload(
        "b2_padding_f32_bwd", "mha_bwd", "f32", B=16, H=8, Lq=512, Lk=512, D=64,
        mask=MASK_KV_LEN, len_range=(1, 512),
        note="backward (dq, dk, dv) of the c2 padding-mask workload, fp32; dout iid N(0,1)"),
    "b3_causal_f32_bwd": Workload(
        "b3_causal_f32_bwd", "mha_bwd", "f32", B=2, H=16, Lq=1024, Lk=1024, D=128,
        mask=MASK_CAUSAL, note="backward of causal self-attention, fp32, D=128; dout iid N(0,1)"),
    "b5_causal_bf16_bwd": Workload(
        "b5_causal_bf16_bwd", "mha_bwd", "bf16", B=1, H=32, Lq=2048, Lk=2048, D=128,
        mask=MASK_CAUSAL, qk_std=math.sqrt(2.5),
        note="backward of the c3 causal bf16 workload (fp32 arithmetic, bf16 gradients); "
             "dout iid N(0,1)"),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _normal(g, shape, std, dtype):
    t = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def lengths(g, B, len_range):
    lo, hi = len_range
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int32)


def make(w: Workload, seed: int = 0):
    """Host tensors for workload `w`: dict with q/k/v (or x, gamma, beta, k, v),
    kv_lengths (int32 [B] or None), and the scalars scale, eps."""
    g = _gen(seed)
    dt = DTYPES[w.dtype]
    out = {"scale": w.scale, "kv_lengths": None}
    if w.kind in ("mha", "mha_bwd"):
        out["q"] = _normal(g, (w.B, w.H, w.Lq, w.D), w.qk_std, dt)
        out["k"] = _normal(g, (w.B, w.H, w.Lk, w.D), w.qk_std, dt)
        out["v"] = _normal(g, (w.B, w.H, w.Lk, w.D), w.v_std, dt)
        if w.kind == "mha_bwd":
            out["dout"] = _normal(g, (w.B, w.H, w.Lq, w.D), 1.0, dt)
    elif w.kind in ("prenorm", "prenorm_residual"):
        N = w.H * w.D
        out["x"] = _normal(g, (w.B, w.Lq, N), w.qk_std, dt)
        out["gamma"] = (torch.randn((N,), generator=g, dtype=torch.float32) * w.gamma_std
                        + w.gamma_mean)
        out["beta"] = torch.randn((N,), generator=g, dtype=torch.float32) * w.beta_std
        out["k"] = _normal(g, (w.B, w.H, w.Lk, w.D), 1.0, dt)
        out["v"] = _normal(g, (w.B, w.H, w.Lk, w.D), w.v_std, dt)
        out["eps"] = w.eps
    else:
        raise ValueError(w.kind)
    if w.mask & MASK_KV_LEN and w.len_range is not None:
        out["kv_lengths"] = lengths(g, w.B, w.len_range)
    return out


def small(kind="mha", dtype="f32", B=2, H=2, Lq=70, Lk=70, D=64, mask=MASK_CAUSAL,
          qk_std=1.0, len_range=None, name="small"):
    """A Workload for parity tests at sizes the oracle finishes in seconds."""
    return Workload(name, kind, dtype, B, H, Lq, Lk, D, mask, qk_std=qk_std,
                    len_range=len_range)
