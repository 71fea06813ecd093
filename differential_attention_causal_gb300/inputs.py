"""Seeded synthetic inputs for the differential-attention forward.

This module holds NO arithmetic of the method: it only draws random tensors
in a fixed order with a seeded ``torch.Generator`` so that the CUDA path and
the CPU oracle see the same values.  It imports nothing else from this
package and nothing from the oracle.

Recipe (shapes follow the workloads named in ``WORKLOADS``):
  * one ``torch.Generator(device)`` seeded with ``seed`` (default 0);
  * draw order: q, k, v, then the lambda inputs;
  * q, k, v ~ N(0, 1) drawn in fp32, then rounded to the workload dtype;
  * DIFF V1 lambda vectors lam_q1, lam_k1, lam_q2, lam_k2 ~ N(0, 0.1), fp32,
    length d (the initialisation in "How best to implement a differential
    transformer?", first CausalSelfAttention);
  * DIFF V2 lambda logits ~ N(0, 1), fp32, one per (token, output head);
  * large tensors are drawn batch entry by batch entry (same generator, in
    order) so that no fp32 copy of a multi-GB tensor is ever held.

V1 q and k are drawn as one interleaved (B, T, 2H, d) tensor each, as the
nanoGPT issue lays them out; q1 = q[:, :, 0::2], q2 = q[:, :, 1::2] (and the
same for k) are strided views.  v is (B, T, H, 2d).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

_DT = {"fp32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class V1Shape:
    """DIFF V1: H diff heads, q/k head dim d, v head dim 2d."""
    B: int
    T: int
    H: int
    d: int
    layer_index: int
    dtype: str = "bf16"


@dataclass(frozen=True)
class V2Shape:
    """DIFF V2 prefill: Hq query heads (Hq/2 pairs), Hkv kv heads, head dim D."""
    B: int
    T: int
    Hq: int
    Hkv: int
    D: int
    dtype: str = "bf16"


@dataclass(frozen=True)
class DecodeShape:
    """DIFF V2 decode: one new query token per sequence, L cached rows."""
    B: int
    L: int
    Hq: int
    Hkv: int
    D: int
    dtype: str = "bf16"


# The five workloads, named by what they are.
WORKLOADS = {
    "v1_fp32_B1_T64_H2_d32": V1Shape(1, 64, 2, 32, 1, "fp32"),
    "v1_bf16_B4_T2048_H16_d64": V1Shape(4, 2048, 16, 64, 12, "bf16"),
    "v2_bf16_B8_T4096_Hq32_Hkv8_D128": V2Shape(8, 4096, 32, 8, 128, "bf16"),
    "v2_decode_bf16_B64_L32768_Hq64_Hkv8_D128": DecodeShape(64, 32768, 64, 8, 128, "bf16"),
    "v1_bf16_B1_T32768_H12_d128": V1Shape(1, 32768, 12, 128, 27, "bf16"),
}


def _gen(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, dtype, g, device) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 one leading index at a time, rounded to dtype."""
    out = torch.empty(shape, dtype=dtype, device=device)
    for i in range(shape[0]):
        x = torch.randn(shape[1:], generator=g, dtype=torch.float32, device=device)
        if std != 1.0:
            x.mul_(std)
        out[i].copy_(x)
    return out


def make_v1(s: V1Shape, seed: int = 0, device="cpu") -> dict:
    """q, k (B,T,2H,d); v (B,T,H,2d); lam_q1, lam_k1, lam_q2, lam_k2 (d,) fp32."""
    g = _gen(seed, device)
    dt = _DT[s.dtype]
    q = _normal((s.B, s.T, 2 * s.H, s.d), 1.0, dt, g, device)
    k = _normal((s.B, s.T, 2 * s.H, s.d), 1.0, dt, g, device)
    v = _normal((s.B, s.T, s.H, 2 * s.d), 1.0, dt, g, device)
    lam = [torch.randn(s.d, generator=g, dtype=torch.float32, device=device) * 0.1
           for _ in range(4)]
    return {"q": q, "k": k, "v": v,
            "q1": q[:, :, 0::2], "q2": q[:, :, 1::2],
            "k1": k[:, :, 0::2], "k2": k[:, :, 1::2],
            "lam_q1": lam[0], "lam_k1": lam[1], "lam_q2": lam[2], "lam_k2": lam[3],
            "layer_index": s.layer_index}


def make_v2(s: V2Shape, seed: int = 0, device="cpu") -> dict:
    """q (B,T,Hq,D); k, v (B,T,Hkv,D); lam (B,T,Hq/2) fp32 logits."""
    g = _gen(seed, device)
    dt = _DT[s.dtype]
    q = _normal((s.B, s.T, s.Hq, s.D), 1.0, dt, g, device)
    k = _normal((s.B, s.T, s.Hkv, s.D), 1.0, dt, g, device)
    v = _normal((s.B, s.T, s.Hkv, s.D), 1.0, dt, g, device)
    lam = torch.randn((s.B, s.T, s.Hq // 2), generator=g, dtype=torch.float32, device=device)
    return {"q": q, "k": k, "v": v, "lam": lam}


def make_decode(s: DecodeShape, seed: int = 0, device="cpu") -> dict:
    """q (B,Hq,D); k_cache, v_cache (B,L,Hkv,D); lam (B,Hq/2) fp32 logits."""
    g = _gen(seed, device)
    dt = _DT[s.dtype]
    q = _normal((s.B, s.Hq, s.D), 1.0, dt, g, device)
    k = _normal((s.B, s.L, s.Hkv, s.D), 1.0, dt, g, device)
    v = _normal((s.B, s.L, s.Hkv, s.D), 1.0, dt, g, device)
    lam = torch.randn((s.B, s.Hq // 2), generator=g, dtype=torch.float32, device=device)
    return {"q": q, "k_cache": k, "v_cache": v, "lam": lam}


def make(shape, seed: int = 0, device="cpu") -> dict:
    if isinstance(shape, V1Shape):
        return make_v1(shape, seed, device)
    if isinstance(shape, V2Shape):
        return make_v2(shape, seed, device)
    if isinstance(shape, DecodeShape):
        return make_decode(shape, seed, device)
    raise TypeError(type(shape))
