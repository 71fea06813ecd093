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

Paired Head Attention inputs: q, k, v (B, T, H, D) ~ N(0, 1), drawn in that
order (the pages give no workload; the shapes are the V2 prefill's query heads).

Decode inputs: V2 q (B, Hq, D) and caches (B, L, Hkv, D); V1 q1, q2 (B, H, d),
caches k1, k2 (B, L, H, d) and v (B, L, H, 2d), drawn in that order, each
contiguous (a cache is written one row per token, so the two branches' keys
live in separate arrays).  With per-sequence lengths the lengths are drawn
last, uniform on 1 .. L (torch.randint); cache rows past a sequence's length
are drawn like the rest, so they hold ordinary values that must not count.
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
class PairedShape:
    """Paired Head Attention: H heads (H/2 interleaved pairs), head dim D."""
    B: int
    T: int
    H: int
    D: int
    dtype: str = "bf16"


@dataclass(frozen=True)
class DecodeShape:
    """DIFF V2 decode: one new query token per sequence, L cached rows
    (varlen: sequence b attends its first lens[b] rows)."""
    B: int
    L: int
    Hq: int
    Hkv: int
    D: int
    dtype: str = "bf16"
    varlen: bool = False


@dataclass(frozen=True)
class V1DecodeShape:
    """DIFF V1 decode: one new query token per sequence, L cached rows of k1,
    k2 (head dim d) and v (2d) per diff head."""
    B: int
    L: int
    H: int
    d: int
    layer_index: int
    dtype: str = "bf16"
    varlen: bool = False


# The five workloads, named by what they are.
WORKLOADS = {
    "v1_fp32_B1_T64_H2_d32": V1Shape(1, 64, 2, 32, 1, "fp32"),
    "v1_bf16_B4_T2048_H16_d64": V1Shape(4, 2048, 16, 64, 12, "bf16"),
    "v2_bf16_B8_T4096_Hq32_Hkv8_D128": V2Shape(8, 4096, 32, 8, 128, "bf16"),
    "v2_decode_bf16_B64_L32768_Hq64_Hkv8_D128": DecodeShape(64, 32768, 64, 8, 128, "bf16"),
    "v1_bf16_B1_T32768_H12_d128": V1Shape(1, 32768, 12, 128, 27, "bf16"),
    # decode beyond the five: per-sequence lengths, and DIFF V1 decode
    "v2_decode_varlen_bf16_B64_L32768_Hq64_Hkv8_D128": DecodeShape(64, 32768, 64, 8, 128, "bf16", True),
    "v1_decode_bf16_B32_L16384_H12_d128": V1DecodeShape(32, 16384, 12, 128, 27, "bf16"),
    # Paired Head Attention on the V2 prefill's query-head shapes
    "paired_bf16_B8_T4096_H32_D128": PairedShape(8, 4096, 32, 128, "bf16"),
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


def make_paired(s: PairedShape, seed: int = 0, device="cpu") -> dict:
    """q, k, v (B,T,H,D), drawn in that order."""
    g = _gen(seed, device)
    dt = _DT[s.dtype]
    q = _normal((s.B, s.T, s.H, s.D), 1.0, dt, g, device)
    k = _normal((s.B, s.T, s.H, s.D), 1.0, dt, g, device)
    v = _normal((s.B, s.T, s.H, s.D), 1.0, dt, g, device)
    return {"q": q, "k": k, "v": v}


def make_decode(s: DecodeShape, seed: int = 0, device="cpu") -> dict:
    """q (B,Hq,D); k_cache, v_cache (B,L,Hkv,D); lam (B,Hq/2) fp32 logits."""
    g = _gen(seed, device)
    dt = _DT[s.dtype]
    q = _normal((s.B, s.Hq, s.D), 1.0, dt, g, device)
    k = _normal((s.B, s.L, s.Hkv, s.D), 1.0, dt, g, device)
    v = _normal((s.B, s.L, s.Hkv, s.D), 1.0, dt, g, device)
    lam = torch.randn((s.B, s.Hq // 2), generator=g, dtype=torch.float32, device=device)
    out = {"q": q, "k_cache": k, "v_cache": v, "lam": lam}
    if s.varlen:
        out["cache_lens"] = _lens(s.B, s.L, g, device)
    return out


def _lens(B: int, L: int, g, device) -> torch.Tensor:
    return torch.randint(1, L + 1, (B,), generator=g, dtype=torch.int64, device=device).to(torch.int32)


def make_v1_decode(s: V1DecodeShape, seed: int = 0, device="cpu") -> dict:
    """q1, q2 (B,H,d); k1_cache, k2_cache (B,L,H,d); v_cache (B,L,H,2d);
    lam_q1, lam_k1, lam_q2, lam_k2 (d,) fp32; cache_lens (B,) int32 if varlen."""
    g = _gen(seed, device)
    dt = _DT[s.dtype]
    q1 = _normal((s.B, s.H, s.d), 1.0, dt, g, device)
    q2 = _normal((s.B, s.H, s.d), 1.0, dt, g, device)
    k1 = _normal((s.B, s.L, s.H, s.d), 1.0, dt, g, device)
    k2 = _normal((s.B, s.L, s.H, s.d), 1.0, dt, g, device)
    v = _normal((s.B, s.L, s.H, 2 * s.d), 1.0, dt, g, device)
    lam = [torch.randn(s.d, generator=g, dtype=torch.float32, device=device) * 0.1
           for _ in range(4)]
    out = {"q1": q1, "q2": q2, "k1_cache": k1, "k2_cache": k2, "v_cache": v,
           "lam_q1": lam[0], "lam_k1": lam[1], "lam_q2": lam[2], "lam_k2": lam[3],
           "layer_index": s.layer_index}
    if s.varlen:
        out["cache_lens"] = _lens(s.B, s.L, g, device)
    return out


def make_grad_out(shape, dtype: str = "bf16", seed: int = 0, device="cpu") -> torch.Tensor:
    """Upstream gradient dL/dout ~ N(0, 1) of the given output shape, drawn in
    fp32 with its own generator (seed + 1000003) and rounded to dtype."""
    g = _gen(int(seed) + 1000003, device)
    return _normal(tuple(shape), 1.0, _DT[dtype], g, device)


def make_lambda_proj(B: int, T: int, C: int, P: int, dtype: str = "bf16", seed: int = 0, device="cpu") -> dict:
    """Inputs of DIFF V2's projected lambda: the layer input x (B, T, C) ~ N(0, 1)
    and a random-init projection w (C, P) ~ N(0, 0.02^2) (no trained weights
    exist here), drawn in that order with their own generator (seed + 2000003)."""
    g = _gen(int(seed) + 2000003, device)
    x = _normal((B, T, C), 1.0, _DT[dtype], g, device)
    w = _normal((C, P), 0.02, _DT[dtype], g, device)
    return {"x": x, "w_lam": w}


def make(shape, seed: int = 0, device="cpu") -> dict:
    if isinstance(shape, V1Shape):
        return make_v1(shape, seed, device)
    if isinstance(shape, V2Shape):
        return make_v2(shape, seed, device)
    if isinstance(shape, DecodeShape):
        return make_decode(shape, seed, device)
    if isinstance(shape, V1DecodeShape):
        return make_v1_decode(shape, seed, device)
    if isinstance(shape, PairedShape):
        return make_paired(shape, seed, device)
    raise TypeError(type(shape))
