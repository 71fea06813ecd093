"""GPU checks of the DIFF V2 forward with the rotary embedding folded in
(diffattn_v2_fwd_rope): k rotated in place by the first launch, q rotated tile
by tile inside the prefill kernel.

Two kinds of check:
  * bit equality with the two-call path it replaces (diffattn_prologue on q
    and k, then diffattn_v2_fwd): both form cos / sin with one shared function
    and rotate with the same fma form, rounding to bf16 the same way, so the
    outputs and the rotated k must be identical, and q must be untouched;
  * parity with the fp64 oracle: oracle.v2_fwd on oracle.rope(q), oracle.rope(k)
    (rotary embedding of "How best to implement a differential transformer?",
    the issue's apply_rotary_pos_emb before the attention; DiffAttnV2 of
    "Differential Transformer V2"), within the bf16 bound of the other
    attention outputs (max abs <= 2e-2, rel L2 <= 5e-3).
"""
import numpy as np
import pytest
import torch

import oracle
import rescale_cases as rc
from differential_attention_causal_gb300 import inputs

from test_gpu_parity import assert_parity, binding, built  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu

SHAPES = [  # B, T, Hq, Hkv, D, pos0
    (2, 300, 8, 2, 128, 0),
    (1, 129, 4, 2, 64, 5000),
    (1, 1, 2, 1, 128, 7),
    (3, 640, 4, 1, 128, 123456),
    (1, 1000, 16, 2, 64, 0),
    (2, 257, 12, 3, 128, 31),
]


def _inputs(B, T, Hq, Hkv, D, seed):
    return inputs.make_v2(inputs.V2Shape(B, T, Hq, Hkv, D, "bf16"), seed=seed)


def _two_call(xd, pos0):
    q, k = xd["q"].clone(), xd["k"].clone()
    binding().prologue(q=q, k=k, pos0=pos0)
    return binding().v2_fwd(q, k, xd["v"], xd["lam"]), k


@pytest.mark.parametrize("B,T,Hq,Hkv,D,pos0", SHAPES)
def test_fused_rope_matches_two_calls_bit_for_bit(B, T, Hq, Hkv, D, pos0):
    x = _inputs(B, T, Hq, Hkv, D, seed=T + Hq)
    xd = {n: v.cuda() for n, v in x.items()}
    ref_out, ref_k = _two_call(xd, pos0)
    q0, k = xd["q"].clone(), xd["k"].clone()
    out = binding().v2_fwd_rope(xd["q"], k, xd["v"], xd["lam"], pos0=pos0)
    assert binding().last_launch_count() == 2
    torch.cuda.synchronize()
    assert torch.equal(xd["q"], q0), "q must be left as it is"
    assert torch.equal(k, ref_k), "k must be rotated in place as the prologue rotates it"
    assert torch.equal(out, ref_out), f"max diff {(out.float() - ref_out.float()).abs().max().item():.3e}"
    assert binding().device_error() == 0


@pytest.mark.parametrize("B,T,Hq,Hkv,D,pos0", SHAPES)
def test_fused_rope_vs_oracle(B, T, Hq, Hkv, D, pos0):
    x = _inputs(B, T, Hq, Hkv, D, seed=7 * T + D)
    xd = {n: v.cuda() for n, v in x.items()}
    out = binding().v2_fwd_rope(xd["q"], xd["k"], xd["v"], xd["lam"], pos0=pos0)
    ref = oracle.v2_fwd(oracle.rope(x["q"], pos0=pos0), oracle.rope(x["k"], pos0=pos0), x["v"], x["lam"])
    assert_parity(out, ref, "bf16")


def test_fused_rope_positions_and_repeat_calls():
    """Large position offsets (angles of ~10^5 rad, reduced modulo 2 pi in
    float arithmetic) and calls of different T in a row: still equal to the
    two-call path, and repeated calls give the same bits."""
    D = 128
    for T, pos0 in ((700, 0), (300, 90000), (1, 5), (129, 16000000)):
        x = _inputs(1, T, 4, 2, D, seed=T)
        xd = {n: v.cuda() for n, v in x.items()}
        ref_out, ref_k = _two_call(xd, pos0)
        outs = []
        for _ in range(2):
            k = xd["k"].clone()
            outs.append(binding().v2_fwd_rope(xd["q"], k, xd["v"], xd["lam"], pos0=pos0))
            assert torch.equal(k, ref_k)
        assert torch.equal(outs[0], ref_out) and torch.equal(outs[1], ref_out)
    assert binding().device_error() == 0


def test_fused_rope_lazy_rescale():
    """Planted per-key-tile score levels (as in rescale_cases) through the
    Q-rotating kernel.  The planted components sit in channel pair
    (D/2 - 1, D - 1), the slowest rotary frequency, with channel D - 1 of q
    and k set to 0, and the rotary base is 1e30, so that this pair turns by
    less than 1e-25 rad and keeps its values exactly (the planted keys are
    large: a rotation would round them to bf16 differently than the fp64
    oracle's exact rotation, a difference of the input's precision, not of
    the kernel); the other pairs turn by up to pos rad as usual.  The
    branches are checked on the host from the rotated bf16 q, k that the
    two-call path produces (the same bits the kernel rotates to), then the
    fused output must equal the two-call output and match the oracle."""
    B, T, Hq, Hkv, D = 1, 1024, 4, 2, 128
    G = Hq // Hkv
    x = _inputs(B, T, Hq, Hkv, D, seed=11)
    c = D // 2 - 1
    lv = rc.key_channel0(T, D, rc.targets((T + 127) // 128)).to(x["k"].dtype)
    x["q"][:, :, :, c] = rc.A
    x["q"][:, :, :, D - 1] = 0
    x["k"][:, :, :, c] = lv[None, :, None]
    x["k"][:, :, :, D - 1] = 0
    xd = {n: v.cuda() for n, v in x.items()}
    base = 1e30
    q2, ref_k = xd["q"].clone(), xd["k"].clone()
    binding().prologue(q=q2, k=ref_k, base=base)
    ref_out = binding().v2_fwd(q2, ref_k, xd["v"], xd["lam"])
    qr = q2
    rot = {"q": qr.cpu(), "k": ref_k.cpu()}
    for head in (0, Hq - 1):
        resc, stale = rc.v2_decisions(rot, 0, head, G)
        assert (resc > 0).sum() >= 64, np.bincount(resc)
        assert (stale > 4.0).sum() >= 64, stale.max()
    k = xd["k"].clone()
    out = binding().v2_fwd_rope(xd["q"], k, xd["v"], xd["lam"], base=base)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(k, ref_k)
    ref = oracle.v2_fwd(oracle.rope(x["q"], base=base), oracle.rope(x["k"], base=base), x["v"], x["lam"])
    assert_parity(out, ref, "bf16")


def test_fused_rope_argument_checks():
    lib = binding().lib()
    A = 0x10000
    f = lambda **kw: lib.diffattn_v2_fwd_rope(*[kw.get(n, dv) for n, dv in (  # noqa: E731
        ("q", A), ("k", A), ("v", A), ("lam", A), ("out", A), ("B", 1), ("T", 8), ("Hq", 4), ("Hkv", 2),
        ("D", 128), ("pos0", 0), ("base", 1e4), ("dtype", 1), ("stream", None))])
    assert f(out=None) == 1
    assert f(q=None) == 1
    assert f(T=0) == 2
    assert f(base=0.0) == 2
    assert f(Hkv=3) == 4                       # Hq not a multiple of Hkv
    assert f(D=32) == 3
    assert f(dtype=0) == 3                     # fp32 not supported here
    assert f(k=A + 4) == 5
    assert f(dtype=4) == 8


@pytest.mark.slow
def test_fused_rope_v2_prefill_workload_sampled():
    """The V2 prefill workload (B 8, T 4096, Hq 32, Hkv 8, D 128) through the
    fused call: the whole output equal to the two-call path, and sampled rows
    of two batch entries against the oracle."""
    s = inputs.WORKLOADS["v2_bf16_B8_T4096_Hq32_Hkv8_D128"]
    x = inputs.make_v2(s, seed=0, device="cuda")
    ref_out, ref_k = _two_call(x, 0)
    q0, k0 = x["q"].clone(), x["k"].clone()
    out = binding().v2_fwd_rope(x["q"], x["k"], x["v"], x["lam"])
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    assert torch.equal(x["k"], ref_k)
    assert torch.equal(x["q"], q0)
    P = s.Hq // 2
    r = np.random.default_rng(3)
    for b in (0, s.B - 1):
        ts = np.concatenate([[0, 127, 128, s.T - 1], r.integers(0, s.T, 12)])
        rows = [(t * P + int(r.integers(P))) for t in ts]
        ref = oracle.v2_fwd(oracle.rope(q0[b:b + 1].cpu()), oracle.rope(k0[b:b + 1].cpu()), x["v"][b:b + 1].cpu(),
                            x["lam"][b:b + 1].cpu(), rows=rows)
        got = out[b].reshape(s.T * P, s.D)[torch.as_tensor(rows, device="cuda")]
        assert_parity(got, ref, "bf16")
