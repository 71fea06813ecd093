"""GPU parity of the prologue kernel (rotary embedding of q and k in place,
V2 projected lambda logits) through the C ABI against the fp64 oracle.

Tolerances: the rotated q, k are rounded to the input dtype, so the bf16 bound
(max abs <= 2e-2, rel L2 <= 5e-3) and the fp32 bound (max abs <= 1e-4) of the
attention outputs apply; the lambda logits are fp32 sums of C products of
dtype inputs: |err| <= 1e-5 * sum_c |x_c w_c,i| + 1e-6 (fp32 accumulation).
"""
import numpy as np
import pytest
import torch

import oracle
from differential_attention_causal_gb300 import inputs

from test_gpu_parity import assert_parity, binding, built  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def _qk(B, T, Hq, Hk, D, dtype, seed):
    x = inputs.make_v2(inputs.V2Shape(B, T, Hq, Hk, D, dtype), seed=seed)
    return x["q"], x["k"]


def check_lam(got, x, w):
    ref = oracle.lambda_proj(x, w)
    scale = oracle.lambda_proj(np.abs(x.double().numpy()), np.abs(w.double().numpy()))
    got = got.double().cpu().numpy()
    assert np.isfinite(got).all()
    assert (np.abs(got - ref) <= 1e-5 * scale + 1e-6).all(), float(np.abs(got - ref).max())


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("B,T,Hq,Hk,D,pos0", [(2, 37, 4, 2, 128, 0), (1, 100, 8, 1, 64, 30000),
                                              (3, 5, 2, 2, 32, 7), (1, 64, 6, 0, 128, 123456)])
def test_rope(dtype, B, T, Hq, Hk, D, pos0):
    q, k = _qk(B, T, Hq, max(Hk, 1), D, dtype, seed=T + D)
    qd, kd = q.cuda(), k.cuda()
    binding().prologue(q=qd, k=kd if Hk else None, pos0=pos0)
    assert binding().last_launch_count() == 1
    assert_parity(qd, oracle.rope(q, pos0=pos0), dtype)
    if Hk:
        assert_parity(kd, oracle.rope(k, pos0=pos0), dtype)
    else:
        assert torch.equal(kd.cpu(), k)   # untouched


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_rope_and_lambda_in_one_call(dtype):
    B, T, Hq, Hk, D, C, P = 2, 77, 8, 2, 128, 512, 16
    q, k = _qk(B, T, Hq, Hk, D, dtype, seed=5)
    lp = inputs.make_lambda_proj(B, T, C, P, dtype, seed=5)
    qd, kd, xd, wd = q.cuda(), k.cuda(), lp["x"].cuda(), lp["w_lam"].cuda()
    lam = binding().prologue(q=qd, k=kd, pos0=11, x=xd, w_lam=wd)
    assert_parity(qd, oracle.rope(q, pos0=11), dtype)
    assert_parity(kd, oracle.rope(k, pos0=11), dtype)
    check_lam(lam, lp["x"], lp["w_lam"])
    assert binding().device_error() == 0


@pytest.mark.parametrize("C,P", [(128, 8), (2048, 64), (896, 24), (192, 16), (64, 8), (1024, 64), (2048, 16)])
def test_lambda_only(C, P):
    lp = inputs.make_lambda_proj(3, 41, C, P, "bf16", seed=C)
    lam = binding().prologue(x=lp["x"].cuda(), w_lam=lp["w_lam"].cuda())
    check_lam(lam, lp["x"], lp["w_lam"])


def test_prologue_argument_checks():
    lib = binding().lib()
    A = 0x10000
    f = lambda **kw: lib.diffattn_prologue(*[kw.get(n, dv) for n, dv in (  # noqa: E731
        ("q", A), ("k", A), ("B", 1), ("T", 8), ("Hq", 2), ("Hk", 2), ("D", 64), ("pos0", 0), ("base", 1e4),
        ("x", None), ("w", None), ("lam", None), ("C", 0), ("P", 0), ("dtype", 1), ("stream", None))])
    assert f(q=None) == 1
    assert f(x=A) == 1                         # x without w / lam
    assert f(D=96) == 3
    assert f(x=A, w=A, lam=A, C=64, P=12) == 3   # P not a multiple of 8
    assert f(x=A, w=A, lam=A, C=96, P=16) == 3   # C not a multiple of 64
    assert f(q=A + 8) == 5
    assert f(base=0.0) == 2
    assert f(dtype=4) == 8


@pytest.mark.slow
def test_prologue_v2_prefill_workload_sampled():
    """The V2 prefill workload's q (8 x 4096 x 32 x 128) and k (8 x 4096 x 8 x 128),
    x (8 x 4096 x 2048) and w (2048 x 16): sampled rows against the oracle."""
    s = inputs.WORKLOADS["v2_bf16_B8_T4096_Hq32_Hkv8_D128"]
    x = inputs.make_v2(s, seed=0, device="cuda")
    lp = inputs.make_lambda_proj(s.B, s.T, (s.Hq // 2) * s.D, s.Hq // 2, "bf16", seed=0, device="cuda")
    q0, k0 = x["q"].clone(), x["k"].clone()
    lam = binding().prologue(q=x["q"], k=x["k"], x=lp["x"], w_lam=lp["w_lam"])
    r = np.random.default_rng(9)
    for b, t in [(0, 0), (s.B - 1, s.T - 1)] + [(int(r.integers(s.B)), int(r.integers(s.T))) for _ in range(6)]:
        assert_parity(x["q"][b:b + 1, t:t + 1], oracle.rope(q0[b:b + 1, t:t + 1], pos0=t), "bf16")
        assert_parity(x["k"][b:b + 1, t:t + 1], oracle.rope(k0[b:b + 1, t:t + 1], pos0=t), "bf16")
        check_lam(lam[b:b + 1, t:t + 1], lp["x"][b:b + 1, t:t + 1].cpu(), lp["w_lam"].cpu())
