"""Stand-ins for a device memory checker (none runs on this system):

  * the debug build (libdiffattn_debug.so, -DDA_DEBUG_CHECKS), whose kernels
    test every index they write through against the extent of its tensor,
    workspace, shared-memory tile or TMEM allocation and record a failure in
    the stream's error word instead of writing;
  * canary regions around caller-provided outputs, checked after the call.

Every entry point runs on small odd shapes (ragged tails, several tiles).
The debug build must record nothing and give the release build's outputs bit
for bit (the checks only guard the writes), and no write may reach the
canaries.  A self-test shows the check itself fires (an index one past the
end of a buffer, the write skipped).
"""
import pytest
import torch

from differential_attention_causal_gb300 import inputs

from test_gpu_parity import binding, built  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu

LAYER = 3


@pytest.fixture(scope="module", autouse=True)
def debug_lib(built):  # noqa: F811
    from differential_attention_causal_gb300 import build as b
    b.build(debug=True)
    yield
    binding().use_library(False)


def _v1(B, T, H, d, dtype="bf16", seed=0):
    x = inputs.make_v1(inputs.V1Shape(B, T, H, d, LAYER, dtype), seed=seed, device="cuda")
    return x, (x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"], x["lam_q2"], x["lam_k2"])


def _v2(B, T, Hq, Hkv, D, dtype="bf16", seed=0):
    return inputs.make_v2(inputs.V2Shape(B, T, Hq, Hkv, D, dtype), seed=seed, device="cuda")


def case_v1(B, T, H, d, dtype):
    _, a = _v1(B, T, H, d, dtype, seed=T)
    return lambda: {"out": binding().v1_fwd(*a, LAYER)}


def case_v2(B, T, Hq, Hkv, D, dtype):
    x = _v2(B, T, Hq, Hkv, D, dtype, seed=T)
    return lambda: {"out": binding().v2_fwd(x["q"], x["k"], x["v"], x["lam"])}


def case_v2_rope(B, T, Hq, Hkv, D):
    x = _v2(B, T, Hq, Hkv, D, seed=T + 1)

    def run():
        k = x["k"].clone()
        out = binding().v2_fwd_rope(x["q"], k, x["v"], x["lam"], pos0=17)
        return {"out": out, "k": k}
    return run


def case_paired(B, T, H, D):
    x = inputs.make_paired(inputs.PairedShape(B, T, H, D), seed=T, device="cuda")
    return lambda: {"out": binding().paired_fwd(x["q"], x["k"], x["v"])}


def case_v2_decode(B, L, Hq, Hkv, D, varlen):
    x = inputs.make_decode(inputs.DecodeShape(B, L, Hq, Hkv, D, varlen=varlen), seed=L, device="cuda")
    if varlen:
        return lambda: {"out": binding().v2_decode_varlen(x["q"], x["k_cache"], x["v_cache"], x["lam"],
                                                          x["cache_lens"])}
    return lambda: {"out": binding().v2_decode(x["q"], x["k_cache"], x["v_cache"], x["lam"])}


def case_v1_decode(B, L, H, d, varlen):
    x = inputs.make_v1_decode(inputs.V1DecodeShape(B, L, H, d, LAYER, varlen=varlen), seed=L, device="cuda")
    kw = {"cache_lens": x["cache_lens"]} if varlen else {}
    return lambda: {"out": binding().v1_decode(x["q1"], x["q2"], x["k1_cache"], x["k2_cache"], x["v_cache"],
                                               x["lam_q1"], x["lam_k1"], x["lam_q2"], x["lam_k2"], LAYER, **kw)}


def case_prologue(dtype):
    B, T, Hq, Hk, D, C, P = 2, 77, 8, 2, 128, 512, 16
    x = _v2(B, T, Hq, Hk, D, dtype, seed=5)
    lp = inputs.make_lambda_proj(B, T, C, P, dtype, seed=5, device="cuda")

    def run():
        q, k = x["q"].clone(), x["k"].clone()
        lam = binding().prologue(q=q, k=k, pos0=11, x=lp["x"], w_lam=lp["w_lam"])
        return {"q": q, "k": k, "lam": lam}
    return run


def case_v1_train(B, T, H, d, dtype):
    x, a = _v1(B, T, H, d, dtype, seed=T + 2)
    dout = inputs.make_grad_out((B, T, H, 2 * d), dtype, seed=T, device="cuda")

    def run():
        out, saved = binding().v1_fwd_train(*a, LAYER)
        g = binding().v1_bwd(*a, LAYER, dout, saved)
        return {"out": out, **g}
    return run


def case_v2_train(B, T, Hq, Hkv, D, dtype):
    x = _v2(B, T, Hq, Hkv, D, dtype, seed=T + 3)
    dout = inputs.make_grad_out((B, T, Hq // 2, D), dtype, seed=T, device="cuda")

    def run():
        out, saved = binding().v2_fwd_train(x["q"], x["k"], x["v"], x["lam"])
        g = binding().v2_bwd(x["q"], x["k"], x["v"], x["lam"], dout, saved)
        return {"out": out, **g}
    return run


CASES = {
    "v1_bf16_d64": lambda: case_v1(2, 300, 3, 64, "bf16"),
    "v1_bf16_d32": lambda: case_v1(1, 130, 2, 32, "bf16"),
    "v1_bf16_d128": lambda: case_v1(1, 200, 2, 128, "bf16"),
    "v1_fp32_d64": lambda: case_v1(1, 70, 2, 64, "fp32"),
    "v2_bf16_D128": lambda: case_v2(2, 257, 8, 2, 128, "bf16"),
    "v2_bf16_D64": lambda: case_v2(1, 130, 4, 2, 64, "bf16"),
    "v2_fp32_D64": lambda: case_v2(1, 70, 4, 2, 64, "fp32"),
    "v2_rope_D128": lambda: case_v2_rope(2, 257, 8, 2, 128),
    "paired_D64": lambda: case_paired(1, 150, 4, 64),
    "v2_decode": lambda: case_v2_decode(3, 777, 8, 2, 128, False),
    "v2_decode_varlen": lambda: case_v2_decode(3, 777, 8, 2, 128, True),
    "v1_decode": lambda: case_v1_decode(2, 500, 2, 64, False),
    "v1_decode_varlen": lambda: case_v1_decode(2, 500, 2, 64, True),
    "prologue_bf16": lambda: case_prologue("bf16"),
    "prologue_fp32": lambda: case_prologue("fp32"),
    "v1_train_bf16_d64": lambda: case_v1_train(1, 200, 2, 64, "bf16"),
    "v1_train_bf16_d128": lambda: case_v1_train(1, 300, 2, 128, "bf16"),
    "v1_train_fp32_d64": lambda: case_v1_train(1, 70, 2, 64, "fp32"),
    "v2_train_bf16_D128": lambda: case_v2_train(1, 200, 4, 2, 128, "bf16"),
    "v2_train_fp32_D64": lambda: case_v2_train(1, 70, 4, 2, 64, "fp32"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_debug_build_records_nothing_and_matches_release(name):
    bd = binding()
    run = CASES[name]()
    bd.use_library(False)
    ref = run()
    assert bd.stream_error() == 0
    bd.use_library(True)
    try:
        assert bd.debug_checks()
        got = run()
        word = bd.stream_error()
    finally:
        bd.use_library(False)
    assert word == 0, f"bounds check failed: error word {word:#x}"
    for k, r in ref.items():
        assert torch.equal(got[k], r), k


def test_bounds_selftest_both_builds():
    bd = binding()
    assert bd.selftest_bounds() == 0 and not bd.debug_checks()
    bd.use_library(True)
    try:
        assert bd.debug_checks()
        assert bd.selftest_bounds() == 8       # the bounds bit, recorded and cleared again
        assert bd.stream_error() == 0
    finally:
        bd.use_library(False)


# ---------------------------------------------------------------- canaries

GUARD = 64   # elements on each side (128 / 256 bytes: keeps 16-byte alignment)


def guarded(shape, dtype):
    """An output tensor inside a buffer whose margins hold a fixed bit pattern."""
    n = 1
    for s in shape:
        n *= s
    buf = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
    bits = buf.view(torch.int16 if dtype == torch.bfloat16 else torch.int32)
    bits.fill_(0x5A5A if dtype == torch.bfloat16 else 0x5A5A5A5A)
    return buf, buf[GUARD:GUARD + n].view(shape)


def margins_intact(buf):
    bits = buf.view(torch.int16 if buf.dtype == torch.bfloat16 else torch.int32)
    pat = 0x5A5A if buf.dtype == torch.bfloat16 else 0x5A5A5A5A
    return bool((bits[:GUARD] == pat).all()) and bool((bits[-GUARD:] == pat).all())


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_canaries_around_forward_outputs(dtype):
    bd = binding()
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    # V1, ragged T, both supported head dims of the dtype's fast path
    for (B, T, H, d) in ((2, 300, 3, 64), (1, 130, 2, 32), (1, 200, 2, 128)):
        _, a = _v1(B, T, H, d, dtype, seed=B + T)
        buf, out = guarded((B, T, H, 2 * d), dt)
        bd.v1_fwd(*a, LAYER, out=out)
        torch.cuda.synchronize()
        assert margins_intact(buf), ("v1", B, T, H, d)
    for (B, T, Hq, Hkv, D) in ((2, 257, 8, 2, 128), (1, 130, 4, 2, 64)):
        x = _v2(B, T, Hq, Hkv, D, dtype, seed=T)
        buf, out = guarded((B, T, Hq // 2, D), dt)
        bd.v2_fwd(x["q"], x["k"], x["v"], x["lam"], out=out)
        torch.cuda.synchronize()
        assert margins_intact(buf), ("v2", B, T, Hq, Hkv, D)
    assert bd.device_error() == 0


def test_canaries_around_bf16_only_outputs():
    bd = binding()
    dt = torch.bfloat16
    x = inputs.make_paired(inputs.PairedShape(1, 150, 4, 64), seed=1, device="cuda")
    buf, out = guarded(tuple(x["q"].shape), dt)
    bd.paired_fwd(x["q"], x["k"], x["v"], out=out)
    torch.cuda.synchronize()
    assert margins_intact(buf), "paired"
    x = _v2(2, 257, 8, 2, 128, seed=4)
    buf, out = guarded((2, 257, 4, 128), dt)
    bd.v2_fwd_rope(x["q"], x["k"].clone(), x["v"], x["lam"], out=out)
    torch.cuda.synchronize()
    assert margins_intact(buf), "v2_fwd_rope"
    for varlen in (False, True):
        x = inputs.make_decode(inputs.DecodeShape(3, 777, 8, 2, 128, varlen=varlen), seed=2, device="cuda")
        buf, out = guarded((3, 4, 128), dt)
        if varlen:
            bd.v2_decode_varlen(x["q"], x["k_cache"], x["v_cache"], x["lam"], x["cache_lens"], out=out)
        else:
            bd.v2_decode(x["q"], x["k_cache"], x["v_cache"], x["lam"], out=out)
        torch.cuda.synchronize()
        assert margins_intact(buf), ("v2_decode", varlen)
        x = inputs.make_v1_decode(inputs.V1DecodeShape(2, 500, 2, 64, LAYER, varlen=varlen), seed=3, device="cuda")
        buf, out = guarded((2, 2, 128), dt)
        kw = {"cache_lens": x["cache_lens"]} if varlen else {}
        bd.v1_decode(x["q1"], x["q2"], x["k1_cache"], x["k2_cache"], x["v_cache"], x["lam_q1"], x["lam_k1"],
                     x["lam_q2"], x["lam_k2"], LAYER, out=out, **kw)
        torch.cuda.synchronize()
        assert margins_intact(buf), ("v1_decode", varlen)
    assert bd.device_error() == 0
