"""GPU parity for the decode calls beyond the all-L V2 decode: a cache length
per sequence (V2), and DIFF V1 decode (all L rows or per-sequence lengths),
each through the C ABI against the fp64 oracle.

Cache rows at and past a sequence's length are overwritten with NaN before the
call: the definition never reads them, so neither may the kernels (the oracle
is pinned to ignore them as well).  Tolerances as for every bf16 / fp32 path.
"""
import numpy as np
import pytest
import torch

import oracle
from differential_attention_causal_gb300 import inputs

from test_gpu_parity import assert_parity, binding, built, to_dev  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def poison_past_lengths(lens, *caches):
    for b, n in enumerate(lens.tolist()):
        for c in caches:
            c[b, n:] = float("nan")


def lens_with_edges(B, L, seed):
    """Seeded lengths in 1..L that include the unit edges 1, 63, 64, 65 and L."""
    r = np.random.default_rng(seed)
    base = [1, min(63, L), min(64, L), min(65, L), L]
    vals = base + list(r.integers(1, L + 1, max(0, B - len(base))))
    return torch.tensor(vals[:B], dtype=torch.int32)


# ------------------------------------------------------- V2, per-sequence lengths

@pytest.mark.parametrize("B,L,Hq,Hkv,D", [(5, 1000, 16, 2, 128), (7, 200, 8, 2, 128), (6, 777, 16, 4, 64),
                                          (2, 65, 4, 2, 128), (40, 300, 16, 8, 128), (3, 4000, 8, 1, 128)])
def test_decode_varlen_bf16(B, L, Hq, Hkv, D):
    x = inputs.make_decode(inputs.DecodeShape(B, L, Hq, Hkv, D, "bf16"), seed=B + L)
    lens = lens_with_edges(B, L, seed=L)
    poison_past_lengths(lens, x["k_cache"], x["v_cache"])
    xd = to_dev(x)
    y = binding().v2_decode_varlen(xd["q"], xd["k_cache"], xd["v_cache"], xd["lam"], lens.cuda())
    assert binding().last_launch_count() == 3
    ref = oracle.v2_decode(x["q"], x["k_cache"], x["v_cache"], x["lam"], lens=lens)
    assert_parity(y, ref, "bf16")


def test_decode_varlen_all_full_equals_uniform_call():
    """Every length = L gives the same result as the all-L call (same split)."""
    B, L, Hq, Hkv, D = 4, 900, 16, 4, 128
    xd = to_dev(inputs.make_decode(inputs.DecodeShape(B, L, Hq, Hkv, D, "bf16"), seed=5))
    a = binding().v2_decode(xd["q"], xd["k_cache"], xd["v_cache"], xd["lam"])
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    b = binding().v2_decode_varlen(xd["q"], xd["k_cache"], xd["v_cache"], xd["lam"], lens)
    assert torch.equal(a, b)


def test_decode_varlen_fp32():
    B, L = 5, 300
    x = inputs.make_decode(inputs.DecodeShape(B, L, 8, 2, 128, "fp32"), seed=12)
    lens = lens_with_edges(B, L, seed=3)
    poison_past_lengths(lens, x["k_cache"], x["v_cache"])
    xd = to_dev(x)
    y = binding().v2_decode_varlen(xd["q"], xd["k_cache"], xd["v_cache"], xd["lam"], lens.cuda())
    assert_parity(y, oracle.v2_decode(x["q"], x["k_cache"], x["v_cache"], x["lam"], lens=lens), "fp32")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_decode_length_out_of_range_is_clamped_and_reported(dtype):
    """Lengths 0 and L + 5 are clamped to 1 and L by the kernels' own checks and
    the device error word records it (DA_ERR_BAD_LENGTH, bit 4)."""
    B, L = 3, 200
    x = inputs.make_decode(inputs.DecodeShape(B, L, 8, 2, 128, dtype), seed=21)
    xd = to_dev(x)
    bad = torch.tensor([0, L + 5, 77], dtype=torch.int32)
    y = binding().v2_decode_varlen(xd["q"], xd["k_cache"], xd["v_cache"], xd["lam"], bad.cuda())
    assert binding().device_error() == 4
    ref = oracle.v2_decode(x["q"], x["k_cache"], x["v_cache"], x["lam"], lens=np.array([1, L, 77]))
    assert_parity(y, ref, dtype)


def test_decode_varlen_argument_checks():
    bd = binding()
    xd = to_dev(inputs.make_decode(inputs.DecodeShape(2, 100, 8, 2, 128, "bf16"), seed=0))
    with pytest.raises(ValueError):
        bd.v2_decode_varlen(xd["q"], xd["k_cache"], xd["v_cache"], xd["lam"],
                            torch.tensor([5, 6], dtype=torch.int64, device="cuda"))
    out = torch.empty((2, 4, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(bd.decode_workspace_size(2, 100, 8, 2, 128), dtype=torch.uint8, device="cuda")
    rc = bd.lib().diffattn_v2_decode_varlen(xd["q"].data_ptr(), xd["k_cache"].data_ptr(), xd["v_cache"].data_ptr(),
                                            xd["lam"].data_ptr(), None, out.data_ptr(), ws.data_ptr(), ws.numel(),
                                            2, 100, 8, 2, 128, 1, None)
    assert rc == 1   # DA_ERR_NULL_PTR: lengths are required by this entry point


@pytest.mark.slow
def test_decode_varlen_full_workload_sampled():
    """B=64, L=32768 allocated rows, 64 query heads, 8 kv heads, D=128, lengths uniform
    on 1..L: sampled (b, pair) rows, rows past each length set to NaN."""
    s = inputs.WORKLOADS["v2_decode_varlen_bf16_B64_L32768_Hq64_Hkv8_D128"]
    x = inputs.make_decode(s, seed=0, device="cuda")
    lens = x["cache_lens"]
    poison_past_lengths(lens, x["k_cache"], x["v_cache"])
    y = binding().v2_decode_varlen(x["q"], x["k_cache"], x["v_cache"], x["lam"], lens)
    P = s.Hq // 2
    rng = np.random.default_rng(4)
    rows = sorted(set([0, P - 1, s.B * P - 1] + list(rng.integers(0, s.B * P, 10))))
    lens_h = lens.cpu().numpy()
    for (qs, ks, vs, ls, local), rid in zip(oracle.decode_gather(x["q"], x["k_cache"], x["v_cache"], x["lam"], rows),
                                           rows):
        n = int(lens_h[rid // P])
        ref = oracle.v2_decode(qs, ks[:, :n], vs[:, :n], ls, rows=[local])
        assert_parity(y.reshape(-1, s.D)[rid:rid + 1], ref, "bf16")
    del x
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ V1 decode

def run_v1_decode(xd, lens=None):
    return binding().v1_decode(xd["q1"], xd["q2"], xd["k1_cache"], xd["k2_cache"], xd["v_cache"], xd["lam_q1"],
                               xd["lam_k1"], xd["lam_q2"], xd["lam_k2"], xd["layer_index"], cache_lens=lens)


def oracle_v1_decode(x, lens=None, rows=None):
    return oracle.v1_decode(x["q1"], x["q2"], x["k1_cache"], x["k2_cache"], x["v_cache"], x["lam_q1"],
                            x["lam_k1"], x["lam_q2"], x["lam_k2"], x["layer_index"], lens=lens, rows=rows)


@pytest.mark.parametrize("B,L,H,d,varlen", [(3, 1000, 4, 64, False), (2, 1, 2, 128, False), (1, 5000, 2, 128, False),
                                            (4, 777, 3, 128, True), (5, 130, 16, 64, True), (9, 64, 12, 128, True),
                                            (2, 2049, 16, 64, False), (3, 500, 4, 32, False), (4, 300, 3, 32, True)])
def test_v1_decode_bf16(B, L, H, d, varlen):
    x = inputs.make_v1_decode(inputs.V1DecodeShape(B, L, H, d, 12, "bf16"), seed=B * 7 + L)
    lens = None
    if varlen:
        lens = lens_with_edges(B, L, seed=B)
        poison_past_lengths(lens, x["k1_cache"], x["k2_cache"], x["v_cache"])
    xd = to_dev(x)
    y = run_v1_decode(xd, None if lens is None else lens.cuda())
    assert binding().last_launch_count() == (3 if varlen else 2)
    assert_parity(y, oracle_v1_decode(x, lens=lens), "bf16")


@pytest.mark.parametrize("d,varlen", [(32, False), (64, True), (128, False)])
def test_v1_decode_fp32(d, varlen):
    B, L, H = 3, 257, 2
    x = inputs.make_v1_decode(inputs.V1DecodeShape(B, L, H, d, 1, "fp32"), seed=d)
    lens = None
    if varlen:
        lens = lens_with_edges(B, L, seed=d)
        poison_past_lengths(lens, x["k1_cache"], x["k2_cache"], x["v_cache"])
    xd = to_dev(x)
    y = run_v1_decode(xd, None if lens is None else lens.cuda())
    assert_parity(y, oracle_v1_decode(x, lens=lens), "fp32")


@pytest.mark.parametrize("d", [64, 128])
def test_v1_decode_matches_last_prefill_row(d):
    """V1 decode of the last token equals the last row of the V1 prefill on the same rows."""
    B, T, H = 2, 300, 3
    x = inputs.make_v1(inputs.V1Shape(B, T, H, d, 5, "bf16"), seed=d + 1)
    xd = to_dev(x)
    pre = binding().v1_fwd(xd["q1"], xd["q2"], xd["k1"], xd["k2"], xd["v"], xd["lam_q1"], xd["lam_k1"],
                           xd["lam_q2"], xd["lam_k2"], 5)
    dec_in = {"q1": xd["q1"][:, -1].contiguous(), "q2": xd["q2"][:, -1].contiguous(),
              "k1_cache": xd["k1"].contiguous(), "k2_cache": xd["k2"].contiguous(), "v_cache": xd["v"],
              "lam_q1": xd["lam_q1"], "lam_k1": xd["lam_k1"], "lam_q2": xd["lam_q2"], "lam_k2": xd["lam_k2"],
              "layer_index": 5}
    dec = run_v1_decode(dec_in)
    ref = oracle.v1_fwd(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"], x["lam_q2"],
                        x["lam_k2"], 5)[:, -1]
    assert_parity(dec, ref, "bf16")
    assert_parity(pre[:, -1], ref, "bf16")


def test_v1_decode_argument_checks():
    bd = binding()
    xd = to_dev(inputs.make_v1_decode(inputs.V1DecodeShape(2, 100, 2, 64, 0, "bf16"), seed=0))
    assert bd.v1_decode_workspace_size(2, 100, 2, 64) > 0
    assert bd.v1_decode_workspace_size(2, 100, 2, 32) > 0    # d = 32: the d = 64 kernels on zero-filled boxes
    assert bd.v1_decode_workspace_size(2, 100, 2, 48) == 0
    # the size covers per-sequence lengths (the larger need): 16 bytes less fails that call
    small = torch.empty(bd.v1_decode_workspace_size(2, 100, 2, 64) - 16, dtype=torch.uint8, device="cuda")
    lens = torch.tensor([100, 7], dtype=torch.int32, device="cuda")
    for kw in ({"cache_lens": lens, "workspace": small},
               {"workspace": torch.empty(64, dtype=torch.uint8, device="cuda")}):
        with pytest.raises(bd.DiffAttnError) as e:
            bd.v1_decode(xd["q1"], xd["q2"], xd["k1_cache"], xd["k2_cache"], xd["v_cache"], xd["lam_q1"],
                         xd["lam_k1"], xd["lam_q2"], xd["lam_k2"], 0, **kw)
        assert e.value.code == 6


@pytest.mark.slow
@pytest.mark.parametrize("varlen", [False, True])
def test_v1_decode_full_workload_sampled(varlen):
    """B=32, L=16384, H=12, d=128 (6.4 GB of cache): sampled (b, h) rows, in the
    launch configuration the bench uses; with varlen, seeded lengths on 1..L."""
    s = inputs.WORKLOADS["v1_decode_bf16_B32_L16384_H12_d128"]
    if varlen:
        s = inputs.V1DecodeShape(s.B, s.L, s.H, s.d, s.layer_index, s.dtype, True)
    x = inputs.make_v1_decode(s, seed=0, device="cuda")
    lens = x.get("cache_lens")
    if lens is not None:
        poison_past_lengths(lens, x["k1_cache"], x["k2_cache"], x["v_cache"])
    y = run_v1_decode(x, lens)
    rng = np.random.default_rng(6)
    rows = sorted(set([0, s.H - 1, s.B * s.H - 1] + list(rng.integers(0, s.B * s.H, 6))))
    for rid in rows:
        b, h = rid // s.H, rid % s.H
        n = s.L if lens is None else int(lens[b])
        sl = {"q1": x["q1"][b:b + 1, h:h + 1], "q2": x["q2"][b:b + 1, h:h + 1],
              "k1_cache": x["k1_cache"][b:b + 1, :n, h:h + 1], "k2_cache": x["k2_cache"][b:b + 1, :n, h:h + 1],
              "v_cache": x["v_cache"][b:b + 1, :n, h:h + 1]}
        sl.update({k: x[k] for k in ("lam_q1", "lam_k1", "lam_q2", "lam_k2", "layer_index")})
        ref = oracle_v1_decode(sl)
        assert_parity(y.reshape(-1, 2 * s.d)[rid:rid + 1], ref, "bf16")
    del x
    torch.cuda.empty_cache()
