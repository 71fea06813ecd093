"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerances (from the workload statement):
  fp32: max abs error <= 1e-4
  bf16: max abs error <= 2e-2 and relative L2 <= 5e-3
The oracle reads exactly the (rounded) values the GPU reads.  Small shapes are
compared element by element over every output; the full-size workloads are
compared on sampled rows (rows are independent by definition, so a sampled
row is checked exactly), in the same launch configuration the bench uses.
"""
import numpy as np
import pytest
import torch

import oracle
from differential_attention_causal_gb300 import inputs

pytestmark = pytest.mark.gpu

FP32_ATOL = 1e-4
BF16_ATOL, BF16_RL2 = 2e-2, 5e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    from differential_attention_causal_gb300 import build as b
    b.build()
    oracle.build()
    torch.cuda.set_device(0)
    yield


def binding():
    from differential_attention_causal_gb300 import binding as bd
    return bd


def assert_parity(got, ref, dtype):
    got = got.detach().float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    if dtype == "fp32":
        assert err <= FP32_ATOL, f"max abs {err:.3e}"
    else:
        rl2 = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert err <= BF16_ATOL and rl2 <= BF16_RL2, f"max abs {err:.3e}, rel L2 {rl2:.3e}"
    assert binding().device_error() == 0


def to_dev(x):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}


def run_v1(xd, layer, out=None):
    return binding().v1_fwd(xd["q1"], xd["q2"], xd["k1"], xd["k2"], xd["v"], xd["lam_q1"], xd["lam_k1"],
                            xd["lam_q2"], xd["lam_k2"], layer, out=out)


def oracle_v1(x, layer, rows=None):
    return oracle.v1_fwd(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"],
                         x["lam_q2"], x["lam_k2"], layer, rows=rows)


# ------------------------------------------------------------------- DIFF V1

def test_v1_fp32_tiny_workload():
    """B=1, T=64, 2 diff heads, d=32, dv=64, layer_index=1, seed 0."""
    s = inputs.WORKLOADS["v1_fp32_B1_T64_H2_d32"]
    x = inputs.make_v1(s, seed=0)
    y = run_v1(to_dev(x), s.layer_index)
    assert_parity(y, oracle_v1(x, s.layer_index), "fp32")


@pytest.mark.parametrize("B,T,H,d,layer", [(2, 77, 3, 64, 5), (1, 130, 1, 128, 27), (1, 1, 2, 32, 0)])
def test_v1_fp32_shapes(B, T, H, d, layer):
    s = inputs.V1Shape(B, T, H, d, layer, "fp32")
    x = inputs.make_v1(s, seed=3)
    y = run_v1(to_dev(x), layer)
    assert_parity(y, oracle_v1(x, layer), "fp32")


@pytest.mark.parametrize("B,T,H,layer", [(2, 300, 3, 4), (1, 1, 1, 0), (1, 127, 2, 12), (1, 128, 2, 12),
                                         (1, 129, 2, 12), (3, 256, 2, 1)])
def test_v1_bf16_d64(B, T, H, layer):
    s = inputs.V1Shape(B, T, H, 64, layer, "bf16")
    x = inputs.make_v1(s, seed=B * 1000 + T)
    y = run_v1(to_dev(x), layer)
    assert_parity(y, oracle_v1(x, layer), "bf16")


@pytest.mark.parametrize("B,T,H,layer", [(2, 77, 3, 5), (1, 1, 1, 0), (1, 129, 2, 12), (2, 300, 2, 27)])
def test_v1_bf16_d32(B, T, H, layer):
    # d = 32 (dv = 64) runs the d = 64 kernel on q / k boxes zero-filled past column 32
    s = inputs.V1Shape(B, T, H, 32, layer, "bf16")
    x = inputs.make_v1(s, seed=B * 1000 + T + 32)
    y = run_v1(to_dev(x), layer)
    assert_parity(y, oracle_v1(x, layer), "bf16")
    assert binding().device_error() == 0


def test_v1_bf16_lambda_zero_and_separate_tensors():
    """lam = 0 (lq1 = lk1 = 0, lq2.lk2 = ln(1 + lam_init)); q1/q2/k1/k2 as separate tensors
    and a strided output view."""
    B, T, H, d, layer = 1, 200, 2, 64, 2
    s = inputs.V1Shape(B, T, H, d, layer, "bf16")
    x = inputs.make_v1(s, seed=11)
    lam_init = oracle.lambda_init(layer)
    x["lam_q1"] = torch.zeros(d)
    x["lam_k1"] = torch.zeros(d)
    x["lam_q2"] = torch.zeros(d)
    x["lam_q2"][0] = float(np.log1p(lam_init))
    x["lam_k2"] = torch.zeros(d)
    x["lam_k2"][0] = 1.0
    for n in ("q1", "q2", "k1", "k2"):
        x[n] = x[n].contiguous()
    xd = to_dev(x)
    big = torch.zeros((B, T, H + 1, 2 * d), dtype=torch.bfloat16, device="cuda")
    out = big[:, :, 1:]
    run_v1(xd, layer, out=out)
    assert_parity(out, oracle_v1(x, layer), "bf16")
    assert big[:, :, 0].abs().max().item() == 0.0   # nothing written outside the view


def test_v1_bf16_full_workload_sampled():
    """B=4, T=2048, 16 diff heads, d=64, dv=128, layer_index=12, seed 0: sampled rows."""
    s = inputs.WORKLOADS["v1_bf16_B4_T2048_H16_d64"]
    x = inputs.make_v1(s, seed=0)
    y = run_v1(to_dev(x), s.layer_index)
    rng = np.random.default_rng(0)
    ts = [0, 1, 2, 127, 128, 129, 1023, 1024, 2046, 2047]
    rows = [(b * s.T + t) * s.H + h for b in range(s.B) for h in range(s.H) for t in ts]
    rows += list(rng.integers(0, s.B * s.T * s.H, 400))
    rows = np.array(rows, dtype=np.int64)
    ref = oracle_v1(x, s.layer_index, rows=rows)
    assert_parity(y.reshape(-1, 2 * s.d)[torch.from_numpy(rows).cuda()], ref, "bf16")


@pytest.mark.parametrize("B,T,H,layer", [(2, 300, 2, 27), (1, 1, 1, 0), (1, 128, 2, 5), (1, 129, 1, 5),
                                         (1, 520, 3, 27)])
def test_v1_bf16_d128_two_pass(B, T, H, layer):
    """d = 128, dv = 256: the two-pass kernel (row statistics, then one combined PV)."""
    s = inputs.V1Shape(B, T, H, 128, layer, "bf16")
    x = inputs.make_v1(s, seed=7 * T + H)
    y = run_v1(to_dev(x), layer)
    assert_parity(y, oracle_v1(x, layer), "bf16")


def test_v1_bf16_d128_full_workload_sampled():
    """B=1, T=32768, 12 diff heads, d=128, dv=256, layer_index=27, seed 0: sampled rows."""
    s = inputs.WORKLOADS["v1_bf16_B1_T32768_H12_d128"]
    x = inputs.make_v1(s, seed=0)
    y = run_v1(to_dev(x), s.layer_index)
    rng = np.random.default_rng(5)
    ts = [0, 1, 127, 128, 16383, 32766, 32767]
    rows = [(t * s.H + h) for h in range(s.H) for t in ts]
    rows += list(rng.integers(0, s.T * s.H, 120))
    rows = np.array(rows, dtype=np.int64)
    ref = oracle_v1(x, s.layer_index, rows=rows)
    assert_parity(y.reshape(-1, 2 * s.d)[torch.from_numpy(rows).cuda()], ref, "bf16")


# ------------------------------------------------------------------- DIFF V2

@pytest.mark.parametrize("B,T,Hq,Hkv,D", [(2, 200, 8, 2, 128), (1, 129, 4, 2, 128), (1, 1, 8, 4, 128),
                                          (2, 150, 8, 1, 64), (1, 384, 16, 4, 128)])
def test_v2_bf16(B, T, Hq, Hkv, D):
    s = inputs.V2Shape(B, T, Hq, Hkv, D, "bf16")
    x = inputs.make_v2(s, seed=T + Hq)
    xd = to_dev(x)
    y = binding().v2_fwd(xd["q"], xd["k"], xd["v"], xd["lam"])
    assert_parity(y, oracle.v2_fwd(x["q"], x["k"], x["v"], x["lam"]), "bf16")


def test_v2_bf16_sigmoid_zero_is_plain_gqa_attention():
    s = inputs.V2Shape(1, 257, 8, 2, 128, "bf16")
    x = inputs.make_v2(s, seed=5)
    x["lam"] = torch.full_like(x["lam"], -1e4)
    xd = to_dev(x)
    y = binding().v2_fwd(xd["q"], xd["k"], xd["v"], xd["lam"])
    assert_parity(y, oracle.v2_fwd(x["q"], x["k"], x["v"], x["lam"]), "bf16")


@pytest.mark.parametrize("B,T,Hq,Hkv,D", [(2, 100, 8, 2, 128), (1, 33, 4, 1, 64)])
def test_v2_fp32(B, T, Hq, Hkv, D):
    s = inputs.V2Shape(B, T, Hq, Hkv, D, "fp32")
    x = inputs.make_v2(s, seed=7)
    xd = to_dev(x)
    y = binding().v2_fwd(xd["q"], xd["k"], xd["v"], xd["lam"])
    assert_parity(y, oracle.v2_fwd(x["q"], x["k"], x["v"], x["lam"]), "fp32")


def test_v2_bf16_full_workload_sampled():
    """B=8, T=4096, 32 query heads (16 pairs), 8 kv heads, D=128: sampled rows."""
    s = inputs.WORKLOADS["v2_bf16_B8_T4096_Hq32_Hkv8_D128"]
    x = inputs.make_v2(s, seed=0)
    xd = to_dev(x)
    y = binding().v2_fwd(xd["q"], xd["k"], xd["v"], xd["lam"])
    P = s.Hq // 2
    rng = np.random.default_rng(1)
    ts = [0, 1, 127, 128, 2047, 4095]
    rows = [(b * s.T + t) * P + i for b in range(s.B) for i in range(P) for t in ts]
    rows += list(rng.integers(0, s.B * s.T * P, 300))
    rows = np.array(rows, dtype=np.int64)
    ref = oracle.v2_fwd(x["q"], x["k"], x["v"], x["lam"], rows=rows)
    assert_parity(y.reshape(-1, s.D)[torch.from_numpy(rows).cuda()], ref, "bf16")


@pytest.mark.slow
def test_v2_bf16_beyond_2_31_elements():
    """B=2048, T=136 (a ragged last query tile), 64 query heads, 8 kv heads, D=128:
    q holds 2^31 + 2^27 elements (4.6 GB), past what a 32-bit element offset
    reaches; sampled rows of the first and last batch entries against the oracle
    (inputs drawn on the device)."""
    s = inputs.V2Shape(2048, 136, 64, 8, 128, "bf16")
    assert s.B * s.T * s.Hq * s.D > 2 ** 31
    xd = inputs.make_v2(s, seed=3, device="cuda")
    y = binding().v2_fwd(xd["q"], xd["k"], xd["v"], xd["lam"])
    assert binding().device_error() == 0
    P = s.Hq // 2
    rows = np.array([t * P + i for t in (0, 1, 127, 128, 135) for i in range(P)], dtype=np.int64)
    for b in (0, 1, s.B - 2, s.B - 1):
        xb = {n: xd[n][b:b + 1].contiguous().cpu() for n in ("q", "k", "v", "lam")}
        ref = oracle.v2_fwd(xb["q"], xb["k"], xb["v"], xb["lam"], rows=rows)
        assert_parity(y[b].reshape(-1, s.D)[torch.from_numpy(rows).cuda()], ref, "bf16")


@pytest.mark.slow
def test_v1_bf16_beyond_2_31_elements():
    """B=2048, T=136, 64 diff heads, d=64: q, k (B, T, 2H, d) and v, out (B, T, H, 2d)
    each hold 2^31 + 2^27 elements (4.6 GB); sampled rows of the first and last
    batch entries against the oracle (inputs drawn on the device)."""
    s = inputs.V1Shape(2048, 136, 64, 64, 5, "bf16")
    assert s.B * s.T * 2 * s.H * s.d > 2 ** 31
    xd = inputs.make_v1(s, seed=4, device="cuda")
    y = run_v1(xd, s.layer_index)
    assert binding().device_error() == 0
    rows = np.array([t * s.H + h for t in (0, 1, 127, 128, 135) for h in range(s.H)], dtype=np.int64)
    for b in (0, 1, s.B - 2, s.B - 1):
        xb = {n: (xd[n][b:b + 1].contiguous().cpu() if n in ("q1", "q2", "k1", "k2", "v") else xd[n].cpu())
              for n in ("q1", "q2", "k1", "k2", "v", "lam_q1", "lam_k1", "lam_q2", "lam_k2")}
        ref = oracle_v1(xb, s.layer_index, rows=rows)
        assert_parity(y[b].reshape(-1, 2 * s.d)[torch.from_numpy(rows).cuda()], ref, "bf16")


@pytest.mark.slow
def test_v1_bf16_d128_beyond_2_31_elements():
    """The two-pass kernel (d=128, dv=256) with B=2048, T=136, 32 heads: q, k
    (B, T, 2H, d) and v, out (B, T, H, 2d) hold 2^31 + 2^27 elements each;
    sampled rows of the first and last batch entries against the oracle."""
    s = inputs.V1Shape(2048, 136, 32, 128, 27, "bf16")
    assert s.B * s.T * 2 * s.H * s.d > 2 ** 31
    xd = inputs.make_v1(s, seed=8, device="cuda")
    y = run_v1(xd, s.layer_index)
    assert binding().device_error() == 0
    rows = np.array([t * s.H + h for t in (0, 1, 127, 128, 135) for h in range(s.H)], dtype=np.int64)
    for b in (0, s.B - 1):
        xb = {n: (xd[n][b:b + 1].contiguous().cpu() if n in ("q1", "q2", "k1", "k2", "v") else xd[n].cpu())
              for n in ("q1", "q2", "k1", "k2", "v", "lam_q1", "lam_k1", "lam_q2", "lam_k2")}
        ref = oracle_v1(xb, s.layer_index, rows=rows)
        assert_parity(y[b].reshape(-1, 2 * s.d)[torch.from_numpy(rows).cuda()], ref, "bf16")


# ------------------------------------------------------------ DIFF V2 decode

@pytest.mark.parametrize("B,L,Hq,Hkv,D", [(3, 1000, 16, 2, 128), (1, 1, 8, 1, 128), (2, 63, 8, 2, 128),
                                          (2, 64, 8, 2, 128), (2, 65, 4, 2, 128), (4, 777, 16, 4, 64),
                                          (1, 5000, 4, 2, 128), (40, 130, 16, 8, 128)])
def test_decode_bf16(B, L, Hq, Hkv, D):
    s = inputs.DecodeShape(B, L, Hq, Hkv, D, "bf16")
    x = inputs.make_decode(s, seed=L + B)
    xd = to_dev(x)
    y = binding().v2_decode(xd["q"], xd["k_cache"], xd["v_cache"], xd["lam"])
    assert binding().last_launch_count() == 2
    assert_parity(y, oracle.v2_decode(x["q"], x["k_cache"], x["v_cache"], x["lam"]), "bf16")


def test_decode_matches_last_prefill_row():
    """Decode of the last token equals the last row of a V2 prefill on the same K/V."""
    B, T, Hq, Hkv, D = 2, 300, 8, 2, 128
    x = inputs.make_v2(inputs.V2Shape(B, T, Hq, Hkv, D, "bf16"), seed=9)
    xd = to_dev(x)
    pre = binding().v2_fwd(xd["q"], xd["k"], xd["v"], xd["lam"])
    dec = binding().v2_decode(xd["q"][:, -1].contiguous(), xd["k"], xd["v"], xd["lam"][:, -1].contiguous())
    ref = oracle.v2_decode(x["q"][:, -1], x["k"], x["v"], x["lam"][:, -1])
    assert_parity(dec, ref, "bf16")
    assert_parity(pre[:, -1], ref, "bf16")


def test_decode_fp32():
    s = inputs.DecodeShape(2, 500, 8, 2, 128, "fp32")
    x = inputs.make_decode(s, seed=4)
    xd = to_dev(x)
    y = binding().v2_decode(xd["q"], xd["k_cache"], xd["v_cache"], xd["lam"])
    assert_parity(y, oracle.v2_decode(x["q"], x["k_cache"], x["v_cache"], x["lam"]), "fp32")


def test_decode_workspace_checks():
    bd = binding()
    s = inputs.DecodeShape(2, 100, 8, 2, 128, "bf16")
    xd = to_dev(inputs.make_decode(s, seed=0))
    need = bd.decode_workspace_size(2, 100, 8, 2, 128)
    assert need > 0
    # the size covers per-sequence lengths (the larger need): 16 bytes less fails that call
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    lens = torch.tensor([100, 3], dtype=torch.int32, device="cuda")
    with pytest.raises(bd.DiffAttnError) as e:
        bd.v2_decode_varlen(xd["q"], xd["k_cache"], xd["v_cache"], xd["lam"], lens, workspace=small)
    assert e.value.code == 6
    with pytest.raises(bd.DiffAttnError) as e:
        bd.v2_decode(xd["q"], xd["k_cache"], xd["v_cache"], xd["lam"],
                     workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
    assert e.value.code == 6


@pytest.mark.slow
def test_decode_full_workload_sampled():
    """B=64, L=32768, 64 query heads (32 pairs), 8 kv heads, D=128: sampled (b, pair) rows.
    The 8.6 GB cache is drawn on the device with the seeded generator."""
    s = inputs.WORKLOADS["v2_decode_bf16_B64_L32768_Hq64_Hkv8_D128"]
    x = inputs.make_decode(s, seed=0, device="cuda")
    y = binding().v2_decode(x["q"], x["k_cache"], x["v_cache"], x["lam"])
    P = s.Hq // 2
    rng = np.random.default_rng(2)
    rows = sorted(set([0, 1, P - 1, s.B * P - 1] + list(rng.integers(0, s.B * P, 12))))
    for (qs, ks, vs, ls, local), rid in zip(oracle.decode_gather(x["q"], x["k_cache"], x["v_cache"], x["lam"], rows),
                                           rows):
        ref = oracle.v2_decode(qs, ks, vs, ls, rows=[local])
        got = y.reshape(-1, s.D)[rid:rid + 1]
        assert_parity(got, ref, "bf16")
    del x
    torch.cuda.empty_cache()


def test_deterministic_and_stream():
    """Two calls give bit-identical results, also on a side stream."""
    s = inputs.V2Shape(1, 300, 8, 2, 128, "bf16")
    xd = to_dev(inputs.make_v2(s, seed=3))
    a = binding().v2_fwd(xd["q"], xd["k"], xd["v"], xd["lam"])
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        b = binding().v2_fwd(xd["q"], xd["k"], xd["v"], xd["lam"])
    st.synchronize()
    assert torch.equal(a, b)
    assert binding().device_error() == 0
