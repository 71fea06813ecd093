"""GPU parity of the backward (training) path through the C ABI against the
fp64 oracle's gradients, on the same bf16-rounded inputs and upstream
gradient.  Also: the training forward's output equals the plain forward's.

Tolerance for bf16 gradients (per tensor, against the fp64 oracle):
relative L2 <= 5e-3 and max abs <= 5e-2 * max|ref|.  Each gradient element
is an fp32 sum of products carrying up to three bf16 roundings (P or dS fed
to the tensor cores, the bf16 operand, the upstream gradient of branch 1):
independent relative errors of 2^-9 each give about 3^(1/2) 2^-9 = 3.4e-3
in L2, which the measured errors (2.3e-3 to 4e-3) match; the L2 bound is the
forward's.  The max-abs term allows a single element the sum of the three
worst-case roundings on a gradient whose terms partly cancel.  The
V1 lambda-vector gradients are one scalar dL/dlam = -sum dx . a2 (times
fixed vectors), a sum whose terms cancel: its error is bounded against the
size of those terms, |err| <= 1e-2 * sum |dx_c a2_c| (the oracle reports that
sum), carried through the same fixed factors.
"""
import numpy as np
import pytest
import torch

import oracle
from differential_attention_causal_gb300 import inputs

from test_gpu_parity import binding, built, to_dev  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu

RL2, MAXREL = 5e-3, 5e-2


def check_grad(name, got, ref, report=None, rl2_bound=RL2):
    got = got.detach().float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    assert np.isfinite(got).all(), name
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    rl2 = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    if report is not None:
        report[name] = (float(err / max(scale, 1e-30)), float(rl2))
    assert rl2 <= rl2_bound and err <= MAXREL * scale, \
        f"{name}: max abs {err:.3e} (ref max {scale:.3e}), rel L2 {rl2:.3e}"


def check_lambda_vectors(g, ref, x, report):
    """dlq1 = dlam e1 lk1, dlk1 = dlam e1 lq1, dlq2 = -dlam e2 lk2, dlk2 = -dlam e2 lq2
    with e_b = exp(lq_b . lk_b): each element's error is bounded by
    1e-2 * dlam_abs * e_b * |the fixed factor|."""
    lv = {k: x[k].double().numpy() for k in ("lam_q1", "lam_k1", "lam_q2", "lam_k2")}
    e1 = np.exp((lv["lam_q1"] * lv["lam_k1"]).sum())
    e2 = np.exp((lv["lam_q2"] * lv["lam_k2"]).sum())
    factors = {"dlam_q1": e1 * lv["lam_k1"], "dlam_k1": e1 * lv["lam_q1"],
               "dlam_q2": e2 * lv["lam_k2"], "dlam_k2": e2 * lv["lam_q2"]}
    for n, f in factors.items():
        got = g[n].detach().double().cpu().numpy()
        err = np.abs(got - ref[n])
        bound = 1e-2 * ref["dlam_abs"] * np.abs(f) + 1e-7
        report[n] = (float((err / bound).max()), float(np.linalg.norm(got - ref[n]) /
                                                       max(np.linalg.norm(ref[n]), 1e-30)))
        assert (err <= bound).all(), f"{n}: err / bound = {(err / bound).max():.3f}"


def v1_case(B, T, H, seed, layer=12, d=64):
    x = inputs.make_v1(inputs.V1Shape(B, T, H, d, layer, "bf16"), seed=seed)
    dout = inputs.make_grad_out((B, T, H, 2 * d), "bf16", seed=seed)
    return x, dout


def run_v1(xd, dout_d, layer):
    bd = binding()
    out, saved = bd.v1_fwd_train(xd["q1"], xd["q2"], xd["k1"], xd["k2"], xd["v"], xd["lam_q1"], xd["lam_k1"],
                                 xd["lam_q2"], xd["lam_k2"], layer)
    g = bd.v1_bwd(xd["q1"], xd["q2"], xd["k1"], xd["k2"], xd["v"], xd["lam_q1"], xd["lam_k1"], xd["lam_q2"],
                  xd["lam_k2"], layer, dout_d, saved)
    return out, g


@pytest.mark.parametrize("B,T,H", [(1, 128, 1), (2, 200, 3), (1, 384, 2), (2, 64, 2), (1, 1, 1), (1, 700, 1)])
def test_v1_backward(B, T, H):
    check_v1_backward(B, T, H, 64)


@pytest.mark.parametrize("B,T,H", [(1, 128, 1), (2, 200, 3), (1, 1, 1), (1, 384, 2), (1, 700, 1), (1, 1300, 2)])
def test_v1_backward_d128(B, T, H):
    # d = 128, dv = 256: the two-pass training forward (two launches: output, x and
    # the log-sum-exp; then a2) and the split backward (row pass, lambda, per-branch
    # dK, dV, per-branch dQ: five launches)
    check_v1_backward(B, T, H, 128)


@pytest.mark.parametrize("B,T,H", [(1, 128, 1), (2, 200, 3), (1, 1, 1), (1, 300, 2)])
def test_v1_backward_d32(B, T, H):
    # d = 32 runs the d = 64 kernels on zero-filled q / k boxes; dq, dk keep 32 channels
    check_v1_backward(B, T, H, 32)


def check_v1_backward(B, T, H, d):
    x, dout = v1_case(B, T, H, seed=T + B + d, d=d)
    xd, dd = to_dev(x), dout.cuda()
    out, g = run_v1(xd, dd, 12)
    assert binding().last_launch_count() == (5 if d == 128 else 4)
    assert binding().device_error() == 0
    plain = binding().v1_fwd(xd["q1"], xd["q2"], xd["k1"], xd["k2"], xd["v"], xd["lam_q1"], xd["lam_k1"],
                             xd["lam_q2"], xd["lam_k2"], 12)
    # the same arithmetic; the training build of the kernel may contract a
    # multiply-add differently, which can move a bf16 output by one unit
    assert torch.allclose(out.float(), plain.float(), rtol=2 ** -7, atol=1e-6)
    ref = oracle.v1_bwd(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"], x["lam_q2"],
                        x["lam_k2"], 12, dout)
    rep = {}
    for n in ("dq1", "dq2", "dk1", "dk2", "dv"):
        if T == 1 and n != "dv":
            # one key: the scores carry no gradient, the oracle's are exactly 0.  At
            # d = 128 the saved x is the two-pass forward's, formed from the combined
            # P = e1 / l1 - lam e2 / l2 rounded to bf16, so a1 = x + lam a2 and with it
            # D1 = g . a1 differ from g . v by that rounding: dP - D leaves a residue
            # of the order of 2^-9 |D| scaled by |k| / sqrt(d) (measured 2.4e-6)
            assert g[n].abs().max().item() <= (1e-5 if d == 128 else 1e-6)
            continue
        check_grad(n, g[n], ref[n], rep)
    check_lambda_vectors(g, ref, x, rep)
    print(f"V1 B{B} T{T} H{H} d{d}", {k: f"{a:.2e}/{b:.2e}" for k, (a, b) in rep.items()})


@pytest.mark.parametrize("B,T,Hq,Hkv,D", [(1, 128, 4, 2, 128), (2, 200, 8, 2, 128), (1, 300, 4, 1, 64),
                                          (1, 256, 16, 2, 128), (2, 77, 4, 2, 64)])
def test_v2_backward(B, T, Hq, Hkv, D):
    s = inputs.V2Shape(B, T, Hq, Hkv, D, "bf16")
    x = inputs.make_v2(s, seed=T + Hq)
    dout = inputs.make_grad_out((B, T, Hq // 2, D), "bf16", seed=T)
    xd, dd = to_dev(x), dout.cuda()
    bd = binding()
    out, saved = bd.v2_fwd_train(xd["q"], xd["k"], xd["v"], xd["lam"])
    assert torch.allclose(out.float(), bd.v2_fwd(xd["q"], xd["k"], xd["v"], xd["lam"]).float(), rtol=2 ** -7,
                          atol=1e-6)
    g = bd.v2_bwd(xd["q"], xd["k"], xd["v"], xd["lam"], dd, saved)
    assert bd.last_launch_count() == 3
    assert bd.device_error() == 0
    ref = oracle.v2_bwd(x["q"], x["k"], x["v"], x["lam"], dout)
    rep = {}
    for n in ("dq", "dk", "dv", "dlam"):
        check_grad(n, g[n], ref[n], rep)
    print(f"V2 B{B} T{T} Hq{Hq} Hkv{Hkv} D{D}", {k: f"{a:.2e}/{b:.2e}" for k, (a, b) in rep.items()})


def test_backward_argument_checks():
    bd = binding()
    assert bd.lib().diffattn_v1_train_saved_size(1, 128, 2, 128, 1) > 0    # bf16 d = 128: the split backward
    assert bd.lib().diffattn_v1_train_saved_size(1, 128, 2, 128, 0) > 0    # fp32 d = 128: CUDA-core backward
    assert bd.lib().diffattn_v1_train_saved_size(1, 128, 2, 32, 1) > 0     # bf16 d = 32: the d = 64 kernels
    assert bd.lib().diffattn_v2_bwd_workspace_size(1, 128, 6, 2, 128, 1) > 0
    x = to_dev(inputs.make_v2(inputs.V2Shape(1, 64, 4, 2, 128, "bf16"), seed=1))
    out, saved = bd.v2_fwd_train(x["q"], x["k"], x["v"], x["lam"])
    dout = torch.zeros_like(out)
    with pytest.raises(bd.DiffAttnError) as e:
        bd.v2_bwd(x["q"], x["k"], x["v"], x["lam"], dout, saved[:1024])
    assert e.value.code == 6


@pytest.mark.slow
def test_v1_backward_beyond_2_31_elements():
    """B=2048, T=136 (ragged last tile), 64 heads, d=64: q, k, v, dout and every
    gradient hold 2^31 + 2^27 elements, the saved fp32 tensors 9 GB each; two heads
    of the first and of the last batch entry against the oracle (inputs drawn on
    the device, one batch entry at a time copied back for the oracle)."""
    s = inputs.V1Shape(2048, 136, 64, 64, 5, "bf16")
    assert s.B * s.T * 2 * s.H * s.d > 2 ** 31
    xd = inputs.make_v1(s, seed=6, device="cuda")
    dd = inputs.make_grad_out((s.B, s.T, s.H, 2 * s.d), "bf16", seed=6, device="cuda")
    _, g = run_v1(xd, dd, s.layer_index)
    assert binding().device_error() == 0
    heads = [0, s.H - 1]
    for b in (0, s.B - 1):
        xb = {n: xd[n][b:b + 1].contiguous().cpu() for n in ("q1", "q2", "k1", "k2", "v")}
        ref = oracle.v1_bwd(xb["q1"], xb["q2"], xb["k1"], xb["k2"], xb["v"], xd["lam_q1"].cpu(),
                            xd["lam_k1"].cpu(), xd["lam_q2"].cpu(), xd["lam_k2"].cpu(), s.layer_index,
                            dd[b:b + 1].cpu(), heads=heads)
        for n in ("dq1", "dq2", "dk1", "dk2", "dv"):
            got = g[n][b:b + 1].float().cpu().permute(0, 2, 1, 3).reshape(s.H, s.T, -1)[heads]
            want = ref[n].transpose(0, 2, 1, 3).reshape(s.H, s.T, -1)[heads]
            check_grad(n, got, want)
    del g, xd, dd
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_v1_backward_full_workload_sampled_heads():
    """B=4, T=2048, 16 heads, d=64 (the bench's V1 workload and launch): gradients of
    three sampled (b, h) heads against the oracle (heads are independent in V1;
    the lambda-vector gradients need every head and are checked at small sizes)."""
    s = inputs.WORKLOADS["v1_bf16_B4_T2048_H16_d64"]
    x = inputs.make_v1(s, seed=0)
    dout = inputs.make_grad_out((s.B, s.T, s.H, 2 * s.d), "bf16", seed=0)
    xd, dd = to_dev(x), dout.cuda()
    _, g = run_v1(xd, dd, s.layer_index)
    heads = [0, 21, s.B * s.H - 1]
    ref = oracle.v1_bwd(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"], x["lam_q2"],
                        x["lam_k2"], s.layer_index, dout, heads=heads)
    for n in ("dq1", "dq2", "dk1", "dk2", "dv"):
        got = g[n].float().cpu().permute(0, 2, 1, 3).reshape(s.B * s.H, s.T, -1)[heads]
        want = ref[n].transpose(0, 2, 1, 3).reshape(s.B * s.H, s.T, -1)[heads]
        check_grad(n, got, want)


@pytest.mark.slow
def test_v2_backward_long_sequence():
    """T=4096 (the V2 prefill workload's length), 4 query heads over 2 kv heads, D=128."""
    s = inputs.V2Shape(1, 4096, 4, 2, 128, "bf16")
    x = inputs.make_v2(s, seed=5)
    dout = inputs.make_grad_out((s.B, s.T, s.Hq // 2, s.D), "bf16", seed=5)
    xd, dd = to_dev(x), dout.cuda()
    bd = binding()
    _, saved = bd.v2_fwd_train(xd["q"], xd["k"], xd["v"], xd["lam"])
    g = bd.v2_bwd(xd["q"], xd["k"], xd["v"], xd["lam"], dd, saved)
    ref = oracle.v2_bwd(x["q"], x["k"], x["v"], x["lam"], dout)
    for n in ("dq", "dk", "dv", "dlam"):
        check_grad(n, g[n], ref[n])


# ------------------------------------------------------------------ fp32 path
# fp32 everywhere (CUDA cores, exact fp32 sums): the bound is the fp32 one of
# the forward, max abs <= 1e-4 absolute; the lambda-vector gradients against
# the size of the terms that cancel in dL/dlam, as for bf16 but at 1e-4.

def check_f32(name, got, ref):
    got = got.detach().double().cpu().numpy().reshape(ref.shape)
    err = np.abs(got - ref).max()
    print(f"fp32 {name}: max abs {err:.3e} (max |ref| {np.abs(ref).max():.3e})")
    assert np.isfinite(got).all() and err <= 1e-4, f"{name}: max abs {err:.3e}"


@pytest.mark.parametrize("B,T,H,d", [(2, 45, 2, 32), (1, 70, 3, 64), (1, 33, 2, 128)])
def test_v1_backward_fp32(B, T, H, d):
    x = inputs.make_v1(inputs.V1Shape(B, T, H, d, 3, "fp32"), seed=T)
    dout = inputs.make_grad_out((B, T, H, 2 * d), "fp32", seed=T)
    xd, dd = to_dev(x), dout.cuda()
    out, g = run_v1(xd, dd, 3)
    assert binding().last_launch_count() == 4
    assert binding().device_error() == 0
    plain = binding().v1_fwd(xd["q1"], xd["q2"], xd["k1"], xd["k2"], xd["v"], xd["lam_q1"], xd["lam_k1"],
                             xd["lam_q2"], xd["lam_k2"], 3)
    assert torch.equal(out, plain)
    ref = oracle.v1_bwd(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"], x["lam_q2"],
                        x["lam_k2"], 3, dout)
    for n in ("dq1", "dq2", "dk1", "dk2", "dv"):
        check_f32(n, g[n], ref[n])
    lv = {k: x[k].double().numpy() for k in ("lam_q1", "lam_k1", "lam_q2", "lam_k2")}
    e1 = np.exp((lv["lam_q1"] * lv["lam_k1"]).sum())
    e2 = np.exp((lv["lam_q2"] * lv["lam_k2"]).sum())
    for n, f in {"dlam_q1": e1 * lv["lam_k1"], "dlam_k1": e1 * lv["lam_q1"],
                 "dlam_q2": e2 * lv["lam_k2"], "dlam_k2": e2 * lv["lam_q2"]}.items():
        err = np.abs(g[n].double().cpu().numpy() - ref[n])
        assert (err <= 1e-4 * ref["dlam_abs"] * np.abs(f) + 1e-7).all(), n


@pytest.mark.parametrize("B,T,Hq,Hkv,D", [(2, 40, 4, 2, 64), (1, 57, 8, 2, 128)])
def test_v2_backward_fp32(B, T, Hq, Hkv, D):
    x = inputs.make_v2(inputs.V2Shape(B, T, Hq, Hkv, D, "fp32"), seed=T)
    dout = inputs.make_grad_out((B, T, Hq // 2, D), "fp32", seed=T)
    xd, dd = to_dev(x), dout.cuda()
    bd = binding()
    out, saved = bd.v2_fwd_train(xd["q"], xd["k"], xd["v"], xd["lam"])
    assert torch.equal(out, bd.v2_fwd(xd["q"], xd["k"], xd["v"], xd["lam"]))
    g = bd.v2_bwd(xd["q"], xd["k"], xd["v"], xd["lam"], dd, saved)
    assert bd.last_launch_count() == 3
    assert bd.device_error() == 0
    ref = oracle.v2_bwd(x["q"], x["k"], x["v"], x["lam"], dout)
    for n in ("dq", "dk", "dv", "dlam"):
        check_f32(n, g[n], ref[n])


def test_v1_backward_d128_long_context_workload():
    """B=1, T=32768, 12 diff heads, d=128, dv=256, layer_index=27 (the long-context
    V1 workload), in the launch the bench times.  Row i's dq1, dq2 depend only on
    tokens 0..i (its keys, values and its own upstream gradient), so the first
    T0 = 1024 rows of two heads are checked element by element against the
    oracle's gradients of the same inputs cut at T0.  dK and dV of every key
    depend on all later rows; for them the full-size property checked is that
    each head's keys' dk sum to zero (sum_j dS_ij = 0 for every row), bounded
    by the sum of |dk| times the bf16 rounding scale."""
    s = inputs.WORKLOADS["v1_bf16_B1_T32768_H12_d128"]
    xd = inputs.make_v1(s, seed=2, device="cuda")
    dd = inputs.make_grad_out((s.B, s.T, s.H, 2 * s.d), "bf16", seed=2, device="cuda")
    _, g = run_v1(xd, dd, s.layer_index)
    assert binding().device_error() == 0
    T0, heads = 1024, [0, s.H - 1]
    xc = {n: xd[n][:, :T0, heads].contiguous().cpu() for n in ("q1", "q2", "k1", "k2", "v")}
    ref = oracle.v1_bwd(xc["q1"], xc["q2"], xc["k1"], xc["k2"], xc["v"], xd["lam_q1"].cpu(), xd["lam_k1"].cpu(),
                        xd["lam_q2"].cpu(), xd["lam_k2"].cpu(), s.layer_index, dd[:, :T0, heads].cpu())
    for n in ("dq1", "dq2"):
        check_grad(n, g[n][:, :T0, heads], ref[n])
    for n in ("dk1", "dk2"):
        gk = g[n].float()
        tot = gk.sum(dim=1).abs()                     # (B, H, d): sum over keys
        scale = gk.abs().sum(dim=1)
        assert bool((tot <= 1e-2 * scale + 1e-3).all()), (n, float((tot / (scale + 1e-30)).max()))
    assert torch.isfinite(g["dv"].float()).all()
    del g, xd, dd
    torch.cuda.empty_cache()
