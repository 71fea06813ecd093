"""Pins for the oracle's gradients (DIFF V1 and V2 backward), independent of
its code:
  * fp64 autograd through library formulations of the forward (the nanoGPT
    issue's four causal SDPA calls + library rms_norm + lambda from the
    vectors for V1; SDPA over all query heads with repeat_interleave'd kv
    heads and the sigmoid gate for V2);
  * central finite differences of the oracle's own (pinned) forward along
    random directions, for every input including the lambda vectors and
    logits;
  * closed forms: sum over keys of dk is 0 for every head and branch
    (softmax is shift invariant), sum over keys of dv equals the summed
    upstream gradients of the branches, T = 1 gives dq = dk = 0.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from test_oracle_pins import rng_arrays


def _t(a, grad=True):
    x = torch.from_numpy(np.ascontiguousarray(a)).clone()
    x.requires_grad_(grad)
    return x


def _v1_autograd(q1, q2, k1, k2, v, lv, layer, dout):
    ts = [_t(a) for a in (q1, q2, k1, k2, v)]
    ls = [_t(a) for a in lv]
    tq1, tq2, tk1, tk2, tv = ts
    d = q1.shape[-1]
    perm = lambda a: a.permute(0, 2, 1, 3)  # noqa: E731
    v1, v2 = tv[..., :d], tv[..., d:]
    a11 = F.scaled_dot_product_attention(perm(tq1), perm(tk1), perm(v1), is_causal=True)
    a12 = F.scaled_dot_product_attention(perm(tq1), perm(tk1), perm(v2), is_causal=True)
    a21 = F.scaled_dot_product_attention(perm(tq2), perm(tk2), perm(v1), is_causal=True)
    a22 = F.scaled_dot_product_attention(perm(tq2), perm(tk2), perm(v2), is_causal=True)
    lam_init = 0.8 - 0.6 * np.exp(-0.3 * layer)
    lam = torch.exp((ls[0] * ls[1]).sum()) - torch.exp((ls[2] * ls[3]).sum()) + lam_init
    x = torch.cat([a11, a12], -1) - lam * torch.cat([a21, a22], -1)
    y = F.rms_norm(x, (2 * d,), eps=1e-5) * (1 - lam_init)
    (y.permute(0, 2, 1, 3) * torch.from_numpy(dout)).sum().backward()
    names = ["dq1", "dq2", "dk1", "dk2", "dv", "dlam_q1", "dlam_k1", "dlam_q2", "dlam_k2"]
    return dict(zip(names, [a.grad.numpy() for a in ts + ls]))


def _v2_autograd(q, k, v, lam, dout):
    tq, tk, tv, tl = (_t(a) for a in (q, k, v, lam))
    G = q.shape[2] // k.shape[2]
    perm = lambda a: a.permute(0, 2, 1, 3)  # noqa: E731
    a = F.scaled_dot_product_attention(perm(tq), perm(tk).repeat_interleave(G, 1), perm(tv).repeat_interleave(G, 1),
                                       is_causal=True)
    out = a[:, 0::2] - torch.sigmoid(tl).permute(0, 2, 1).unsqueeze(-1) * a[:, 1::2]
    (out.permute(0, 2, 1, 3) * torch.from_numpy(dout)).sum().backward()
    return {"dq": tq.grad.numpy(), "dk": tk.grad.numpy(), "dv": tv.grad.numpy(), "dlam": tl.grad.numpy()}


def _v1_case(seed, B, T, H, d):
    q1, q2, k1, k2 = rng_arrays(seed, *[(B, T, H, d)] * 4)
    v, dout = rng_arrays(seed + 1, (B, T, H, 2 * d), (B, T, H, 2 * d))
    lv = rng_arrays(seed + 2, *[(d,)] * 4, std=0.3)
    return q1, q2, k1, k2, v, lv, dout


@pytest.mark.parametrize("B,T,H,d,layer", [(2, 23, 3, 8, 4), (1, 17, 2, 16, 0)])
def test_v1_bwd_matches_autograd_of_library_forward(oracle, B, T, H, d, layer):
    q1, q2, k1, k2, v, lv, dout = _v1_case(40 + T, B, T, H, d)
    got = oracle.v1_bwd(q1, q2, k1, k2, v, *lv, layer, dout)
    ref = _v1_autograd(q1, q2, k1, k2, v, lv, layer, dout)
    for n, r in ref.items():
        np.testing.assert_allclose(got[n], r, rtol=1e-9, atol=1e-11, err_msg=n)


@pytest.mark.parametrize("B,T,Hq,Hkv,D", [(2, 19, 8, 2, 8), (1, 13, 4, 1, 16), (2, 11, 12, 3, 4)])
def test_v2_bwd_matches_autograd_of_library_forward(oracle, B, T, Hq, Hkv, D):
    q, = rng_arrays(50 + T, (B, T, Hq, D))
    k, v = rng_arrays(51 + T, (B, T, Hkv, D), (B, T, Hkv, D))
    lam, dout = rng_arrays(52 + T, (B, T, Hq // 2), (B, T, Hq // 2, D))
    got = oracle.v2_bwd(q, k, v, lam, dout)
    ref = _v2_autograd(q, k, v, lam, dout)
    for n, r in ref.items():
        np.testing.assert_allclose(got[n], r, rtol=1e-9, atol=1e-11, err_msg=n)


def test_v1_bwd_finite_differences_of_the_forward(oracle):
    """<grad, u> equals (L(x + eps u) - L(x - eps u)) / (2 eps), L = sum(dout * out)."""
    B, T, H, d, layer = 1, 9, 2, 4, 3
    q1, q2, k1, k2, v, lv, dout = _v1_case(60, B, T, H, d)
    g = oracle.v1_bwd(q1, q2, k1, k2, v, *lv, layer, dout)
    base = [q1, q2, k1, k2, v] + lv
    names = ["dq1", "dq2", "dk1", "dk2", "dv", "dlam_q1", "dlam_k1", "dlam_q2", "dlam_k2"]
    r = np.random.default_rng(61)
    eps = 1e-5
    for idx, n in enumerate(names):
        u = r.standard_normal(base[idx].shape)
        plus = [a.copy() for a in base]
        minus = [a.copy() for a in base]
        plus[idx] = plus[idx] + eps * u
        minus[idx] = minus[idx] - eps * u
        lp = (oracle.v1_fwd(*plus[:5], *plus[5:], layer) * dout).sum()
        lm = (oracle.v1_fwd(*minus[:5], *minus[5:], layer) * dout).sum()
        fd = (lp - lm) / (2 * eps)
        an = (g[n] * u).sum()
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (n, fd, an)


def test_v2_bwd_finite_differences_of_the_forward(oracle):
    B, T, Hq, Hkv, D = 1, 8, 4, 2, 4
    q, = rng_arrays(70, (B, T, Hq, D))
    k, v = rng_arrays(71, (B, T, Hkv, D), (B, T, Hkv, D))
    lam, dout = rng_arrays(72, (B, T, Hq // 2), (B, T, Hq // 2, D))
    g = oracle.v2_bwd(q, k, v, lam, dout)
    base = [q, k, v, lam]
    r = np.random.default_rng(73)
    eps = 1e-5
    for idx, n in enumerate(["dq", "dk", "dv", "dlam"]):
        u = r.standard_normal(base[idx].shape)
        plus = [a.copy() for a in base]
        minus = [a.copy() for a in base]
        plus[idx] = plus[idx] + eps * u
        minus[idx] = minus[idx] - eps * u
        fd = ((oracle.v2_fwd(*plus) - oracle.v2_fwd(*minus)) * dout).sum() / (2 * eps)
        an = (g[n] * u).sum()
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (n, fd, an)


def _v1_x_library(q1, q2, k1, k2, v, lam):
    """x = a1 - lam a2 by library causal SDPA (fp64), shape (B, T, H, 2d)."""
    perm = lambda a: torch.from_numpy(np.ascontiguousarray(a)).permute(0, 2, 1, 3)  # noqa: E731
    a1 = F.scaled_dot_product_attention(perm(q1), perm(k1), perm(v), is_causal=True)
    a2 = F.scaled_dot_product_attention(perm(q2), perm(k2), perm(v), is_causal=True)
    return (a1 - lam * a2).permute(0, 2, 1, 3).numpy()


def test_bwd_closed_forms(oracle):
    # V1: sum_j dk_b[j] = 0 per head and branch; sum_j dv[j] = (1 - lam) sum_i dx_i
    B, T, H, d, layer = 2, 14, 2, 8, 5
    q1, q2, k1, k2, v, lv, dout = _v1_case(80, B, T, H, d)
    g = oracle.v1_bwd(q1, q2, k1, k2, v, *lv, layer, dout)
    for n in ("dk1", "dk2"):
        np.testing.assert_allclose(g[n].sum(axis=1), 0.0, atol=1e-12)
    lam_init, lam = oracle.lambda_init(layer), oracle.lambda_full(*lv, layer)
    x = _t(_v1_x_library(q1, q2, k1, k2, v, lam))
    (F.rms_norm(x, (2 * d,), eps=1e-5) * (1 - lam_init) * torch.from_numpy(dout)).sum().backward()
    np.testing.assert_allclose(g["dv"].sum(axis=1), (1 - lam) * x.grad.numpy().sum(axis=1), rtol=1e-9, atol=1e-11)
    # V2: sum_j dk[j] = 0 per kv head; sum_j dv[j] = sum over the group's pairs of (1 - sigmoid) dout
    B, T, Hq, Hkv, D = 2, 12, 8, 2, 4
    q, = rng_arrays(81, (B, T, Hq, D))
    k, v = rng_arrays(82, (B, T, Hkv, D), (B, T, Hkv, D))
    lam, dout = rng_arrays(83, (B, T, Hq // 2), (B, T, Hq // 2, D))
    g = oracle.v2_bwd(q, k, v, lam, dout)
    np.testing.assert_allclose(g["dk"].sum(axis=1), 0.0, atol=1e-12)
    w = (1 - 1 / (1 + np.exp(-lam)))[..., None] * dout           # (B,T,P,D)
    G = Hq // Hkv
    want = w.reshape(B, T, Hkv, G // 2, D).sum(axis=(1, 3))
    np.testing.assert_allclose(g["dv"].sum(axis=1), want, rtol=1e-10, atol=1e-12)
    # T = 1: a single key, so the scores carry no gradient
    g1 = oracle.v2_bwd(q[:, :1], k[:, :1], v[:, :1], lam[:, :1], dout[:, :1])
    assert np.abs(g1["dq"]).max() == 0.0 and np.abs(g1["dk"]).max() == 0.0


def test_bwd_head_subsets(oracle):
    """Subsets of heads / kv groups reproduce the full result on those units."""
    B, T, H, d = 2, 10, 3, 4
    q1, q2, k1, k2, v, lv, dout = _v1_case(90, B, T, H, d)
    full = oracle.v1_bwd(q1, q2, k1, k2, v, *lv, 2, dout)
    sub = oracle.v1_bwd(q1, q2, k1, k2, v, *lv, 2, dout, heads=[1, 5])
    for n in ("dq1", "dk2", "dv"):
        fb = full[n].transpose(0, 2, 1, 3).reshape(B * H, T, -1)
        sb = sub[n].transpose(0, 2, 1, 3).reshape(B * H, T, -1)
        np.testing.assert_array_equal(sb[[1, 5]], fb[[1, 5]])
        assert np.abs(sb[[0, 2, 3, 4]]).max() == 0.0
