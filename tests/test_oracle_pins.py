"""Pins for the fp64 oracle: it is checked against things other than itself.

Each test ties the oracle to what the pages or the mathematics fix:
  * values printed on the pages (tests/golden/page_constants.txt);
  * closed forms worked out by hand for tiny inputs;
  * library attention routines in other formulations (torch's fp64
    scaled_dot_product_attention and rms_norm; the nanoGPT issue's
    four-call split of v and its materialised-weights form);
  * invariants the definition implies (identical branches, T = 1,
    causality, batch permutation, decode == last prefill row).
A plausible slip in the oracle (scale, mask offset, lambda sign, eps
placement, missing (1 - lam_init), wrong head pairing or GQA mapping, an
off-by-one in the decode key count) fails at least one of these.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def page_constants():
    vals = {}
    with open(os.path.join(GOLDEN, "page_constants.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                vals[k] = float(v)
    return vals


def rng_arrays(seed, *shapes, std=1.0):
    r = np.random.default_rng(seed)
    return [r.standard_normal(s) * std for s in shapes]


# ---------------------------------------------------------------- lambda ---

def test_lambda_init_printed_value_and_shape(oracle):
    c = page_constants()
    # layer 0: 0.8 - 0.6 = 0.2 exactly as stated with the workload description
    assert oracle.lambda_init(0) == pytest.approx(c["lam_init_layer0"], abs=1e-15)
    # the schedule rises towards 0.8 and its gap to 0.8 shrinks by e^{0.3} per layer
    prev = oracle.lambda_init(0)
    for L in range(1, 40):
        cur = oracle.lambda_init(L)
        assert prev < cur < c["lam_init_a"]
        ratio = (c["lam_init_a"] - prev) / (c["lam_init_a"] - cur)
        assert ratio == pytest.approx(math.e ** c["lam_init_c"], rel=1e-8)  # gap to 0.8 cancels
        prev = cur
    assert oracle.lambda_init(200) == pytest.approx(c["lam_init_a"], abs=1e-15)


def test_lambda_full_closed_forms(oracle):
    z = np.zeros(8)
    # all-zero vectors: exp(0) - exp(0) + lam_init
    assert oracle.lambda_full(z, z, z, z, 5) == pytest.approx(oracle.lambda_init(5), abs=1e-15)
    # lq1.lk1 = ln 2, lq2.lk2 = 0  ->  2 - 1 + lam_init
    a = np.zeros(8); a[3] = math.log(2.0)
    b = np.zeros(8); b[3] = 1.0
    assert oracle.lambda_full(a, b, z, z, 3) == pytest.approx(1.0 + oracle.lambda_init(3), abs=1e-14)
    # the branch-2 term enters with a minus sign: lq2.lk2 = ln 3 -> 1 - 3 + lam_init
    assert oracle.lambda_full(z, z, a * math.log(3.0) / math.log(2.0), b, 0) == pytest.approx(
        1.0 - 3.0 + 0.2, abs=1e-14)


# --------------------------------------------------------------- rmsnorm ---

def test_rmsnorm_matches_library_and_unit_rms(oracle):
    c = page_constants()
    eps = c["rmsnorm_eps"]
    x, small = rng_arrays(1, (16, 128), (4, 64))
    small *= 3e-3  # mean square ~1e-5: eps placement matters here
    for arr in (x, small):
        got = oracle.rmsnorm(arr, eps)
        ref = F.rms_norm(torch.from_numpy(arr), (arr.shape[-1],), eps=eps).numpy()
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)
        ms = (arr ** 2).mean(-1)
        np.testing.assert_allclose((got ** 2).mean(-1), ms / (ms + eps), rtol=1e-12)


# --------------------------------------------------- V1 by hand (T = 2) ---

def test_v1_hand_worked_example(oracle):
    """d = 1 (scale 1), dv = 2, layer 0 (lam_init 0.2), zero lambda vectors (lam = 0.2).

    Row 1, branch 1: logits (0, ln 3) -> weights (1/4, 3/4); branch 2: (ln 3, 0) -> (3/4, 1/4).
    With v0 = (1, 0), v1 = (0, 1): a1 = (1/4, 3/4), a2 = (3/4, 1/4), x = a1 - 0.2 a2 = (0.1, 0.7).
    Row 0 attends only key 0: a1 = a2 = v0, x = 0.8 v0.
    """
    ln3 = math.log(3.0)
    q1 = np.array([1.0, 1.0]).reshape(1, 2, 1, 1)
    k1 = np.array([0.0, ln3]).reshape(1, 2, 1, 1)
    q2 = np.array([1.0, 1.0]).reshape(1, 2, 1, 1)
    k2 = np.array([ln3, 0.0]).reshape(1, 2, 1, 1)
    v = np.array([[1.0, 0.0], [0.0, 1.0]]).reshape(1, 2, 1, 2)
    z = np.zeros(1)
    out = oracle.v1_fwd(q1, q2, k1, k2, v, z, z, z, z, 0)
    eps = page_constants()["rmsnorm_eps"]
    x1 = np.array([0.1, 0.7])
    y1 = x1 / math.sqrt(0.25 + eps) * 0.8
    x0 = np.array([0.8, 0.0])
    y0 = x0 / math.sqrt(0.32 + eps) * 0.8
    np.testing.assert_allclose(out[0, 1, 0], y1, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(out[0, 0, 0], y0, rtol=1e-13, atol=1e-15)


# ------------------------------------- V1 against library formulations ---

def _v1_four_sdpa(q1, q2, k1, k2, v, lq1, lk1, lq2, lk2, layer_index):
    """The nanoGPT issue's first variant: four causal SDPA calls on the two halves of v,
    concatenated, combined with lambda, RMSNorm (library), times (1 - lam_init)."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).permute(0, 2, 1, 3)  # (B,H,T,*)
    d = q1.shape[-1]
    v1, v2 = v[..., :d], v[..., d:]
    a11 = F.scaled_dot_product_attention(t(q1), t(k1), t(v1), is_causal=True)
    a12 = F.scaled_dot_product_attention(t(q1), t(k1), t(v2), is_causal=True)
    a21 = F.scaled_dot_product_attention(t(q2), t(k2), t(v1), is_causal=True)
    a22 = F.scaled_dot_product_attention(t(q2), t(k2), t(v2), is_causal=True)
    attn1 = torch.cat([a11, a12], dim=-1)
    attn2 = torch.cat([a21, a22], dim=-1)
    lam_init = 0.8 - 0.6 * torch.exp(torch.tensor(-0.3 * layer_index, dtype=torch.float64))
    lam = (torch.exp((torch.from_numpy(lq1) * torch.from_numpy(lk1)).sum())
           - torch.exp((torch.from_numpy(lq2) * torch.from_numpy(lk2)).sum()) + lam_init)
    y = F.rms_norm(attn1 - lam * attn2, (2 * d,), eps=1e-5) * (1 - lam_init)
    return y.permute(0, 2, 1, 3).numpy()


def _v1_weights_form(q1, q2, k1, k2, v, lam, lam_init):
    """The nanoGPT issue's second variant: materialised causal weights,
    (A1 - lam A2) @ v, then RMSNorm (its LayerNorm replaced per DiffAttnV1)."""
    B, T, H, d = q1.shape
    out = np.empty(v.shape)
    mask = np.tril(np.ones((T, T), dtype=bool))
    for b in range(B):
        for h in range(H):
            ws = []
            for q, k in ((q1, k1), (q2, k2)):
                s = q[b, :, h] @ k[b, :, h].T / math.sqrt(d)
                s = np.where(mask, s, -np.inf)
                s = np.exp(s - s.max(-1, keepdims=True))
                ws.append(s / s.sum(-1, keepdims=True))
            x = (ws[0] - lam * ws[1]) @ v[b, :, h]
            out[b, :, h] = x / np.sqrt((x ** 2).mean(-1, keepdims=True) + 1e-5) * (1 - lam_init)
    return out


@pytest.mark.parametrize("B,T,H,d,layer", [(2, 37, 3, 8, 4), (1, 20, 1, 16, 0), (3, 9, 2, 4, 27)])
def test_v1_matches_four_sdpa_formulation(oracle, B, T, H, d, layer):
    q1, q2, k1, k2 = rng_arrays(10 + T, *[(B, T, H, d)] * 4)
    (v,) = rng_arrays(20 + T, (B, T, H, 2 * d))
    lq1, lk1, lq2, lk2 = rng_arrays(30 + T, *[(d,)] * 4, std=0.5)
    got = oracle.v1_fwd(q1, q2, k1, k2, v, lq1, lk1, lq2, lk2, layer)
    ref = _v1_four_sdpa(q1, q2, k1, k2, v, lq1, lk1, lq2, lk2, layer)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)
    lam_init = oracle.lambda_init(layer)
    lam = oracle.lambda_full(lq1, lk1, lq2, lk2, layer)
    ref2 = _v1_weights_form(q1, q2, k1, k2, v, lam, lam_init)
    np.testing.assert_allclose(got, ref2, rtol=1e-10, atol=1e-12)


def test_v1_lambda_zero_reduces_to_plain_attention(oracle):
    """lam = 0 (lq1 = lk1 = 0, lq2.lk2 = ln(1 + lam_init)): out = (1-lam_init) RMSNorm(SDPA(q1,k1,v))."""
    B, T, H, d, layer = 2, 33, 2, 8, 3
    q1, q2, k1, k2 = rng_arrays(5, *[(B, T, H, d)] * 4)
    (v,) = rng_arrays(6, (B, T, H, 2 * d))
    lam_init = oracle.lambda_init(layer)
    z = np.zeros(d)
    lq2 = np.zeros(d); lq2[0] = math.log(1.0 + lam_init)
    lk2 = np.zeros(d); lk2[0] = 1.0
    assert oracle.lambda_full(z, z, lq2, lk2, layer) == pytest.approx(0.0, abs=1e-14)
    got = oracle.v1_fwd(q1, q2, k1, k2, v, z, z, lq2, lk2, layer)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).permute(0, 2, 1, 3)
    a = F.scaled_dot_product_attention(t(q1), t(k1), t(v), is_causal=True)
    ref = (F.rms_norm(a, (2 * d,), eps=1e-5) * (1 - lam_init)).permute(0, 2, 1, 3).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_v1_identical_branches(oracle):
    """q1 = q2, k1 = k2 -> x = (1 - lam) A; y = sign(1-lam) A / sqrt(mean A^2 + eps/(1-lam)^2) (1-lam_init)."""
    B, T, H, d, layer = 1, 25, 2, 8, 2
    q, k = rng_arrays(7, (B, T, H, d), (B, T, H, d))
    (v,) = rng_arrays(8, (B, T, H, 2 * d))
    for lq1_scale in (0.1, 2.0):  # lam below and above 1
        lq1 = np.full(d, lq1_scale / math.sqrt(d)); lk1 = np.full(d, 1.0 / math.sqrt(d))
        z = np.zeros(d)
        lam = oracle.lambda_full(lq1, lk1, z, z, layer)
        lam_init = oracle.lambda_init(layer)
        got = oracle.v1_fwd(q, q, k, k, v, lq1, lk1, z, z, layer)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).permute(0, 2, 1, 3)
        A = F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True).permute(0, 2, 1, 3).numpy()
        ref = (np.sign(1 - lam) * A / np.sqrt((A ** 2).mean(-1, keepdims=True) + 1e-5 / (1 - lam) ** 2)
               * (1 - lam_init))
        np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_first_row_is_first_value_row(oracle):
    """Row 0 (and T = 1) attends only key 0: V1 x = (1 - lam) v0; V2 out = (1 - sigmoid) v_g[0]."""
    d, layer = 8, 1
    q1, q2, k1, k2 = rng_arrays(9, *[(2, 1, 3, d)] * 4)
    (v,) = rng_arrays(10, (2, 1, 3, 2 * d))
    lq1, lk1, lq2, lk2 = rng_arrays(11, *[(d,)] * 4, std=0.1)
    lam = oracle.lambda_full(lq1, lk1, lq2, lk2, layer)
    lam_init = oracle.lambda_init(layer)
    got = oracle.v1_fwd(q1, q2, k1, k2, v, lq1, lk1, lq2, lk2, layer)
    x = (1 - lam) * v
    ref = x / np.sqrt((x ** 2).mean(-1, keepdims=True) + 1e-5) * (1 - lam_init)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)
    # V2: Hq = 8, Hkv = 2 (G = 4)
    q, = rng_arrays(12, (2, 1, 8, d))
    k, vv = rng_arrays(13, (2, 1, 2, d), (2, 1, 2, d))
    (lg,) = rng_arrays(14, (2, 1, 4))
    got2 = oracle.v2_fwd(q, k, vv, lg)
    sig = 1 / (1 + np.exp(-lg))
    for i in range(4):
        g = (2 * i) // 4
        np.testing.assert_allclose(got2[:, 0, i], (1 - sig[:, 0, i, None]) * vv[:, 0, g], rtol=1e-12, atol=1e-14)


# -------------------------------------------------------------------- V2 ---

def _v2_library(q, k, v, lam):
    """torch SDPA over all Hq heads with kv head h // G (groups contiguous), then
    attn[:, 0::2] - sigmoid(lam) * attn[:, 1::2] ("Differential Transformer V2", DiffAttnV2)."""
    G = q.shape[2] // k.shape[2]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).permute(0, 2, 1, 3)
    kk = t(k).repeat_interleave(G, dim=1)
    vv = t(v).repeat_interleave(G, dim=1)
    attn = F.scaled_dot_product_attention(t(q), kk, vv, is_causal=True)  # (B,Hq,T,D)
    a1, a2 = attn[:, 0::2], attn[:, 1::2]
    s = torch.sigmoid(torch.from_numpy(lam)).permute(0, 2, 1).unsqueeze(-1)
    return (a1 - s * a2).permute(0, 2, 1, 3).numpy()


@pytest.mark.parametrize("B,T,Hq,Hkv,D", [(2, 29, 8, 2, 8), (1, 17, 4, 1, 16), (2, 12, 12, 3, 4)])
def test_v2_matches_library_gqa(oracle, B, T, Hq, Hkv, D):
    q, = rng_arrays(40 + T, (B, T, Hq, D))
    k, v = rng_arrays(41 + T, (B, T, Hkv, D), (B, T, Hkv, D))
    (lam,) = rng_arrays(42 + T, (B, T, Hq // 2))
    got = oracle.v2_fwd(q, k, v, lam)
    np.testing.assert_allclose(got, _v2_library(q, k, v, lam), rtol=1e-10, atol=1e-12)


def test_v2_sigmoid_zero_gives_even_head_attention(oracle):
    B, T, Hq, Hkv, D = 1, 21, 8, 2, 8
    q, = rng_arrays(50, (B, T, Hq, D))
    k, v = rng_arrays(51, (B, T, Hkv, D), (B, T, Hkv, D))
    lam = np.full((B, T, Hq // 2), -1e4)  # sigmoid -> 0
    got = oracle.v2_fwd(q, k, v, lam)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).permute(0, 2, 1, 3)
    for i in range(Hq // 2):
        g = (2 * i) // (Hq // Hkv)
        a = F.scaled_dot_product_attention(t(q[:, :, 2 * i:2 * i + 1]), t(k[:, :, g:g + 1]),
                                           t(v[:, :, g:g + 1]), is_causal=True)
        np.testing.assert_allclose(got[:, :, i], a.permute(0, 2, 1, 3)[:, :, 0].numpy(),
                                   rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- decode ---

def test_decode_matches_library_and_last_prefill_row(oracle):
    B, L, Hq, Hkv, D = 2, 45, 8, 2, 16
    k, v = rng_arrays(60, (B, L, Hkv, D), (B, L, Hkv, D))
    qfull, = rng_arrays(61, (B, L, Hq, D))
    (lamfull,) = rng_arrays(62, (B, L, Hq // 2))
    q, lam = qfull[:, -1], lamfull[:, -1]
    got = oracle.v2_decode(q, k, v, lam)
    # (a) the last row of a causal prefill over the same L rows
    pre = oracle.v2_fwd(qfull, k, v, lamfull)
    np.testing.assert_allclose(got, pre[:, -1], rtol=1e-12, atol=1e-14)
    # (b) library attention of one query over all L keys (no mask)
    G = Hq // Hkv
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    qq = t(q).unsqueeze(2)                                   # (B,Hq,1,D)
    kk = t(k).permute(0, 2, 1, 3).repeat_interleave(G, 1)    # (B,Hq,L,D)
    vv = t(v).permute(0, 2, 1, 3).repeat_interleave(G, 1)
    a = F.scaled_dot_product_attention(qq, kk, vv)[:, :, 0]  # (B,Hq,D)
    ref = a[:, 0::2] - torch.sigmoid(t(lam)).unsqueeze(-1) * a[:, 1::2]
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12)


def _v1_decode_library(q1, q2, k1, k2, v, lam, lam_init, lens):
    """V1 decode by library calls, one sequence at a time: the new token's two
    softmax attentions over the first len_b cached rows (torch fp64 SDPA, no
    mask), lambda combination, library RMSNorm, times (1 - lam_init)."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    out = []
    for b, n in enumerate(lens):
        kk1 = t(k1[b, :n]).permute(1, 0, 2)          # (H,n,d)
        kk2 = t(k2[b, :n]).permute(1, 0, 2)
        vv = t(v[b, :n]).permute(1, 0, 2)            # (H,n,2d)
        a1 = F.scaled_dot_product_attention(t(q1[b]).unsqueeze(1), kk1, vv)[:, 0]
        a2 = F.scaled_dot_product_attention(t(q2[b]).unsqueeze(1), kk2, vv)[:, 0]
        out.append(F.rms_norm(a1 - lam * a2, (v.shape[-1],), eps=1e-5) * (1 - lam_init))
    return torch.stack(out).numpy()


def test_v1_decode_matches_library_and_last_prefill_row(oracle):
    B, L, H, d, layer = 2, 33, 3, 8, 5
    q1f, q2f, k1, k2 = rng_arrays(64, *[(B, L, H, d)] * 4)
    (v,) = rng_arrays(65, (B, L, H, 2 * d))
    lv = rng_arrays(66, *[(d,)] * 4, std=0.5)
    got = oracle.v1_decode(q1f[:, -1], q2f[:, -1], k1, k2, v, *lv, layer)
    # (a) the last row of a causal V1 prefill over the same L rows
    pre = oracle.v1_fwd(q1f, q2f, k1, k2, v, *lv, layer)
    np.testing.assert_allclose(got, pre[:, -1], rtol=1e-12, atol=1e-14)
    # (b) library attention of one query over all L keys
    lam_init, lam = oracle.lambda_init(layer), oracle.lambda_full(*lv, layer)
    ref = _v1_decode_library(q1f[:, -1], q2f[:, -1], k1, k2, v, lam, lam_init, [L] * B)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_decode_lengths_read_only_each_sequence_rows(oracle):
    """Per-sequence cache lengths: rows past len_b are never read (they hold
    NaN here), and each sequence matches library attention over its prefix."""
    B, L, Hq, Hkv, D = 3, 40, 8, 2, 8
    lens = np.array([40, 17, 1])
    q, = rng_arrays(67, (B, Hq, D))
    k, v = rng_arrays(68, (B, L, Hkv, D), (B, L, Hkv, D))
    (lam,) = rng_arrays(69, (B, Hq // 2))
    for b, n in enumerate(lens):
        k[b, n:] = np.nan
        v[b, n:] = np.nan
    got = oracle.v2_decode(q, k, v, lam, lens=lens)
    assert np.isfinite(got).all()
    G = Hq // Hkv
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    for b, n in enumerate(lens):
        kk = t(k[b, :n]).permute(1, 0, 2).repeat_interleave(G, 0)
        vv = t(v[b, :n]).permute(1, 0, 2).repeat_interleave(G, 0)
        a = F.scaled_dot_product_attention(t(q[b]).unsqueeze(1), kk, vv)[:, 0]
        ref = a[0::2] - torch.sigmoid(t(lam[b])).unsqueeze(-1) * a[1::2]
        np.testing.assert_allclose(got[b], ref.numpy(), rtol=1e-10, atol=1e-12)
    # a single cached row: both heads of a pair return that row's value
    g_of_pair = (2 * np.arange(Hq // 2)) // G
    one = (1 - 1 / (1 + np.exp(-lam[2])))[:, None] * v[2, 0, g_of_pair]
    np.testing.assert_allclose(got[2], one, rtol=1e-13, atol=1e-15)

    H, d, layer = 2, 4, 3
    q1, q2 = rng_arrays(70, (B, H, d), (B, H, d))
    k1, k2 = rng_arrays(71, (B, L, H, d), (B, L, H, d))
    (vv,) = rng_arrays(72, (B, L, H, 2 * d))
    lv = rng_arrays(73, *[(d,)] * 4, std=0.5)
    for b, n in enumerate(lens):
        k1[b, n:] = np.nan
        k2[b, n:] = np.nan
        vv[b, n:] = np.nan
    got1 = oracle.v1_decode(q1, q2, k1, k2, vv, *lv, layer, lens=lens)
    assert np.isfinite(got1).all()
    lam_init, lamf = oracle.lambda_init(layer), oracle.lambda_full(*lv, layer)
    ref1 = _v1_decode_library(q1, q2, k1, k2, vv, lamf, lam_init, lens)
    np.testing.assert_allclose(got1, ref1, rtol=1e-10, atol=1e-12)
    # a single cached row: x = (1 - lam) v0, so the output is v0 / rms(v0)
    # (sign of 1 - lam) times (1 - lam_init), up to the eps inside the root
    v0 = vv[2, 0]
    x = (1 - lamf) * v0
    closed = x / np.sqrt((x * x).mean(-1, keepdims=True) + 1e-5) * (1 - lam_init)
    np.testing.assert_allclose(got1[2], closed, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------ invariants ---

def test_causality_future_rows_do_not_matter(oracle):
    B, T, H, d, layer = 1, 30, 2, 8, 5
    q1, q2, k1, k2 = rng_arrays(70, *[(B, T, H, d)] * 4)
    (v,) = rng_arrays(71, (B, T, H, 2 * d))
    lam = rng_arrays(72, *[(d,)] * 4, std=0.1)
    base = oracle.v1_fwd(q1, q2, k1, k2, v, *lam, layer)
    cut = 17
    k1b, k2b, vb = k1.copy(), k2.copy(), v.copy()
    k1b[:, cut:] += 5.0; k2b[:, cut:] -= 3.0; vb[:, cut:] *= -2.0
    pert = oracle.v1_fwd(q1, q2, k1b, k2b, vb, *lam, layer)
    np.testing.assert_array_equal(base[:, :cut], pert[:, :cut])
    assert not np.allclose(base[:, cut:], pert[:, cut:])


def test_batch_permutation_and_row_subset(oracle):
    B, T, Hq, Hkv, D = 3, 19, 8, 2, 8
    q, = rng_arrays(80, (B, T, Hq, D))
    k, v = rng_arrays(81, (B, T, Hkv, D), (B, T, Hkv, D))
    (lam,) = rng_arrays(82, (B, T, Hq // 2))
    full = oracle.v2_fwd(q, k, v, lam)
    perm = [2, 0, 1]
    permuted = oracle.v2_fwd(q[perm], k[perm], v[perm], lam[perm])
    np.testing.assert_array_equal(permuted, full[perm])
    rows = np.array([0, 5, 77, B * T * (Hq // 2) - 1])
    sub = oracle.v2_fwd(q, k, v, lam, rows=rows)
    np.testing.assert_array_equal(sub, full.reshape(-1, D)[rows])
    # V1 subset too
    q1, q2, k1, k2 = rng_arrays(83, *[(2, 11, 3, 4)] * 4)
    (vv,) = rng_arrays(84, (2, 11, 3, 8))
    lv = rng_arrays(85, *[(4,)] * 4, std=0.1)
    f1 = oracle.v1_fwd(q1, q2, k1, k2, vv, *lv, 7)
    r1 = np.array([3, 40, 65])
    np.testing.assert_array_equal(oracle.v1_fwd(q1, q2, k1, k2, vv, *lv, 7, rows=r1),
                                  f1.reshape(-1, 8)[r1])


def test_thread_count_does_not_change_result(oracle):
    q1, q2, k1, k2 = rng_arrays(90, *[(1, 40, 2, 8)] * 4)
    (v,) = rng_arrays(91, (1, 40, 2, 16))
    lam = rng_arrays(92, *[(8,)] * 4, std=0.1)
    a = oracle.v1_fwd(q1, q2, k1, k2, v, *lam, 2, nthreads=1)
    b = oracle.v1_fwd(q1, q2, k1, k2, v, *lam, 2, nthreads=7)
    np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------ row log-sum-exp

def test_lse_closed_forms(oracle):
    """q = 0: every visible score is 0, so row t normalises t + 1 ones and
    lse = log(t + 1) exactly; T = 1: lse = q0 . k0 / sqrt(d)."""
    rng = np.random.default_rng(40)
    q = np.zeros((2, 9, 4, 8))
    k = rng.standard_normal((2, 9, 2, 8))
    got = oracle.lse(q, k)
    want = np.broadcast_to(np.log(np.arange(1, 10, dtype=np.float64)), got.shape)
    assert np.abs(got - want).max() < 1e-14
    q1 = rng.standard_normal((1, 1, 2, 16))
    k1 = rng.standard_normal((1, 1, 2, 16))
    got = oracle.lse(q1, k1)[0, :, 0]
    want = (q1[0, 0] * k1[0, 0]).sum(-1) / 4.0
    assert np.abs(got - want).max() < 1e-14


@pytest.mark.parametrize("Hq,Hk", [(3, 3), (8, 2)])
def test_lse_matches_library_logsumexp(oracle, Hq, Hk):
    """Against torch.logsumexp of the causally masked, 1/sqrt(d)-scaled fp64
    scores, query head h reading key head h / (Hq / Hk)."""
    rng = np.random.default_rng(41 + Hq)
    B, T, d = 2, 23, 16
    q = rng.standard_normal((B, T, Hq, d)) * 2.0
    k = rng.standard_normal((B, T, Hk, d))
    qt = torch.from_numpy(q).permute(0, 2, 1, 3)                          # (B, Hq, T, d)
    kt = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(Hq // Hk, dim=1)
    s = qt @ kt.transpose(-1, -2) / np.sqrt(d)
    mask = torch.ones(T, T, dtype=torch.bool).tril()
    want = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1).numpy()
    got = oracle.lse(q, k)
    assert np.abs(got - want).max() < 1e-12
