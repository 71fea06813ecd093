"""Pins for the oracle's Paired Head Attention (modded-nanogpt pull request
"New Record: Paired Head Attention (-3.5s, -65 steps)", section "Updates in
PR"), independent of its code:
  * the page's worked interleave order and its visibility example, stored in
    tests/golden/paired_heads.txt;
  * torch's fp64 causal scaled_dot_product_attention run on the interleaved
    sequence, built here by a reshape rather than by index arithmetic;
  * closed forms at T = 1 and for a pair of identical heads (every earlier
    key then counts twice).
A wrong interleave order, an off-by-one in the causal limit, swapped heads or
a wrong scale fails at least one of them.
"""
import os

import numpy as np
import torch
import torch.nn.functional as F

from test_oracle_pins import rng_arrays

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "paired_heads.txt")


def golden():
    order, visible = None, []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if not line:
                continue
            if line[0] == "interleave":
                order = [tuple(int(x) for x in tok[1:].split("_h")) for tok in line[1:]]
            elif line[0] == "visible":
                visible.append(tuple(int(x) for x in line[1:]))
    return order, visible


def library_paired(q, k, v):
    """Interleave by reshape, one causal SDPA call, de-interleave."""
    B, T, H, D = q.shape

    def inter(x):
        return torch.from_numpy(np.ascontiguousarray(
            x.reshape(B, T, H // 2, 2, D).transpose(0, 2, 1, 3, 4).reshape(B, H // 2, 2 * T, D)))

    o = F.scaled_dot_product_attention(inter(q), inter(k), inter(v), is_causal=True).numpy()
    return o.reshape(B, H // 2, T, 2, D).transpose(0, 2, 1, 3, 4).reshape(B, T, H, D)


def test_paired_page_interleave_order(oracle):
    # q = 0: every visible position gets the same weight, so with one-hot values
    # marking each (token, head) the output lists exactly the visible positions.
    order, _ = golden()
    T, H, D = 3, 2, len(order)
    v = np.zeros((1, T, H, D))
    for pos, (tok, head) in enumerate(order):
        v[0, tok - 1, head - 1, pos] = 1.0
    q = np.zeros((1, T, H, D))
    k = rng_arrays(310, (1, T, H, D))[0]
    out = oracle.paired_fwd(q, k, v)
    for t in range(T):
        for e in range(H):
            n = order.index((t + 1, e + 1)) + 1          # positions up to and including its own
            want = np.zeros(D)
            want[:n] = 1.0 / n
            np.testing.assert_allclose(out[0, t, e], want, rtol=0, atol=1e-15)


def test_paired_page_visibility_example(oracle):
    _, visible = golden()
    T, H, D = 4, 2, 8
    q, k, v = rng_arrays(311, (1, T, H, D), (1, T, H, D), (1, T, H, D))
    base = oracle.paired_fwd(q, k, v)
    for tq, hq, hk, first, last in visible:
        for tk in range(1, T + 1):
            k2, v2 = k.copy(), v.copy()
            k2[0, tk - 1, hk - 1] += 1.5
            v2[0, tk - 1, hk - 1] += 2.0
            out = oracle.paired_fwd(q, k2, v2)
            moved = np.abs(out[0, tq - 1, hq - 1] - base[0, tq - 1, hq - 1]).max()
            if first <= tk <= last:
                assert moved > 1e-6, (tq, hq, hk, tk)
            else:
                assert moved == 0.0, (tq, hq, hk, tk)


def test_paired_matches_library_sdpa_on_interleaved(oracle):
    q, k, v = rng_arrays(312, (2, 13, 4, 8), (2, 13, 4, 8), (2, 13, 4, 8))
    np.testing.assert_allclose(oracle.paired_fwd(q, k, v), library_paired(q, k, v), rtol=1e-12, atol=1e-12)
    rows = np.array([0, 5, 51, 103])
    np.testing.assert_allclose(oracle.paired_fwd(q, k, v, rows=rows),
                               library_paired(q, k, v).reshape(-1, 8)[rows], rtol=1e-12, atol=1e-12)


def test_paired_closed_forms(oracle):
    D = 8
    # T = 1: the first head sees only its own key; the second sees both keys of the token
    q, k, v = rng_arrays(313, (3, 1, 2, D), (3, 1, 2, D), (3, 1, 2, D))
    out = oracle.paired_fwd(q, k, v)
    np.testing.assert_allclose(out[:, 0, 0], v[:, 0, 0], rtol=0, atol=1e-15)
    s = np.einsum("bd,bhd->bh", q[:, 0, 1], k[:, 0]) / np.sqrt(D)
    w = np.exp(s - s.max(1, keepdims=True))
    w /= w.sum(1, keepdims=True)
    np.testing.assert_allclose(out[:, 0, 1], np.einsum("bh,bhd->bd", w, v[:, 0]), rtol=1e-13)
    # identical heads: the second head's query at token t sees every key of
    # tokens 0..t twice -- plain causal attention; the first sees token t once
    T = 9
    q1, k1, v1 = rng_arrays(314, (1, T, 1, D), (1, T, 1, D), (1, T, 1, D))
    q, k, v = (np.concatenate([x, x], axis=2) for x in (q1, k1, v1))
    out = oracle.paired_fwd(q, k, v)
    plain = F.scaled_dot_product_attention(*(torch.from_numpy(x.transpose(0, 2, 1, 3).copy()) for x in (q1, k1, v1)),
                                           is_causal=True).numpy().transpose(0, 2, 1, 3)
    np.testing.assert_allclose(out[:, :, 1], plain[:, :, 0], rtol=1e-12, atol=1e-13)
    for t in range(T):
        x = k1[0, :t + 1, 0] @ q1[0, t, 0] / np.sqrt(D)
        m = np.full(t + 1, 2.0)
        m[t] = 1.0
        w = m * np.exp(x - x.max())
        np.testing.assert_allclose(out[0, t, 0], (w / w.sum()) @ v1[0, :t + 1, 0], rtol=1e-12, atol=1e-13)
