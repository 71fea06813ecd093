"""Inputs that drive the prefill kernels' online softmax through its rare
branches, and a host-side check that they do.

The one-pass prefill keeps, per query row and branch, a reference maximum
m_ref (scores in log2 units, s * log2(e) / sqrt(d)) and rescales the O
accumulator in tensor memory only when a later key tile's maximum exceeds
m_ref by more than 8; in between, P = 2^(s - m_ref) may grow up to 2^8.
With q, k ~ N(0, 1) the first key tile's maximum is never exceeded by that
much, so plain random inputs never take the rescale.  Here channel 0 of
every query holds a constant ``A`` and channel 0 of every key a value chosen
so that the key tile containing it scores about ``target[tile]`` log2 units
above the noise of the other channels: the targets step up by more than 8
at some tiles (a rescale), by 4 to 8 at others (P up to 2^8 under a stale
maximum) and step down at others.

``walk_decisions`` replays the kernel's decision rule on the exact scores of
the rounded inputs (fp64) so that a test can assert, before any launch, that
the inputs take both branches.  It is test infrastructure: it computes no
output of the method, only which branch each (row, key tile) takes.
"""
from __future__ import annotations

import math

import numpy as np
import torch

LOG2E = 1.4426950408889634
A = 8.0            # channel 0 of every query
THRESH = 8.0       # the kernel's rescale threshold, log2 units

# per key tile: the tile's planted score level (log2 units); steps of
# +5 (no rescale, P up to 2^5), +8.5 (rescale), -1.5, +7 (stale max, P up to
# 2^7), +11 (rescale), -3, +7.5, +13 (rescale), ... repeated with an offset
_PATTERN = [0.0, 5.0, 13.5, 12.0, 19.0, 30.0, 27.0, 34.5, 47.5, 40.0, 55.0, 61.0, 75.0, 71.0, 78.0, 90.0]


def targets(n_tiles: int, shift: int = 0) -> np.ndarray:
    """Planted level of each key tile; a branch may use a shifted pattern."""
    out = []
    for j in range(n_tiles):
        k = j + shift
        out.append(_PATTERN[k % len(_PATTERN)] + 90.0 * (k // len(_PATTERN)) - _PATTERN[shift % len(_PATTERN)])
    return np.asarray(out)


def key_channel0(n_keys: int, d: int, tgt: np.ndarray, keys_per_tile: int = 128) -> torch.Tensor:
    """Channel-0 value of each key so that A * k0 * log2(e) / sqrt(d) rises
    from tgt[tile] to tgt[tile] + 0.5 across the tile."""
    j = np.arange(n_keys)
    lvl = tgt[j // keys_per_tile] + 0.5 * (j % keys_per_tile) / keys_per_tile
    return torch.from_numpy(lvl * math.sqrt(d) / (LOG2E * A)).float()


def plant_v1(x: dict, d: int):
    """V1 inputs (make_v1 layout): branch 1 follows the pattern, branch 2 the
    pattern shifted by three tiles."""
    T = x["q"].shape[1]
    n = (T + 127) // 128
    x["q"][:, :, :, 0] = A
    k0_1 = key_channel0(T, d, targets(n, 0)).to(x["k"].dtype)
    k0_2 = key_channel0(T, d, targets(n, 3)).to(x["k"].dtype)
    x["k"][:, :, 0::2, 0] = k0_1[None, :, None]
    x["k"][:, :, 1::2, 0] = k0_2[None, :, None]


def plant_v2(x: dict, D: int):
    T = x["q"].shape[1]
    x["q"][:, :, :, 0] = A
    x["k"][:, :, :, 0] = key_channel0(T, D, targets((T + 127) // 128)).to(x["k"].dtype)[None, :, None]


def plant_paired(x: dict, D: int):
    """Paired Head Attention: key tiles are 128 interleaved positions = 64
    tokens of both heads of a pair."""
    T = x["q"].shape[1]
    x["q"][:, :, :, 0] = A
    x["k"][:, :, :, 0] = key_channel0(T, D, targets((2 * T + 127) // 128), keys_per_tile=64).to(
        x["k"].dtype)[None, :, None]


def walk_decisions(q: torch.Tensor, k: torch.Tensor, limit, n_tiles_of_row, keys_per_tile: int = 128):
    """Replay the online-softmax decisions for the rows of one head.

    q (R, d) query rows, k (N, d) keys (exact rounded values), limit[r] the
    last key row r sees, n_tiles_of_row[r] the key tiles the kernel walks for
    row r.  Returns (rescales, stale): per row, the number of key tiles after
    the first whose maximum rose above m_ref + 8 (the kernel rescales O), and
    the largest exponent s - m_ref of a P value written under a maximum that
    was not updated (between 0 and 8)."""
    q64, k64 = q.double(), k.double()
    s = (q64 @ k64.T) * (LOG2E / math.sqrt(q.shape[1]))
    R, N = s.shape
    col = torch.arange(N)
    s = torch.where(col[None, :] <= torch.as_tensor(limit)[:, None], s, torch.full_like(s, -math.inf))
    n_t = (N + keys_per_tile - 1) // keys_per_tile
    pad = n_t * keys_per_tile - N
    if pad:
        s = torch.cat([s, torch.full((R, pad), -math.inf, dtype=s.dtype)], 1)
    tmax = s.view(R, n_t, keys_per_tile).max(-1).values.numpy()
    resc = np.zeros(R, dtype=np.int64)
    stale = np.zeros(R)
    for r in range(R):
        m_ref = -math.inf
        for j in range(int(n_tiles_of_row[r])):
            m_new = max(m_ref, tmax[r, j])
            if m_new > m_ref + THRESH:
                if j > 0:
                    resc[r] += 1
                m_ref = m_new
            elif j > 0 and tmax[r, j] > -math.inf:
                stale[r] = max(stale[r], tmax[r, j] - m_ref)
    return resc, stale


def v1_decisions(x: dict, b: int, h: int, branch: int):
    T = x["q"].shape[1]
    q = (x["q1"] if branch == 0 else x["q2"])[b, :, h]
    k = (x["k1"] if branch == 0 else x["k2"])[b, :, h]
    t = np.arange(T)
    return walk_decisions(q, k, t, t // 128 + 1)


def v2_decisions(x: dict, b: int, head: int, G: int):
    T = x["q"].shape[1]
    t = np.arange(T)
    return walk_decisions(x["q"][b, :, head], x["k"][b, :, head // G], t, t // 128 + 1)


def paired_decisions(x: dict, b: int, head: int):
    """Row t of head 2i + e sees interleaved positions 0 .. 2t + e; the kernel
    walks key tiles 0 .. min(2 qt + 2, tiles) - 1 for query tile qt."""
    T = x["q"].shape[1]
    i, e = head // 2, head % 2
    kk = torch.stack([x["k"][b, :, 2 * i], x["k"][b, :, 2 * i + 1]], 1).reshape(2 * T, -1)
    t = np.arange(T)
    n_kt = (2 * T + 127) // 128
    return walk_decisions(x["q"][b, :, head], kk, 2 * t + e, np.minimum(2 * (t // 128) + 2, n_kt))
