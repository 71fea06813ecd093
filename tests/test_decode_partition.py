"""Host-side check of the split-KV decode's work partition (no GPU).

The decode kernels split the flat list of 64-key units over (sequence b,
kv head g, key block) evenly across `grid` CTAs: CTA c takes units
[c N / grid, (c+1) N / grid).  Each CTA writes one partial per (b, g) segment
it touches into slot (b * Hkv + g) + c, and the combine for (b, g) reads the
CTAs from cta_of(first unit) to cta_of(last unit), skipping CTAs whose range
is empty.  These tests restate that arithmetic and check, for uniform and
per-sequence lengths and for any grid, that
  * every slot index is unique and below B * Hkv + grid - 1 (the workspace);
  * the CTAs the combine reads for a segment are exactly those that wrote it.
"""
import numpy as np
import pytest

KEYS = 64


def partition(lens, Hkv, L, num_sms):
    B = len(lens)
    sb = [(n + KEYS - 1) // KEYS for n in lens]
    cum = np.concatenate([[0], np.cumsum([Hkv * x for x in sb])])
    N = int(cum[-1])
    grid = min(B * Hkv * ((L + KEYS - 1) // KEYS), num_sms)   # planned on the host from L
    seq = np.repeat(np.arange(B), [Hkv * x for x in sb])
    written = set()
    for c in range(grid):
        for u in range(c * N // grid, (c + 1) * N // grid):
            b = int(seq[u])
            g = (u - int(cum[b])) // sb[b]
            written.add((b * Hkv + g, c))
    return B, sb, cum, N, grid, written


def combine_ctas(b, g, sb, cum, N, grid):
    f = int(cum[b]) + g * sb[b]
    cta_of = lambda u: ((u + 1) * grid - 1) // N  # noqa: E731
    return {c for c in range(cta_of(f), cta_of(f + sb[b] - 1) + 1) if c * N // grid != (c + 1) * N // grid}


def check(lens, Hkv, L, num_sms):
    B, sb, cum, N, grid, written = partition(lens, Hkv, L, num_sms)
    slots = [bg + c for bg, c in written]
    assert len(slots) == len(set(slots))
    assert max(slots) <= B * Hkv + grid - 2
    for b in range(B):
        for g in range(Hkv):
            want = {c for bg, c in written if bg == b * Hkv + g}
            assert want and combine_ctas(b, g, sb, cum, N, grid) == want


@pytest.mark.parametrize("num_sms", [152, 33, 7, 1])
def test_uniform_lengths(num_sms):
    for B, L, Hkv in [(64, 32768, 8), (1, 1, 1), (3, 65, 2), (40, 130, 8), (5, 4097, 4)]:
        check([L] * B, Hkv, L, num_sms)


@pytest.mark.parametrize("num_sms", [152, 33, 7, 1])
def test_per_sequence_lengths(num_sms):
    r = np.random.default_rng(num_sms)
    for _ in range(150):
        B = int(r.integers(1, 40))
        L = int(r.integers(1, 3000))
        Hkv = int(r.choice([1, 2, 4, 8, 12]))
        check(list(r.integers(1, L + 1, B)), Hkv, L, num_sms)


def test_short_sequences_leave_ctas_without_units():
    """The case that needs the skip: 120 units over 152 CTAs (lengths 1, 63,
    64, 65, 777, 705 with 4 kv heads)."""
    lens = [1, 63, 64, 65, 777, 705]
    B, sb, cum, N, grid, written = partition(lens, 4, 777, 152)
    assert N < grid
    check(lens, 4, 777, 152)
