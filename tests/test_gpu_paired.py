"""GPU parity of Paired Head Attention (modded-nanogpt pull request "New
Record: Paired Head Attention (-3.5s, -65 steps)") through the C ABI against
the fp64 oracle.  bf16 tolerance: max abs error <= 2e-2 and relative L2
<= 5e-3, as for the other bf16 paths.  The shapes span several 128-position
key tiles of the interleaved sequence (2T positions) and ragged tails; the
full-size workload is checked on sampled rows in the bench's launch.
"""
import numpy as np
import pytest
import torch

import oracle
from differential_attention_causal_gb300 import inputs
from test_gpu_parity import assert_parity, to_dev

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("B,T,H,D", [(2, 200, 4, 128), (1, 129, 2, 128), (1, 1, 2, 128), (1, 64, 2, 128),
                                     (2, 150, 4, 64), (1, 384, 8, 64), (1, 65, 2, 64), (3, 97, 6, 128)])
def test_paired_bf16(B, T, H, D):
    s = inputs.PairedShape(B, T, H, D, "bf16")
    x = inputs.make_paired(s, seed=T + H)
    xd = to_dev(x)
    y = binding().paired_fwd(xd["q"], xd["k"], xd["v"])
    assert_parity(y, oracle.paired_fwd(x["q"], x["k"], x["v"]), "bf16")


def test_paired_bf16_identical_heads_and_no_stray_writes():
    # the second head of each pair a copy of the first: its output is plain
    # causal attention of the first head (every key counted twice); the
    # output buffer is followed by a guard that must stay untouched
    B, T, H, D = 2, 211, 4, 128
    x = inputs.make_paired(inputs.PairedShape(B, T, H, D, "bf16"), seed=3)
    for n in ("q", "k", "v"):
        x[n][:, :, 1::2] = x[n][:, :, 0::2]
    xd = to_dev(x)
    n = B * T * H * D
    buf = torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[:n].view(B, T, H, D)
    binding().paired_fwd(xd["q"], xd["k"], xd["v"], out=out)
    torch.cuda.synchronize()
    assert bool((buf[n:] == 7.0).all())
    assert_parity(out, oracle.paired_fwd(x["q"], x["k"], x["v"]), "bf16")


def test_paired_bf16_full_workload_sampled():
    """B=8, T=4096, H=32 (16 pairs), D=128: sampled rows."""
    s = inputs.WORKLOADS["paired_bf16_B8_T4096_H32_D128"]
    x = inputs.make_paired(s, seed=0)
    xd = to_dev(x)
    y = binding().paired_fwd(xd["q"], xd["k"], xd["v"])
    rng = np.random.default_rng(2)
    ts = [0, 1, 63, 64, 127, 128, 2047, 4095]
    rows = [(b * s.T + t) * s.H + h for b in (0, s.B - 1) for h in range(s.H) for t in ts]
    rows += list(rng.integers(0, s.B * s.T * s.H, 300))
    rows = np.array(rows, dtype=np.int64)
    ref = oracle.paired_fwd(x["q"], x["k"], x["v"], rows=rows)
    assert_parity(y.reshape(-1, s.D)[torch.from_numpy(rows).cuda()], ref, "bf16")


@pytest.mark.slow
def test_paired_bf16_beyond_2_31_elements():
    """B=4096, T=136, H=32 (16 pairs), D=128: q, k, v and out hold 2^31 + 2^27
    elements each (4.6 GB); sampled rows of the first and last batch entries
    against the oracle (inputs drawn on the device)."""
    s = inputs.PairedShape(4096, 136, 32, 128, "bf16")
    assert s.B * s.T * s.H * s.D > 2 ** 31
    xd = inputs.make_paired(s, seed=7, device="cuda")
    y = binding().paired_fwd(xd["q"], xd["k"], xd["v"])
    assert binding().device_error() == 0
    rows = np.array([t * s.H + h for t in (0, 1, 63, 64, 127, 128, 135) for h in range(s.H)], dtype=np.int64)
    for b in (0, s.B - 1):
        xb = {n: xd[n][b:b + 1].contiguous().cpu() for n in ("q", "k", "v")}
        ref = oracle.paired_fwd(xb["q"], xb["k"], xb["v"], rows=rows)
        assert_parity(y[b].reshape(-1, s.D)[torch.from_numpy(rows).cuda()], ref, "bf16")
