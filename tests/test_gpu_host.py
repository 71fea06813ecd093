"""The end-to-end DIFF V1 call on host buffers (diffattn_v1_fwd_host): its
output equals the device call's bit for bit (the chunked forwards compute the
same tiles) and matches the fp64 oracle within the bf16 / fp32 tolerances;
the chunking over batch entries covers uneven splits (B = 9 and B = 17 over
8 chunks), single-entry calls and ragged last tiles, and the call is ordered
on a caller's stream."""
import numpy as np
import pytest
import torch

import oracle
from differential_attention_causal_gb300 import inputs
from test_gpu_parity import assert_parity, oracle_v1, run_v1, to_dev

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


def host_call(x, s, stream=None):
    bd = binding()
    pin = {n: x[n].contiguous().pin_memory() for n in ("q", "k", "v", "lam_q1", "lam_k1", "lam_q2", "lam_k2")}
    dt = torch.bfloat16 if s.dtype == "bf16" else torch.float32
    out = torch.empty((s.B, s.T, s.H, 2 * s.d), dtype=dt).pin_memory()
    ws = torch.empty(bd.v1_fwd_host_workspace_size(s.B, s.T, s.H, s.d, dt), dtype=torch.uint8, device="cuda")
    bd.v1_fwd_host(pin["q"], pin["k"], pin["v"], pin["lam_q1"], pin["lam_k1"], pin["lam_q2"], pin["lam_k2"],
                   s.layer_index, out, ws, stream=stream)
    (stream or torch.cuda.current_stream()).synchronize()
    return out, bd.last_launch_count()


def expected_launches(B, T, d, dtype):
    """Chunks of the host call: runs of batch entries, at most 8."""
    return min(B, 8)


@pytest.mark.parametrize("B,T,H,d,layer,dtype", [(3, 200, 2, 64, 1, "bf16"), (9, 129, 2, 64, 0, "bf16"),
                                                 (2, 300, 3, 128, 5, "bf16"), (2, 70, 2, 32, 2, "fp32"),
                                                 (3, 65, 2, 32, 3, "bf16"), (1, 1000, 2, 64, 4, "bf16"),
                                                 (2, 700, 2, 32, 6, "bf16"), (17, 130, 1, 64, 2, "bf16"),
                                                 (4, 1024, 2, 64, 12, "bf16")])
def test_v1_host_matches_device_call_and_oracle(B, T, H, d, layer, dtype):
    s = inputs.V1Shape(B, T, H, d, layer, dtype)
    x = inputs.make_v1(s, seed=B + T)
    got, launches = host_call(x, s)
    assert launches == expected_launches(B, T, d, dtype)
    dev = run_v1(to_dev(x), layer).cpu()
    assert torch.equal(got, dev)
    assert_parity(got, oracle_v1(x, layer), dtype)


def test_v1_host_on_a_side_stream():
    s = inputs.V1Shape(4, 256, 2, 64, 3, "bf16")
    x = inputs.make_v1(s, seed=11)
    side = torch.cuda.Stream()
    got, _ = host_call(x, s, stream=side)
    assert torch.equal(got, run_v1(to_dev(x), s.layer_index).cpu())
    assert binding().device_error() == 0
