"""The allocation-free decode entry point, diffattn_v2_decode_noalloc.

Some callers may not allocate device memory themselves -- a host framework
that owns all device memory through its own pool and passes this library only
inputs and outputs, or a decode loop that cannot take the device-wide
synchronisation a cudaMalloc may cause.  For them the library keeps the
split-KV partials in its own static 8 MiB device buffer.  These tests call that
entry point through the C ABI and check it against diffattn_v2_decode (the
workspace entry point) within the bf16 tolerance used by every parity test,
on two calls in a row whose shapes differ, and check that sizes beyond the
buffer are refused.  This file sorts last so that a run stopping at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

from differential_attention_causal_gb300 import inputs

pytestmark = pytest.mark.gpu

BF16_ATOL, BF16_RL2 = 2e-2, 5e-3
SCRATCH_LIMIT = 8 << 20


@pytest.fixture(scope="module")
def lib():
    from differential_attention_causal_gb300 import build as b
    b.build()
    torch.cuda.set_device(0)
    from differential_attention_causal_gb300 import binding
    return binding.lib()


def _noalloc(lib, x, out):
    q, k, v, lam = x["q"], x["k_cache"], x["v_cache"], x["lam"]
    B, Hq, D = q.shape
    L, Hkv = k.shape[1], k.shape[2]
    return lib.diffattn_v2_decode_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(lam.data_ptr()), ctypes.c_void_p(out.data_ptr()), B, L, Hq, Hkv, D, 1,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_decode_matches_workspace_decode_on_two_calls(lib):
    from differential_attention_causal_gb300 import binding
    shapes = [inputs.DecodeShape(3, 1000, 16, 2, 128, "bf16"),
              inputs.DecodeShape(5, 4097, 32, 4, 128, "bf16")]
    for call, s in enumerate(shapes):
        x = inputs.make_decode(s, seed=100 + call, device="cuda")
        assert binding.decode_workspace_size(s.B, s.L, s.Hq, s.Hkv, s.D) <= SCRATCH_LIMIT
        ref = binding.v2_decode(x["q"], x["k_cache"], x["v_cache"], x["lam"])
        out = torch.full_like(ref, float("nan"))
        rc = _noalloc(lib, x, out)
        assert rc == 0, binding.status_string(rc)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        want = ref.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        err = np.abs(got - want).max()
        rl2 = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert err <= BF16_ATOL and rl2 <= BF16_RL2, (call, err, rl2)
        assert binding.device_error() == 0


def test_noalloc_refuses_sizes_beyond_its_scratch(lib):
    from differential_attention_causal_gb300 import binding
    # many short sequences: one partial slot per (b, kv head), plus one per CTA, overflows 8 MiB
    s = inputs.DecodeShape(300, 64, 16, 8, 128, "bf16")
    assert binding.decode_workspace_size(s.B, s.L, s.Hq, s.Hkv, s.D) > SCRATCH_LIMIT
    x = inputs.make_decode(s, seed=7, device="cuda")
    out = torch.zeros((s.B, s.Hq // 2, s.D), dtype=torch.bfloat16, device="cuda")
    rc = _noalloc(lib, x, out)
    assert rc == 10 and "8 MiB" in binding.status_string(rc)
    torch.cuda.synchronize()
    assert out.abs().max().item() == 0.0          # nothing was enqueued
    with pytest.raises(binding.DiffAttnError):
        binding.v2_decode_noalloc(x["q"], x["k_cache"], x["v_cache"], x["lam"], out=out)
