"""The allocation-free decode entry point, diffattn_v2_decode_noalloc.

Some callers may not allocate device memory themselves -- a host framework
that owns all device memory through its own pool and passes this library only
inputs and outputs, or a decode loop that cannot take the device-wide
synchronisation a cudaMalloc may cause.  For them the library keeps the
split-KV partials in its own static 8 MiB device buffer.  These tests call that
entry point through the C ABI and check it against diffattn_v2_decode (the
workspace entry point), on two calls in a row whose shapes differ: both run
the same plan and kernels on the same inputs, so their outputs must be equal
bit for bit (a partial read from a wrong or stale slot would show up even
where it moves a result by less than the bf16 tolerance).  They also check
that sizes beyond the buffer are refused, and that an invalid call gets the
same status from both entry points.  This file sorts last so that a run stopping at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import pytest
import torch

from differential_attention_causal_gb300 import inputs

pytestmark = pytest.mark.gpu

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
        assert torch.isfinite(out.float()).all()
        assert torch.equal(out, ref), (call, (out.float() - ref.float()).abs().max().item())
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


def test_noalloc_checks_arguments_before_the_scratch_limit(lib):
    """A call that is both invalid and too large for the buffer reports the
    argument error, the same status the workspace entry point gives."""
    from differential_attention_causal_gb300 import binding
    # G = 16 query heads per kv head: more than the bf16 decode supports, and
    # B x Hkv partial slots far beyond 8 MiB
    B, L, Hq, Hkv, D = 4096, 64, 32, 2, 128
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, L, Hkv, D), dtype=torch.bfloat16, device="cuda")
    lam = torch.zeros((B, Hq // 2), dtype=torch.float32, device="cuda")
    out = torch.zeros((B, Hq // 2, D), dtype=torch.bfloat16, device="cuda")
    x = {"q": q, "k_cache": k, "v_cache": k, "lam": lam}
    rc = _noalloc(lib, x, out)
    assert rc == 4, binding.status_string(rc)          # DA_ERR_BAD_GROUP, not DA_ERR_SCRATCH_LIMIT
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    rc2 = lib.diffattn_v2_decode(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                 ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(lam.data_ptr()),
                                 ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                 B, L, Hq, Hkv, D, 1, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc2 == rc
    torch.cuda.synchronize()
    assert out.abs().max().item() == 0.0
