"""ctypes binding over libdiffattn.so (the C ABI in include/diffattn.h).

Argument marshalling only: every step of the differential-attention forward
runs in the library's CUDA kernels.  torch is used for device memory and the
current CUDA stream.  If the library is missing this module raises at first
use -- there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdiffattn.so")
LIB_DEBUG_PATH = os.path.join(_HERE, "libdiffattn_debug.so")

DA_F32, DA_BF16 = 0, 1
STATUS = {
    0: "DA_OK", 1: "DA_ERR_NULL_PTR", 2: "DA_ERR_BAD_SHAPE", 3: "DA_ERR_UNSUPPORTED_DIM",
    4: "DA_ERR_BAD_GROUP", 5: "DA_ERR_MISALIGNED", 6: "DA_ERR_WORKSPACE_TOO_SMALL",
    7: "DA_ERR_CUDA", 8: "DA_ERR_BAD_DTYPE", 9: "DA_ERR_DEVICE_TIMEOUT", 10: "DA_ERR_SCRATCH_LIMIT",
    11: "DA_ERR_BAD_LENGTH", 12: "DA_ERR_DEVICE_BOUNDS",
}
_lock = threading.Lock()
_lib = None


class DiffAttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} returned {STATUS.get(code, code)}: {status_string(code)}")


def lib() -> ctypes.CDLL:
    """Load libdiffattn.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} not found: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            vp, fp, i32, i64 = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            L.diffattn_v1_fwd.restype = i32
            L.diffattn_v1_fwd.argtypes = ([vp] * 5 + [fp] * 4 + [vp] + [i32] * 5 + [i64] * 12 + [i32, vp])
            L.diffattn_v2_fwd.restype = i32
            L.diffattn_v2_fwd.argtypes = [vp, vp, vp, fp, vp] + [i32] * 5 + [i32, vp]
            L.diffattn_v1_fwd_host_workspace_size.restype = ctypes.c_size_t
            L.diffattn_v1_fwd_host_workspace_size.argtypes = [i32] * 5
            L.diffattn_v1_fwd_host.restype = i32
            L.diffattn_v1_fwd_host.argtypes = ([vp, vp, vp, fp, fp, fp, fp, vp] + [i32] * 5
                                               + [vp, ctypes.c_size_t, i32, vp])
            L.diffattn_v2_fwd_rope.restype = i32
            L.diffattn_v2_fwd_rope.argtypes = ([vp, vp, vp, fp, vp] + [i32] * 5 + [i64, ctypes.c_float]
                                               + [i32, vp])
            L.diffattn_paired_fwd.restype = i32
            L.diffattn_paired_fwd.argtypes = [vp, vp, vp, vp] + [i32] * 4 + [i32, vp]
            L.diffattn_v2_decode_workspace_size.restype = ctypes.c_size_t
            L.diffattn_v2_decode_workspace_size.argtypes = [i32] * 6
            L.diffattn_v2_decode.restype = i32
            L.diffattn_v2_decode.argtypes = ([vp, vp, vp, fp, vp, vp, ctypes.c_size_t] + [i32] * 5 + [i32, vp])
            L.diffattn_v2_decode_noalloc.restype = i32
            L.diffattn_v2_decode_noalloc.argtypes = [vp, vp, vp, fp, vp] + [i32] * 5 + [i32, vp]
            L.diffattn_v2_decode_varlen.restype = i32
            L.diffattn_v2_decode_varlen.argtypes = ([vp, vp, vp, fp, vp, vp, vp, ctypes.c_size_t] + [i32] * 5
                                                    + [i32, vp])
            L.diffattn_v1_decode_workspace_size.restype = ctypes.c_size_t
            L.diffattn_v1_decode_workspace_size.argtypes = [i32] * 5
            L.diffattn_v1_decode.restype = i32
            L.diffattn_v1_decode.argtypes = ([vp] * 5 + [fp] * 4 + [vp, vp, vp, ctypes.c_size_t] + [i32] * 5
                                             + [i32, vp])
            sz = ctypes.c_size_t
            for n, k in (("diffattn_v1_train_saved_size", 5), ("diffattn_v1_bwd_workspace_size", 5),
                         ("diffattn_v2_train_saved_size", 6), ("diffattn_v2_bwd_workspace_size", 6),
                         ("diffattn_v1_train_saved_lse_offset", 5), ("diffattn_v2_train_saved_lse_offset", 6)):
                getattr(L, n).restype = sz
                getattr(L, n).argtypes = [i32] * k
            L.diffattn_v1_fwd_train.restype = i32
            L.diffattn_v1_fwd_train.argtypes = ([vp] * 5 + [fp] * 4 + [vp, vp, sz] + [i32] * 5 + [i64] * 12
                                                + [i32, vp])
            L.diffattn_v1_bwd.restype = i32
            L.diffattn_v1_bwd.argtypes = ([vp] * 5 + [fp] * 4 + [vp, vp, sz] + [vp] * 5 + [fp] * 4 + [vp, sz]
                                          + [i32] * 5 + [i64] * 12 + [i32, vp])
            L.diffattn_v2_fwd_train.restype = i32
            L.diffattn_v2_fwd_train.argtypes = [vp, vp, vp, fp, vp, vp, sz] + [i32] * 5 + [i32, vp]
            L.diffattn_v2_bwd.restype = i32
            L.diffattn_v2_bwd.argtypes = ([vp, vp, vp, fp, vp, vp, sz, vp, vp, vp, fp, vp, sz] + [i32] * 5
                                          + [i32, vp])
            L.diffattn_prologue.restype = i32
            L.diffattn_prologue.argtypes = ([vp, vp] + [i32] * 5 + [i64, ctypes.c_float, vp, vp, fp] + [i32] * 2
                                            + [i32, vp])
            L.diffattn_status_string.restype = ctypes.c_char_p
            L.diffattn_status_string.argtypes = [i32]
            L.diffattn_device_error.restype = i32
            L.diffattn_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
            L.diffattn_stream_error.restype = i32
            L.diffattn_stream_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p]
            L.diffattn_selftest_wait_limit.restype = i32
            L.diffattn_selftest_wait_limit.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p]
            L.diffattn_last_launch_count.restype = i32
            L.diffattn_last_launch_count.argtypes = []
            L.diffattn_debug_checks.restype = i32
            L.diffattn_debug_checks.argtypes = []
            L.diffattn_selftest_bounds.restype = i32
            L.diffattn_selftest_bounds.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p]
            _lib = L
    return _lib


def use_library(debug: bool) -> str:
    """Route the calls of this module to libdiffattn_debug.so (debug=True: the
    kernels check the indices they write through, failures are reported as
    DA_ERR_DEVICE_BOUNDS by the error-word calls) or to the release library.
    Each library keeps its own error words.  Returns the path now in use."""
    global _lib, LIB_PATH
    with _lock:
        path = LIB_DEBUG_PATH if debug else os.path.join(_HERE, "libdiffattn.so")
        if path != LIB_PATH:
            LIB_PATH = path
            _lib = None
    return LIB_PATH


def debug_checks() -> bool:
    """True if the library in use was built with the bounds checks."""
    return bool(lib().diffattn_debug_checks())


def selftest_bounds(stream=None) -> int:
    """A warp tests an index past the end of a buffer through the kernels'
    bounds check (the write is skipped in both builds).  Returns the raw error
    word it left (debug build: the bounds bit; release: 0), cleared again;
    raises if the result is not the one of the build."""
    code = ctypes.c_uint32(0)
    rc = lib().diffattn_selftest_bounds(ctypes.byref(code), _stream(stream))
    if rc != 0:
        raise DiffAttnError("diffattn_selftest_bounds", rc)
    return int(code.value)


def status_string(code: int) -> str:
    return lib().diffattn_status_string(int(code)).decode()


def last_launch_count() -> int:
    """Kernel launches enqueued by the last successful call on this thread."""
    return lib().diffattn_last_launch_count()


def selftest_wait_limit(stream=None) -> int:
    """Failure-path self-test (about 2 s): a kernel whose bounded wait nothing
    completes must give up, record the timeout bit and leave the context usable.
    Returns the raw error word it recorded (cleared again); raises if the wait
    did not give up."""
    code = ctypes.c_uint32(0)
    rc = lib().diffattn_selftest_wait_limit(ctypes.byref(code), _stream(stream))
    if rc != 0:
        raise DiffAttnError("diffattn_selftest_wait_limit", rc)
    return int(code.value)


def device_error() -> int:
    """Synchronise the device, then read and clear every stream's error word
    (their OR; 0 = no kernel recorded anything)."""
    code = ctypes.c_uint32(0)
    rc = lib().diffattn_device_error(ctypes.byref(code))
    if rc not in (0, 9, 11, 12):
        raise DiffAttnError("diffattn_device_error", rc)
    return int(code.value)


def stream_error(stream=None) -> int:
    """Synchronise one stream (default: the current one), then read and clear
    its error word (0 = no kernel on it gave up)."""
    code = ctypes.c_uint32(0)
    rc = lib().diffattn_stream_error(ctypes.byref(code), _stream(stream))
    if rc not in (0, 9, 11, 12):
        raise DiffAttnError("diffattn_stream_error", rc)
    return int(code.value)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DA_BF16
    if t.dtype == torch.float32:
        return DA_F32
    raise TypeError(f"unsupported dtype {t.dtype}: use bfloat16 or float32")


def _cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _check(fn: str, rc: int):
    if rc != 0:
        raise DiffAttnError(fn, rc)


def v1_fwd(q1, q2, k1, k2, v, lam_q1, lam_k1, lam_q2, lam_k2, layer_index: int,
           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """DIFF V1 causal forward ("Differential Transformer V2", DiffAttnV1).

    q1, q2, k1, k2: (B, T, H, d) CUDA tensors with the last dim contiguous
    (strided views such as q[:, :, 0::2] of an interleaved (B, T, 2H, d)
    tensor are passed as is); q1/q2 and k1/k2 must share strides.
    v: (B, T, H, 2d).  lam_*: fp32 (d,).  Returns out (B, T, H, 2d).
    """
    for n, t in (("q1", q1), ("q2", q2), ("k1", k1), ("k2", k2), ("v", v)):
        _cuda(t, n)
    B, T, H, d = q1.shape
    if out is None:
        out = torch.empty((B, T, H, 2 * d), dtype=q1.dtype, device=q1.device)
    if q1.stride() != q2.stride() or k1.stride() != k2.stride():
        raise ValueError("q1/q2 and k1/k2 must share strides")
    for t in (q1, k1, v, out):
        if t.stride(-1) != 1:
            raise ValueError("head dimension must be contiguous")
    lams = [x.contiguous() for x in (lam_q1, lam_k1, lam_q2, lam_k2)]
    for x in lams:
        if x.dtype != torch.float32 or not x.is_cuda or x.numel() != d:
            raise ValueError("lambda vectors must be fp32 CUDA tensors of length d")
    dt = _dtype_code(q1)
    qs, ks, vs, os_ = q1.stride(), k1.stride(), v.stride(), out.stride()
    rc = lib().diffattn_v1_fwd(
        q1.data_ptr(), q2.data_ptr(), k1.data_ptr(), k2.data_ptr(), v.data_ptr(),
        *[x.data_ptr() for x in lams], out.data_ptr(),
        B, T, H, d, int(layer_index),
        qs[0], qs[1], qs[2], ks[0], ks[1], ks[2], vs[0], vs[1], vs[2], os_[0], os_[1], os_[2],
        dt, _stream(stream))
    _check("diffattn_v1_fwd", rc)
    return out


def v2_fwd(q, k, v, lam, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """DIFF V2 causal prefill ("Differential Transformer V2", DiffAttnV2).

    q: (B, T, Hq, D), k, v: (B, T, Hkv, D), lam: (B, T, Hq/2) fp32 logits,
    all contiguous CUDA tensors.  Returns out (B, T, Hq/2, D).
    """
    for n, t in (("q", q), ("k", k), ("v", v), ("lam", lam)):
        _cuda(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    if lam.dtype != torch.float32:
        raise ValueError("lam must be fp32")
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty((B, T, Hq // 2, D), dtype=q.dtype, device=q.device)
    rc = lib().diffattn_v2_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), lam.data_ptr(), out.data_ptr(),
                               B, T, Hq, Hkv, D, _dtype_code(q), _stream(stream))
    _check("diffattn_v2_fwd", rc)
    return out


def v2_fwd_rope(q, k, v, lam, pos0: int = 0, base: float = 10000.0, out: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """DIFF V2 causal prefill of rotary-embedded q and k: the same result as
    prologue(q, k, pos0, base) followed by v2_fwd, with q left unchanged (its
    tiles are rotated inside the prefill kernel) and k rotated in place.

    Shapes as for v2_fwd (bf16).  Returns out."""
    for n, t in (("q", q), ("k", k), ("v", v), ("lam", lam)):
        _cuda(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    if lam.dtype != torch.float32:
        raise ValueError("lam must be fp32")
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty((B, T, Hq // 2, D), dtype=q.dtype, device=q.device)
    rc = lib().diffattn_v2_fwd_rope(q.data_ptr(), k.data_ptr(), v.data_ptr(), lam.data_ptr(), out.data_ptr(),
                                    B, T, Hq, Hkv, D, int(pos0), float(base), _dtype_code(q), _stream(stream))
    _check("diffattn_v2_fwd_rope", rc)
    return out


def v1_fwd_host_workspace_size(B: int, T: int, H: int, d: int, dtype=torch.bfloat16) -> int:
    code = DA_BF16 if dtype == torch.bfloat16 else DA_F32
    return int(lib().diffattn_v1_fwd_host_workspace_size(B, T, H, d, code))


def v1_fwd_host(q, k, v, lam_q1, lam_k1, lam_q2, lam_k2, layer_index: int, out: torch.Tensor,
                workspace: torch.Tensor, stream=None) -> torch.Tensor:
    """DIFF V1 forward on HOST tensors (the end-to-end call): q, k (B, T, 2H, d)
    interleaved and v (B, T, H, 2d) contiguous CPU tensors (pinned for the
    copies to overlap), the four lambda vectors fp32 CPU tensors, `out`
    (B, T, H, 2d) a CPU tensor, `workspace` a uint8 CUDA tensor of
    v1_fwd_host_workspace_size() bytes.  Ordered on the current stream."""
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out), ("lam_q1", lam_q1), ("lam_k1", lam_k1),
                 ("lam_q2", lam_q2), ("lam_k2", lam_k2)):
        if t.is_cuda:
            raise ValueError(f"{n} must be a host tensor")
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    _cuda(workspace, "workspace")
    for t in (lam_q1, lam_k1, lam_q2, lam_k2):
        if t.dtype != torch.float32:
            raise ValueError("lambda vectors must be fp32")
    B, T, H2, d = q.shape
    rc = lib().diffattn_v1_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), lam_q1.data_ptr(),
                                    lam_k1.data_ptr(), lam_q2.data_ptr(), lam_k2.data_ptr(), out.data_ptr(),
                                    B, T, H2 // 2, d, layer_index, workspace.data_ptr(), workspace.numel(),
                                    _dtype_code(q), _stream(stream))
    _check("diffattn_v1_fwd_host", rc)
    return out


def paired_fwd(q, k, v, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Paired Head Attention, causal (modded-nanogpt pull request "New Record:
    Paired Head Attention (-3.5s, -65 steps)"): heads 2i and 2i+1 interleaved
    into one sequence of 2T positions with one softmax.

    q, k, v: (B, T, H, D) contiguous bf16 CUDA tensors, H even, D in {64, 128}.
    Returns out (B, T, H, D).
    """
    for n, t in (("q", q), ("k", k), ("v", v)):
        _cuda(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must have the same shape")
    B, T, H, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    rc = lib().diffattn_paired_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, T, H, D,
                                   _dtype_code(q), _stream(stream))
    _check("diffattn_paired_fwd", rc)
    return out


def decode_workspace_size(B: int, L: int, Hq: int, Hkv: int, D: int, dtype=torch.bfloat16) -> int:
    code = DA_BF16 if dtype == torch.bfloat16 else DA_F32
    return int(lib().diffattn_v2_decode_workspace_size(B, L, Hq, Hkv, D, code))


def v2_decode(q, k_cache, v_cache, lam, out: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """DIFF V2 single-token decode against a KV cache.

    q: (B, Hq, D); k_cache, v_cache: (B, L, Hkv, D); lam: (B, Hq/2) fp32.
    workspace: optional uint8 CUDA tensor of at least decode_workspace_size()
    bytes (allocated here with torch when omitted).  Returns out (B, Hq/2, D).
    """
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("lam", lam)):
        _cuda(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    B, Hq, D = q.shape
    L, Hkv = k_cache.shape[1], k_cache.shape[2]
    if out is None:
        out = torch.empty((B, Hq // 2, D), dtype=q.dtype, device=q.device)
    need = decode_workspace_size(B, L, Hq, Hkv, D, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = lib().diffattn_v2_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), lam.data_ptr(),
                                  out.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                  B, L, Hq, Hkv, D, _dtype_code(q), _stream(stream))
    _check("diffattn_v2_decode", rc)
    return out


def v2_decode_noalloc(q, k_cache, v_cache, lam, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """DIFF V2 decode through ``diffattn_v2_decode_noalloc``: no workspace, no
    allocation inside the library (its split-KV partials use the library's
    static 8 MiB device buffer).  For callers that may not allocate device
    memory; ``out`` may be passed in so that this wrapper allocates nothing
    either.  Calls that overlap on the GPU share that buffer and must be
    ordered.  Raises DiffAttnError (DA_ERR_SCRATCH_LIMIT) when the sizes need
    more scratch than the buffer holds."""
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("lam", lam)):
        _cuda(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    B, Hq, D = q.shape
    L, Hkv = k_cache.shape[1], k_cache.shape[2]
    if out is None:
        out = torch.empty((B, Hq // 2, D), dtype=q.dtype, device=q.device)
    rc = lib().diffattn_v2_decode_noalloc(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), lam.data_ptr(),
                                          out.data_ptr(), B, L, Hq, Hkv, D, _dtype_code(q), _stream(stream))
    _check("diffattn_v2_decode_noalloc", rc)
    return out


def _lens_arg(cache_lens, B: int, device) -> torch.Tensor:
    if not isinstance(cache_lens, torch.Tensor) or not cache_lens.is_cuda:
        raise ValueError("cache_lens must be a CUDA tensor")
    if cache_lens.dtype != torch.int32 or cache_lens.numel() != B or not cache_lens.is_contiguous():
        raise ValueError("cache_lens must be a contiguous int32 tensor of B lengths")
    return cache_lens


def v2_decode_varlen(q, k_cache, v_cache, lam, cache_lens, out: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """DIFF V2 decode with a cache length per sequence: sequence b attends
    cache rows 0 .. cache_lens[b]-1.  cache_lens: int32 CUDA tensor (B,), each
    in 1..L (a length out of range is clamped and reported by device_error()).
    Other arguments as v2_decode."""
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("lam", lam)):
        _cuda(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    B, Hq, D = q.shape
    L, Hkv = k_cache.shape[1], k_cache.shape[2]
    _lens_arg(cache_lens, B, q.device)
    if out is None:
        out = torch.empty((B, Hq // 2, D), dtype=q.dtype, device=q.device)
    need = decode_workspace_size(B, L, Hq, Hkv, D, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = lib().diffattn_v2_decode_varlen(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), lam.data_ptr(),
                                         cache_lens.data_ptr(), out.data_ptr(), workspace.data_ptr(),
                                         workspace.numel(), B, L, Hq, Hkv, D, _dtype_code(q), _stream(stream))
    _check("diffattn_v2_decode_varlen", rc)
    return out


def v1_decode_workspace_size(B: int, L: int, H: int, d: int, dtype=torch.bfloat16) -> int:
    code = DA_BF16 if dtype == torch.bfloat16 else DA_F32
    return int(lib().diffattn_v1_decode_workspace_size(B, L, H, d, code))


def v1_decode(q1, q2, k1_cache, k2_cache, v_cache, lam_q1, lam_k1, lam_q2, lam_k2, layer_index: int,
              cache_lens=None, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """DIFF V1 single-token decode ("Differential Transformer V2", DiffAttnV1
    for one new token per sequence).

    q1, q2: (B, H, d); k1_cache, k2_cache: (B, L, H, d); v_cache: (B, L, H, 2d),
    all contiguous CUDA tensors; lam_*: fp32 (d,); cache_lens: optional int32
    CUDA tensor (B,) of rows attended per sequence (default all L).
    Returns out (B, H, 2d).
    """
    for n, t in (("q1", q1), ("q2", q2), ("k1_cache", k1_cache), ("k2_cache", k2_cache), ("v_cache", v_cache)):
        _cuda(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    B, H, d = q1.shape
    L = k1_cache.shape[1]
    lams = [x.contiguous() for x in (lam_q1, lam_k1, lam_q2, lam_k2)]
    for x in lams:
        if x.dtype != torch.float32 or not x.is_cuda or x.numel() != d:
            raise ValueError("lambda vectors must be fp32 CUDA tensors of length d")
    lens_ptr = None
    if cache_lens is not None:
        lens_ptr = _lens_arg(cache_lens, B, q1.device).data_ptr()
    if out is None:
        out = torch.empty((B, H, 2 * d), dtype=q1.dtype, device=q1.device)
    ws_ptr, ws_bytes = None, 0
    if q1.dtype == torch.bfloat16:
        need = v1_decode_workspace_size(B, L, H, d, q1.dtype)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q1.device)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    rc = lib().diffattn_v1_decode(q1.data_ptr(), q2.data_ptr(), k1_cache.data_ptr(), k2_cache.data_ptr(),
                                  v_cache.data_ptr(), *[x.data_ptr() for x in lams], lens_ptr, out.data_ptr(),
                                  ws_ptr, ws_bytes, B, L, H, d, int(layer_index), _dtype_code(q1),
                                  _stream(stream))
    _check("diffattn_v1_decode", rc)
    return out


# ------------------------------------------------------------------ training

def _v1_strides(q1, q2, k1, k2, v, t_out):
    if q1.stride() != q2.stride() or k1.stride() != k2.stride():
        raise ValueError("q1/q2 and k1/k2 must share strides")
    for t in (q1, k1, v, t_out):
        if t.stride(-1) != 1:
            raise ValueError("head dimension must be contiguous")
    qs, ks, vs, os_ = q1.stride(), k1.stride(), v.stride(), t_out.stride()
    return [qs[0], qs[1], qs[2], ks[0], ks[1], ks[2], vs[0], vs[1], vs[2], os_[0], os_[1], os_[2]]


def _lam_vecs(d, *xs):
    out = [x.contiguous() for x in xs]
    for x in out:
        if x.dtype != torch.float32 or not x.is_cuda or x.numel() != d:
            raise ValueError("lambda vectors must be fp32 CUDA tensors of length d")
    return out


def v1_fwd_train(q1, q2, k1, k2, v, lam_q1, lam_k1, lam_q2, lam_k2, layer_index: int, stream=None):
    """DIFF V1 forward that also saves what the backward needs.

    Arguments as v1_fwd.  Returns (out, saved): out (B, T, H, 2d) is the
    forward output, saved an opaque uint8 CUDA tensor for v1_bwd.
    """
    for n, t in (("q1", q1), ("q2", q2), ("k1", k1), ("k2", k2), ("v", v)):
        _cuda(t, n)
    B, T, H, d = q1.shape
    out = torch.empty((B, T, H, 2 * d), dtype=q1.dtype, device=q1.device)
    strides = _v1_strides(q1, q2, k1, k2, v, out)
    lams = _lam_vecs(d, lam_q1, lam_k1, lam_q2, lam_k2)
    nbytes = int(lib().diffattn_v1_train_saved_size(B, T, H, d, _dtype_code(q1)))
    saved = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q1.device)
    rc = lib().diffattn_v1_fwd_train(q1.data_ptr(), q2.data_ptr(), k1.data_ptr(), k2.data_ptr(), v.data_ptr(),
                                     *[x.data_ptr() for x in lams], out.data_ptr(), saved.data_ptr(), saved.numel(),
                                     B, T, H, d, int(layer_index), *strides, _dtype_code(q1), _stream(stream))
    _check("diffattn_v1_fwd_train", rc)
    return out, saved


def saved_lse(saved: torch.Tensor, B: int, T: int, H: int, d: int, dtype: torch.dtype,
              v2: bool = False, Hkv: int = 1) -> torch.Tensor:
    """View of the (2, B, H, T) fp32 row log-sum-exp inside a training
    forward's `saved` (log2 units for bf16, natural for fp32).  V1: H diff
    heads, d the q/k head dim; V2: H = Hq query heads, Hkv kv heads, d = D,
    and the view is (2, B, Hq/2, T)."""
    code = DA_BF16 if dtype == torch.bfloat16 else DA_F32
    if v2:
        off = int(lib().diffattn_v2_train_saved_lse_offset(B, T, H, Hkv, d, code))
        rows = H // 2
    else:
        off = int(lib().diffattn_v1_train_saved_lse_offset(B, T, H, d, code))
        rows = H
    if off == 0:
        raise ValueError("unsupported sizes")
    n = 2 * B * rows * T
    return saved[off:off + 4 * n].view(torch.float32).view(2, B, rows, T)


def v1_bwd(q1, q2, k1, k2, v, lam_q1, lam_k1, lam_q2, lam_k2, layer_index: int, dout, saved,
           workspace: torch.Tensor | None = None, stream=None) -> dict:
    """Gradients of DIFF V1 for upstream gradient dout (the output's shape).

    Returns dq1, dq2 (q's layout: views of one (B, T, 2H, d) tensor when q1,
    q2 are the interleaved views), dk1, dk2 (likewise for k), dv, and the fp32
    lambda-vector gradients dlam_q1, dlam_k1, dlam_q2, dlam_k2.
    """
    B, T, H, d = q1.shape
    if dout.shape != (B, T, H, 2 * d) or dout.dtype != q1.dtype:
        raise ValueError("dout must match the output")
    strides = _v1_strides(q1, q2, k1, k2, v, dout)
    lams = _lam_vecs(d, lam_q1, lam_k1, lam_q2, lam_k2)

    def like(t1, t2):
        # gradients with the inputs' strides: a shared base when the inputs are views of one tensor
        if t1.data_ptr() + t1.element_size() * d == t2.data_ptr() and t1.stride()[2] == 2 * d:
            base = torch.empty((B, T, 2 * H, d), dtype=t1.dtype, device=t1.device)
            return base[:, :, 0::2], base[:, :, 1::2]
        if t1.is_contiguous() and t2.is_contiguous():
            return torch.empty_like(t1), torch.empty_like(t2)
        raise ValueError("q1/q2 (k1/k2) must be contiguous or the (2h, 2h+1) views of one tensor")
    dq1, dq2 = like(q1, q2)
    dk1, dk2 = like(k1, k2)
    if dq1.stride() != q1.stride() or dk1.stride() != k1.stride():
        raise ValueError("unsupported q / k layout")
    dv = torch.empty_like(v)
    if dv.stride() != v.stride():
        raise ValueError("v must be contiguous")
    dl = [torch.empty(d, dtype=torch.float32, device=q1.device) for _ in range(4)]   # fp32 for both dtypes
    need = int(lib().diffattn_v1_bwd_workspace_size(B, T, H, d, _dtype_code(q1)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q1.device)
    rc = lib().diffattn_v1_bwd(q1.data_ptr(), q2.data_ptr(), k1.data_ptr(), k2.data_ptr(), v.data_ptr(),
                               *[x.data_ptr() for x in lams], dout.data_ptr(), saved.data_ptr(), saved.numel(),
                               dq1.data_ptr(), dq2.data_ptr(), dk1.data_ptr(), dk2.data_ptr(), dv.data_ptr(),
                               *[x.data_ptr() for x in dl], workspace.data_ptr(), workspace.numel(),
                               B, T, H, d, int(layer_index), *strides, _dtype_code(q1), _stream(stream))
    _check("diffattn_v1_bwd", rc)
    return {"dq1": dq1, "dq2": dq2, "dk1": dk1, "dk2": dk2, "dv": dv,
            "dlam_q1": dl[0], "dlam_k1": dl[1], "dlam_q2": dl[2], "dlam_k2": dl[3]}


def v2_fwd_train(q, k, v, lam, stream=None):
    """DIFF V2 forward that also saves what the backward needs: (out, saved)."""
    for n, t in (("q", q), ("k", k), ("v", v), ("lam", lam)):
        _cuda(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    out = torch.empty((B, T, Hq // 2, D), dtype=q.dtype, device=q.device)
    nbytes = int(lib().diffattn_v2_train_saved_size(B, T, Hq, Hkv, D, _dtype_code(q)))
    saved = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    rc = lib().diffattn_v2_fwd_train(q.data_ptr(), k.data_ptr(), v.data_ptr(), lam.data_ptr(), out.data_ptr(),
                                     saved.data_ptr(), saved.numel(), B, T, Hq, Hkv, D, _dtype_code(q),
                                     _stream(stream))
    _check("diffattn_v2_fwd_train", rc)
    return out, saved


def v2_bwd(q, k, v, lam, dout, saved, workspace: torch.Tensor | None = None, stream=None) -> dict:
    """Gradients of DIFF V2 for upstream gradient dout (B, T, Hq/2, D):
    dq, dk, dv (bf16, the inputs' shapes) and dlam (fp32, lam's shape)."""
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if dout.shape != (B, T, Hq // 2, D) or not dout.is_contiguous():
        raise ValueError("dout must be a contiguous (B, T, Hq/2, D) tensor")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dlam = torch.empty_like(lam)
    need = int(lib().diffattn_v2_bwd_workspace_size(B, T, Hq, Hkv, D, _dtype_code(q)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = lib().diffattn_v2_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), lam.data_ptr(), dout.data_ptr(),
                               saved.data_ptr(), saved.numel(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                               dlam.data_ptr(), workspace.data_ptr(), workspace.numel(), B, T, Hq, Hkv, D,
                               _dtype_code(q), _stream(stream))
    _check("diffattn_v2_bwd", rc)
    return {"dq": dq, "dk": dk, "dv": dv, "dlam": dlam}


# ------------------------------------------------------------------ prologue

def prologue(q=None, k=None, pos0: int = 0, base: float = 10000.0, x=None, w_lam=None, lam=None, stream=None):
    """Rotary embedding of q (B, T, Hq, D) and k (B, T, Hk, D) in place and, if
    x (B, T, C) and w_lam (C, P) are given, the V2 lambda logits x @ w_lam
    (fp32 (B, T, P), written to lam or a new tensor): one pass over each
    tensor, one kernel for the rotation and one for the logits.
    Returns lam (or None)."""
    ref = q if q is not None else (k if k is not None else x)
    if ref is None:
        raise ValueError("nothing to do")
    for n, t in (("q", q), ("k", k), ("x", x), ("w_lam", w_lam)):
        if t is not None:
            _cuda(t, n)
            if not t.is_contiguous():
                raise ValueError(f"{n} must be contiguous")
    shp = (q if q is not None else k).shape if (q is not None or k is not None) else None
    if shp is not None:
        B, T, _, D = shp
    else:
        B, T, _ = x.shape
        D = 64
    Hq = q.shape[2] if q is not None else 0
    Hk = k.shape[2] if k is not None else 0
    C = P = 0
    if x is not None:
        if w_lam is None:
            raise ValueError("x needs w_lam")
        C, P = w_lam.shape
        if lam is None:
            lam = torch.empty((B, T, P), dtype=torch.float32, device=x.device)
    rc = lib().diffattn_prologue(None if q is None else q.data_ptr(), None if k is None else k.data_ptr(),
                                 B, T, Hq, Hk, D, int(pos0), float(base),
                                 None if x is None else x.data_ptr(), None if w_lam is None else w_lam.data_ptr(),
                                 None if lam is None else lam.data_ptr(), C, P, _dtype_code(ref), _stream(stream))
    _check("diffattn_prologue", rc)
    return lam
