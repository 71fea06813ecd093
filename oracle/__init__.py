"""fp64 CPU oracle for the causal differential-attention forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library never loads it and shares no code with it.

The arithmetic lives in ``diffattn_oracle.c`` (plain loops in double
precision); this module compiles it with gcc, loads it with ctypes and
converts numpy / torch arrays to contiguous float64.

Citations (page titles as printed):
  * "Differential Transformer V2" -- pseudo-code ``DiffAttnV1`` and
    ``DiffAttnV2`` (lam_init schedule, lambda re-parameterisation, rmsnorm,
    (1 - lam_init) scale, paired heads ``attn[:,0::2] - sigmoid(lam)*attn[:,1::2]``,
    GQA groups contiguous, decoding is memory-bound).
  * "How best to implement a differential transformer?" (nanoGPT issue 567) --
    ``RMSNorm(2*head_dim, eps=1e-5, elementwise_affine=False)``, causal mask,
    1/sqrt(head_dim) score scale, head pairing (2h, 2h+1).

Every function here is pinned by ``tests/test_oracle_pins.py`` (closed forms,
library attention routines, invariants, brute force); none is parity-unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "diffattn_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_liboracle.so`` (gcc, -O2, no fast-math)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            lib.oracle_lambda_init.restype = ctypes.c_double
            lib.oracle_lambda_init.argtypes = [ctypes.c_int]
            lib.oracle_lambda_full.restype = ctypes.c_double
            lib.oracle_lambda_full.argtypes = [dp, dp, dp, dp, ctypes.c_int, ctypes.c_double]
            lib.oracle_rmsnorm.restype = None
            lib.oracle_rmsnorm.argtypes = [dp, ctypes.c_int, ctypes.c_double, dp]
            lib.oracle_v1_fwd.restype = ctypes.c_int
            lib.oracle_v1_fwd.argtypes = [dp] * 9 + [ctypes.c_int] * 5 + [i64p, ctypes.c_int64, dp, ctypes.c_int]
            lib.oracle_v2_fwd.restype = ctypes.c_int
            lib.oracle_v2_fwd.argtypes = [dp] * 4 + [ctypes.c_int] * 5 + [i64p, ctypes.c_int64, dp, ctypes.c_int]
            lib.oracle_paired_fwd.restype = ctypes.c_int
            lib.oracle_paired_fwd.argtypes = [dp] * 3 + [ctypes.c_int] * 4 + [i64p, ctypes.c_int64, dp, ctypes.c_int]
            lib.oracle_v2_decode.restype = ctypes.c_int
            lib.oracle_v2_decode.argtypes = ([dp] * 4 + [ctypes.c_int, ctypes.c_int64] + [ctypes.c_int] * 3
                                             + [i64p, i64p, ctypes.c_int64, dp, ctypes.c_int])
            lib.oracle_v1_bwd.restype = ctypes.c_int
            lib.oracle_v1_bwd.argtypes = ([dp] * 10 + [ctypes.c_int] * 5 + [i64p, ctypes.c_int64] + [dp] * 7
                                          + [ctypes.c_int])
            lib.oracle_v2_bwd.restype = ctypes.c_int
            lib.oracle_v2_bwd.argtypes = ([dp] * 5 + [ctypes.c_int] * 5 + [i64p, ctypes.c_int64] + [dp] * 4
                                          + [ctypes.c_int])
            lib.oracle_lse.restype = None
            lib.oracle_lse.argtypes = [dp, dp] + [ctypes.c_int] * 5 + [dp]
            lib.oracle_rope.restype = None
            lib.oracle_rope.argtypes = [dp] + [ctypes.c_int] * 4 + [ctypes.c_int64, ctypes.c_double, dp]
            lib.oracle_lambda_proj.restype = None
            lib.oracle_lambda_proj.argtypes = [dp, dp, ctypes.c_int64, ctypes.c_int, ctypes.c_int, dp]
            lib.oracle_v1_decode.restype = ctypes.c_int
            lib.oracle_v1_decode.argtypes = ([dp] * 9 + [ctypes.c_int, ctypes.c_int64] + [ctypes.c_int] * 3
                                             + [i64p, i64p, ctypes.c_int64, dp, ctypes.c_int])
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f64(x) -> np.ndarray:
    """Any numpy array or CPU torch tensor (fp32/bf16/fp64) -> contiguous float64."""
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _rows(rows):
    if rows is None:
        return None, None, 0
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    return r, r.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), r.size


def lambda_init(layer_index: int) -> float:
    """lam_init = 0.8 - 0.6 exp(-0.3 layer_index) ("Differential Transformer V2", DiffAttnV1)."""
    return _load().oracle_lambda_init(int(layer_index))


def lambda_full(lq1, lk1, lq2, lk2, layer_index: int) -> float:
    """lam = exp(sum(lq1*lk1)) - exp(sum(lq2*lk2)) + lam_init ("Differential Transformer V2")."""
    a = [_f64(x) for x in (lq1, lk1, lq2, lk2)]
    return _load().oracle_lambda_full(*[_ptr(x) for x in a], a[0].size, lambda_init(layer_index))


def rmsnorm(x, eps: float = 1e-5) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) over the last axis, no affine weight (nanoGPT issue 567, subln)."""
    x = _f64(x)
    flat = x.reshape(-1, x.shape[-1])
    out = np.empty_like(flat)
    lib = _load()
    for r in range(flat.shape[0]):
        lib.oracle_rmsnorm(_ptr(flat[r]), flat.shape[1], float(eps), _ptr(out[r]))
    return out.reshape(x.shape)


def v1_fwd(q1, q2, k1, k2, v, lq1, lk1, lq2, lk2, layer_index: int,
           rows=None, nthreads: int | None = None) -> np.ndarray:
    """DIFF V1 causal forward ("Differential Transformer V2", DiffAttnV1).

    q1, q2, k1, k2: (B, T, H, d); v: (B, T, H, 2d); lambda vectors: (d,).
    rows=None returns (B, T, H, 2d); otherwise ``rows`` holds flat ids
    (b*T + t)*H + h and the result is (len(rows), 2d).
    """
    q1, q2, k1, k2, v = (_f64(x) for x in (q1, q2, k1, k2, v))
    lq1, lk1, lq2, lk2 = (_f64(x) for x in (lq1, lk1, lq2, lk2))
    B, T, H, d = q1.shape
    assert v.shape == (B, T, H, 2 * d), v.shape
    for x in (q2, k1, k2):
        assert x.shape == (B, T, H, d)
    r, rp, n = _rows(rows)
    out = np.empty(((n if r is not None else B * T * H), 2 * d), dtype=np.float64)
    rc = _load().oracle_v1_fwd(_ptr(q1), _ptr(q2), _ptr(k1), _ptr(k2), _ptr(v),
                               _ptr(lq1), _ptr(lk1), _ptr(lq2), _ptr(lk2),
                               B, T, H, d, int(layer_index), rp, n, _ptr(out),
                               nthreads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_v1_fwd failed ({rc})")
    return out if r is not None else out.reshape(B, T, H, 2 * d)


def v2_fwd(q, k, v, lam, rows=None, nthreads: int | None = None) -> np.ndarray:
    """DIFF V2 causal prefill ("Differential Transformer V2", DiffAttnV2).

    q: (B, T, Hq, D); k, v: (B, T, Hkv, D); lam: (B, T, Hq/2) logits.
    rows=None returns (B, T, Hq/2, D); otherwise flat ids (b*T + t)*(Hq/2) + i.
    """
    q, k, v, lam = (_f64(x) for x in (q, k, v, lam))
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    assert Hq % 2 == 0 and Hq % Hkv == 0 and (Hq // Hkv) % 2 == 0
    assert k.shape == (B, T, Hkv, D) and v.shape == (B, T, Hkv, D)
    assert lam.shape == (B, T, Hq // 2)
    r, rp, n = _rows(rows)
    out = np.empty(((n if r is not None else B * T * (Hq // 2)), D), dtype=np.float64)
    rc = _load().oracle_v2_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(lam), B, T, Hq, Hkv, D,
                               rp, n, _ptr(out), nthreads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_v2_fwd failed ({rc})")
    return out if r is not None else out.reshape(B, T, Hq // 2, D)


def paired_fwd(q, k, v, rows=None, nthreads: int | None = None) -> np.ndarray:
    """Paired Head Attention (modded-nanogpt pull request "New Record: Paired
    Head Attention (-3.5s, -65 steps)", section "Updates in PR"): heads 2i and 2i+1
    are interleaved into one causal sequence of length 2T (position 2t + e is
    token t of head 2i + e) and attended with one softmax; outputs return to
    (token, head).

    q, k, v: (B, T, H, D), H even.  rows=None returns (B, T, H, D); otherwise
    flat ids (b*T + t)*H + h.
    """
    q, k, v = (_f64(x) for x in (q, k, v))
    B, T, H, D = q.shape
    assert H % 2 == 0 and k.shape == q.shape and v.shape == q.shape
    r, rp, n = _rows(rows)
    out = np.empty(((n if r is not None else B * T * H), D), dtype=np.float64)
    rc = _load().oracle_paired_fwd(_ptr(q), _ptr(k), _ptr(v), B, T, H, D, rp, n, _ptr(out),
                                   nthreads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_paired_fwd failed ({rc})")
    return out if r is not None else out.reshape(B, T, H, D)


def _lens(lens, B, L):
    if lens is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(lens.cpu() if hasattr(lens, "cpu") else lens, dtype=np.int64).reshape(-1))
    assert a.shape == (B,) and (a >= 1).all() and (a <= L).all(), "lens must hold B values in 1..L"
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def v2_decode(q, k_cache, v_cache, lam, rows=None, nthreads: int | None = None, lens=None) -> np.ndarray:
    """DIFF V2 single-token decode against an L-row KV cache.

    q: (B, Hq, D); caches: (B, L, Hkv, D); lam: (B, Hq/2); lens: optional
    (B,) rows attended per sequence (default all L).
    rows=None returns (B, Hq/2, D); otherwise flat ids b*(Hq/2) + i.
    """
    q, k, v, lam = (_f64(x) for x in (q, k_cache, v_cache, lam))
    B, Hq, D = q.shape
    L, Hkv = k.shape[1], k.shape[2]
    assert Hq % Hkv == 0 and (Hq // Hkv) % 2 == 0
    assert k.shape == (B, L, Hkv, D) and v.shape == (B, L, Hkv, D)
    assert lam.shape == (B, Hq // 2)
    la, lp = _lens(lens, B, L)
    r, rp, n = _rows(rows)
    out = np.empty(((n if r is not None else B * (Hq // 2)), D), dtype=np.float64)
    rc = _load().oracle_v2_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(lam), B, L, Hq, Hkv, D,
                                  lp, rp, n, _ptr(out), nthreads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_v2_decode failed ({rc})")
    return out if r is not None else out.reshape(B, Hq // 2, D)


def v1_decode(q1, q2, k1_cache, k2_cache, v_cache, lq1, lk1, lq2, lk2, layer_index: int,
              rows=None, nthreads: int | None = None, lens=None) -> np.ndarray:
    """DIFF V1 single-token decode (the DiffAttnV1 operation for one new token
    against L cached rows; "Differential Transformer V2", DiffAttnV1).

    q1, q2: (B, H, d); k1, k2: (B, L, H, d); v: (B, L, H, 2d); lambda vectors (d,);
    lens: optional (B,) rows attended per sequence.  rows=None returns (B, H, 2d),
    otherwise flat ids b*H + h.
    """
    q1, q2, k1, k2, v = (_f64(x) for x in (q1, q2, k1_cache, k2_cache, v_cache))
    lq1, lk1, lq2, lk2 = (_f64(x) for x in (lq1, lk1, lq2, lk2))
    B, H, d = q1.shape
    L = k1.shape[1]
    assert q2.shape == (B, H, d) and k1.shape == (B, L, H, d) and k2.shape == (B, L, H, d)
    assert v.shape == (B, L, H, 2 * d)
    la, lp = _lens(lens, B, L)
    r, rp, n = _rows(rows)
    out = np.empty(((n if r is not None else B * H), 2 * d), dtype=np.float64)
    rc = _load().oracle_v1_decode(_ptr(q1), _ptr(q2), _ptr(k1), _ptr(k2), _ptr(v), _ptr(lq1), _ptr(lk1),
                                  _ptr(lq2), _ptr(lk2), B, L, H, d, int(layer_index), lp, rp, n, _ptr(out),
                                  nthreads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_v1_decode failed ({rc})")
    return out if r is not None else out.reshape(B, H, 2 * d)


def v1_bwd(q1, q2, k1, k2, v, lq1, lk1, lq2, lk2, layer_index: int, dout, heads=None,
           nthreads: int | None = None) -> dict:
    """Gradients of the DIFF V1 forward for upstream gradient dout (B, T, H, 2d).

    Returns dq1, dq2, dk1, dk2 (B, T, H, d), dv (B, T, H, 2d), dlam_q1,
    dlam_k1, dlam_q2, dlam_k2 (d,) and dlam_abs, the sum of |dx_c a2_c| over
    the terms of dL/dlam = -sum dx_c a2_c (a scale for rounding errors).  heads: optional ids b*H + h; then only
    those heads' gradients are filled (the rest stay 0) and the lambda-vector
    gradients hold only those heads' share.
    """
    q1, q2, k1, k2, v, dout = (_f64(x) for x in (q1, q2, k1, k2, v, dout))
    lq1, lk1, lq2, lk2 = (_f64(x) for x in (lq1, lk1, lq2, lk2))
    B, T, H, d = q1.shape
    assert q2.shape == k1.shape == k2.shape == (B, T, H, d)
    assert v.shape == dout.shape == (B, T, H, 2 * d)
    hs = None if heads is None else np.ascontiguousarray(np.asarray(heads, dtype=np.int64).reshape(-1))
    hp = None if hs is None else hs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    g = {n: np.zeros(sh, dtype=np.float64) for n, sh in
         (("dq1", q1.shape), ("dq2", q1.shape), ("dk1", q1.shape), ("dk2", q1.shape), ("dv", v.shape))}
    dl = np.zeros(4 * d, dtype=np.float64)
    da = np.zeros(1, dtype=np.float64)
    rc = _load().oracle_v1_bwd(_ptr(q1), _ptr(q2), _ptr(k1), _ptr(k2), _ptr(v), _ptr(lq1), _ptr(lk1), _ptr(lq2),
                               _ptr(lk2), _ptr(dout), B, T, H, d, int(layer_index), hp,
                               0 if hs is None else hs.size, _ptr(g["dq1"]), _ptr(g["dq2"]), _ptr(g["dk1"]),
                               _ptr(g["dk2"]), _ptr(g["dv"]), _ptr(dl), _ptr(da), nthreads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_v1_bwd failed ({rc})")
    g.update(dlam_q1=dl[:d], dlam_k1=dl[d:2 * d], dlam_q2=dl[2 * d:3 * d], dlam_k2=dl[3 * d:])
    g["dlam_abs"] = float(da[0])   # sum |dx_c a2_c|: the scale of the terms cancelling in dL/dlam
    return g


def v2_bwd(q, k, v, lam, dout, groups=None, nthreads: int | None = None) -> dict:
    """Gradients of the DIFF V2 prefill for upstream gradient dout (B, T, Hq/2, D).

    Returns dq (B, T, Hq, D), dk, dv (B, T, Hkv, D), dlam (B, T, Hq/2).
    groups: optional kv-group ids b*Hkv + g; then only those groups' heads,
    kv rows and pairs are filled.
    """
    q, k, v, lam, dout = (_f64(x) for x in (q, k, v, lam, dout))
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    assert k.shape == v.shape == (B, T, Hkv, D) and lam.shape == (B, T, Hq // 2)
    assert dout.shape == (B, T, Hq // 2, D)
    gs = None if groups is None else np.ascontiguousarray(np.asarray(groups, dtype=np.int64).reshape(-1))
    gp = None if gs is None else gs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    g = {"dq": np.zeros(q.shape), "dk": np.zeros(k.shape), "dv": np.zeros(v.shape), "dlam": np.zeros(lam.shape)}
    rc = _load().oracle_v2_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(lam), _ptr(dout), B, T, Hq, Hkv, D, gp,
                               0 if gs is None else gs.size, _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]),
                               _ptr(g["dlam"]), nthreads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_v2_bwd failed ({rc})")
    return g


def lse(q, k) -> np.ndarray:
    """Row log-sum-exp (natural log) of the causal scaled scores: for q
    (B, T, Hq, d) and k (B, T, Hk, d), out[b, h, t] = log sum_{j <= t}
    exp(q[b,t,h] . k[b,j,h/(Hq/Hk)] / sqrt(d)) -- the normaliser of each
    row's softmax in "Differential Transformer V2" (DiffAttnV1 / DiffAttnV2,
    each flash_attn_func call) and "How best to implement a differential
    transformer?" (the masked, 1/sqrt(d)-scaled scores).  Returns (B, Hq, T)."""
    q, k = _f64(q), _f64(k)
    B, T, Hq, d = q.shape
    Hk = k.shape[2]
    assert k.shape == (B, T, Hk, d) and Hq % Hk == 0
    out = np.empty((B, Hq, T), dtype=np.float64)
    _load().oracle_lse(_ptr(q), _ptr(k), B, T, Hq, Hk, d, _ptr(out))
    return out


def rope(x, pos0: int = 0, base: float = 10000.0) -> np.ndarray:
    """Rotary position embedding (rotate-half form) of x (B, T, H, D) at
    positions pos0 + t; returns fp64 (B, T, H, D)."""
    x = _f64(x)
    B, T, H, D = x.shape
    assert D % 2 == 0
    out = np.empty_like(x)
    _load().oracle_rope(_ptr(x), B, T, H, D, int(pos0), float(base), _ptr(out))
    return out


def lambda_proj(x, w) -> np.ndarray:
    """Projected lambda logits x @ w: x (..., C), w (C, P) -> (..., P) fp64."""
    x, w = _f64(x), _f64(w)
    C, P = w.shape
    lead = x.shape[:-1]
    assert x.shape[-1] == C
    xf = np.ascontiguousarray(x.reshape(-1, C))
    out = np.empty((xf.shape[0], P), dtype=np.float64)
    _load().oracle_lambda_proj(_ptr(xf), _ptr(w), xf.shape[0], C, P, _ptr(out))
    return out.reshape(*lead, P)


def decode_gather(q, k_cache, v_cache, lam, rows):
    """Copy only the cache slices that the listed decode rows read.

    The decode oracle for row (b, i) touches k/v[b, :, g] with g = 2i/G.  For
    very large caches this returns small contiguous inputs (one batch entry,
    one kv head per listed row) and the row ids that address them, so that
    sampled rows can be checked without converting the whole cache to fp64.
    """
    B, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    P = Hq // 2
    out = []
    for rid in np.asarray(rows, dtype=np.int64).reshape(-1):
        b, i = int(rid) // P, int(rid) % P
        g = (2 * i) // G
        qs = q[b:b + 1, g * G:(g + 1) * G]               # (1, G, D)
        ks = k_cache[b:b + 1, :, g:g + 1]                 # (1, L, 1, D)
        vs = v_cache[b:b + 1, :, g:g + 1]
        ls = lam[b:b + 1, g * G // 2:(g + 1) * G // 2]    # (1, G/2)
        local = i - g * G // 2
        out.append((qs, ks, vs, ls, local))
    return out
