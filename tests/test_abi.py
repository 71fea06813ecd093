"""Host-only checks of the C ABI: the library loads, exports every symbol that
include/diffattn.h declares, and rejects bad arguments before touching CUDA.
No compute call is made here (no GPU in this environment)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "diffattn.h")


@pytest.fixture(scope="module")
def lib():
    from differential_attention_causal_gb300 import build as b
    b.build()
    from differential_attention_causal_gb300 import binding
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(diffattn_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("diffattn_v1_fwd", "diffattn_v2_fwd", "diffattn_v2_decode",
              "diffattn_v2_decode_workspace_size", "diffattn_status_string", "diffattn_device_error",
              "diffattn_v2_decode_varlen", "diffattn_v1_decode", "diffattn_v1_decode_workspace_size",
              "diffattn_paired_fwd", "diffattn_v1_fwd_host", "diffattn_v1_fwd_host_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from differential_attention_causal_gb300 import binding
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (diffattn_\w+)", out))
    for n in declared_functions():
        assert n in exported, n
        assert getattr(lib, n) is not None


def test_status_strings(lib):
    from differential_attention_causal_gb300 import binding
    for code in range(13):
        s = binding.status_string(code)
        assert isinstance(s, str) and s
    assert binding.status_string(0) == "ok"
    assert binding.status_string(1234) == "unknown status"


A = 0x10000  # a 16-byte aligned fake address: validation never dereferences it


def _v1(lib, **kw):
    args = dict(q1=A, q2=A, k1=A, k2=A, v=A, lq1=A, lk1=A, lq2=A, lk2=A, out=A, B=1, T=8, H=2, d=64,
                layer=0, qs=(1024, 128, 64), ks=(1024, 128, 64), vs=(2048, 256, 128), os_=(2048, 256, 128),
                dtype=1)
    args.update(kw)
    a = args
    return lib.diffattn_v1_fwd(a["q1"], a["q2"], a["k1"], a["k2"], a["v"], a["lq1"], a["lk1"], a["lq2"],
                               a["lk2"], a["out"], a["B"], a["T"], a["H"], a["d"], a["layer"], *a["qs"],
                               *a["ks"], *a["vs"], *a["os_"], a["dtype"], None)


def test_v1_argument_checks(lib):
    assert _v1(lib, q2=None) == 1                       # NULL
    assert _v1(lib, lk2=None) == 1
    assert _v1(lib, T=0) == 2                           # bad shape
    assert _v1(lib, layer=-1) == 2
    assert _v1(lib, d=48) == 3                          # bf16 d=48 unsupported
    assert _v1(lib, d=32, v=A + 8) == 5                 # bf16 d=32 passes the dimension check
    assert _v1(lib, d=96) == 3
    assert _v1(lib, d=96, dtype=0) == 3                 # fp32 d=96 unsupported
    assert _v1(lib, v=A + 8) == 5                       # misaligned pointer
    assert _v1(lib, qs=(1024, 127, 64)) == 5            # stride not a multiple of 16 bytes
    assert _v1(lib, os_=(2048, 0, 128)) == 5
    assert _v1(lib, dtype=7) == 8                       # bad dtype


def _v2(lib, **kw):
    a = dict(q=A, k=A, v=A, lam=A, out=A, B=1, T=8, Hq=8, Hkv=2, D=128, dtype=1)
    a.update(kw)
    return lib.diffattn_v2_fwd(a["q"], a["k"], a["v"], a["lam"], a["out"], a["B"], a["T"], a["Hq"], a["Hkv"],
                               a["D"], a["dtype"], None)


def test_v2_argument_checks(lib):
    assert _v2(lib, lam=None) == 1
    assert _v2(lib, B=0) == 2
    assert _v2(lib, Hq=8, Hkv=3) == 4                  # not a multiple
    assert _v2(lib, Hq=6, Hkv=2) == 4                  # odd group size
    assert _v2(lib, D=96) == 3
    assert _v2(lib, out=A + 2) == 5
    assert _v2(lib, dtype=2) == 8


def _paired(lib, **kw):
    a = dict(q=A, k=A, v=A, out=A, B=1, T=8, H=4, D=128, dtype=1)
    a.update(kw)
    return lib.diffattn_paired_fwd(a["q"], a["k"], a["v"], a["out"], a["B"], a["T"], a["H"], a["D"], a["dtype"], None)


def test_paired_argument_checks(lib):
    assert _paired(lib, v=None) == 1
    assert _paired(lib, T=0) == 2
    assert _paired(lib, H=3) == 2                      # heads come in pairs
    assert _paired(lib, D=96) == 3
    assert _paired(lib, dtype=0) == 3                  # fp32: no paired kernel
    assert _paired(lib, out=A + 8) == 5
    assert _paired(lib, dtype=5) == 8


def _host(lib, **kw):
    a = dict(q=A, k=A, v=A, l1=A, l2=A, l3=A, l4=A, out=A, B=2, T=8, H=2, d=64, layer=0, ws=A, wsb=1 << 30,
             dtype=1)
    a.update(kw)
    return lib.diffattn_v1_fwd_host(a["q"], a["k"], a["v"], a["l1"], a["l2"], a["l3"], a["l4"], a["out"], a["B"],
                                    a["T"], a["H"], a["d"], a["layer"], a["ws"], a["wsb"], a["dtype"], None)


def test_v1_host_argument_checks(lib):
    from differential_attention_causal_gb300 import binding
    need = binding.v1_fwd_host_workspace_size(2, 8, 2, 64)
    assert need >= 2 * 8 * 4 * 64 * 2 * 2 + 2 * 8 * 2 * 128 * 2 * 2   # q, k, v, out at least
    assert _host(lib, out=None) == 1
    assert _host(lib, ws=None) == 1
    assert _host(lib, T=0) == 2
    assert _host(lib, layer=-1) == 2
    assert _host(lib, d=48) == 3                       # bf16 d = 48 unsupported
    assert _host(lib, wsb=need - 1) == 6               # workspace too small
    assert _host(lib, ws=A + 16) == 5                  # workspace not 256-byte aligned
    assert _host(lib, dtype=3) == 8
    assert binding.v1_fwd_host_workspace_size(0, 8, 2, 64) == 0


def _dec(lib, **kw):
    a = dict(q=A, k=A, v=A, lam=A, out=A, ws=A, wsb=1 << 20, B=2, L=100, Hq=16, Hkv=2, D=128, dtype=1)
    a.update(kw)
    return lib.diffattn_v2_decode(a["q"], a["k"], a["v"], a["lam"], a["out"], a["ws"], a["wsb"], a["B"], a["L"],
                                  a["Hq"], a["Hkv"], a["D"], a["dtype"], None)


def test_decode_argument_checks(lib):
    assert _dec(lib, k=None) == 1
    assert _dec(lib, L=0) == 2
    assert _dec(lib, Hq=12, Hkv=4) == 4                # odd group size
    assert _dec(lib, D=32) == 3
    assert _dec(lib, v=A + 4) == 5


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from differential_attention_causal_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not found"):
        binding.lib()


def test_oracle_is_not_imported_by_the_product():
    """The CUDA path and the oracle share no code: no product module imports oracle."""
    pkg = os.path.join(ROOT, "differential_attention_causal_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
                assert "diffattn_oracle" not in text, f


def _v1dec(lib, **kw):
    a = dict(q1=A, q2=A, k1=A, k2=A, v=A, lq1=A, lk1=A, lq2=A, lk2=A, lens=None, out=A, ws=A, wsb=1 << 20,
             B=2, L=100, H=2, d=64, layer=0, dtype=1)
    a.update(kw)
    return lib.diffattn_v1_decode(a["q1"], a["q2"], a["k1"], a["k2"], a["v"], a["lq1"], a["lk1"], a["lq2"],
                                  a["lk2"], a["lens"], a["out"], a["ws"], a["wsb"], a["B"], a["L"], a["H"],
                                  a["d"], a["layer"], a["dtype"], None)


def test_v1_decode_argument_checks(lib):
    assert _v1dec(lib, k2=None) == 1
    assert _v1dec(lib, lk1=None) == 1
    assert _v1dec(lib, L=0) == 2
    assert _v1dec(lib, layer=-3) == 2
    assert _v1dec(lib, d=48) == 3          # bf16 decode needs d in {32, 64, 128}
    assert _v1dec(lib, d=96, dtype=0) == 3
    assert _v1dec(lib, q2=A + 8) == 5
    assert _v1dec(lib, lens=A + 2) == 5    # int32 lengths need 4-byte alignment
    assert _v1dec(lib, dtype=5) == 8


def test_v2_decode_varlen_argument_checks(lib):
    def call(**kw):
        a = dict(q=A, k=A, v=A, lam=A, lens=A, out=A, ws=A, wsb=1 << 20, B=2, L=100, Hq=8, Hkv=2, D=128, dtype=1)
        a.update(kw)
        return lib.diffattn_v2_decode_varlen(a["q"], a["k"], a["v"], a["lam"], a["lens"], a["out"], a["ws"],
                                             a["wsb"], a["B"], a["L"], a["Hq"], a["Hkv"], a["D"], a["dtype"], None)
    assert call(lens=None) == 1
    assert call(lens=A + 1) == 5
    assert call(B=0) == 2
    assert call(Hq=6, Hkv=2) == 4          # odd group
    assert call(D=96) == 3
    assert call(k=A + 4) == 5
    assert call(dtype=9) == 8


def test_debug_library_builds_and_exports_the_same_symbols(lib):
    """The debug build (-DDA_DEBUG_CHECKS: bounds checks in every kernel that
    writes through a computed index) links, exports every declared symbol and
    says which build it is; the release build says it has no checks.  Both
    answers are plain host calls, no GPU needed."""
    from differential_attention_causal_gb300 import build as b
    path = b.build(debug=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (diffattn_\w+)", out))
    for n in declared_functions():
        assert n in exported, n
    dbg = ctypes.CDLL(path)
    assert dbg.diffattn_debug_checks() == 1
    assert lib.diffattn_debug_checks() == 0
    dbg.diffattn_status_string.restype = ctypes.c_char_p
    assert b"bounds" in dbg.diffattn_status_string(12)
