"""The C-ABI library on the host, without a GPU: it builds for sm_103a, loads, exports every
symbol include/attnres.h declares, and rejects bad arguments before launching anything.

Every call here either has T = 0 (nothing to launch; pointers may then be NULL) or fails
validation, which happens before any launch: no CUDA call is made and the fake pointers are
never dereferenced.  ``err()`` asserts that a call with T > 0 returned an error."""
import os
import re

import pytest

import depth_wise_softmax_block_b300 as ar
from depth_wise_softmax_block_b300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "attnres.h")
OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3
P = 0x7F0000000000          # a 16-byte aligned fake address (never dereferenced)
PM = P + 8                  # misaligned


def err(status):
    """A call with T > 0 must have failed validation (it would otherwise launch)."""
    assert status != OK
    return status


@pytest.fixture(scope="module")
def lib():
    B.build()
    return ar.library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(attnres_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(lib):
    names = declared_symbols()
    assert "attnres_phase1" in names and "attnres_phase2_merge" in names
    assert "attnres_full_reference_path" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in attnres.h but not exported"
    assert set(names) == set(ar.SIGNATURES), "binding signatures must cover the header"


def test_version_and_strings(lib):
    assert lib.attnres_abi_version() == 9
    for code, name in ar.STATUS.items():
        assert lib.attnres_status_string(code).decode() == name
    assert lib.attnres_status_string(99).decode() == "ATTNRES_ERR_UNKNOWN"


def p1(lib, reps=P, stride=1024 * 64, n=2, T=0, d=64, io=1, u=P, S=4, eps=1e-6, o=P, us=None,
       flags=0, heads=1):
    return lib.attnres_phase1(reps, stride, n, T, d, io, u, us, S, eps, o, None, None, None, flags,
                              heads, None)


def test_phase1_validation(lib):
    assert p1(lib) == OK                                  # T = 0: nothing to do
    assert p1(lib, reps=None, u=None, o=None) == OK       # ... and pointers may be NULL
    assert err(p1(lib, T=4, reps=None)) == INVALID
    assert err(p1(lib, T=4, u=None)) == INVALID
    assert err(p1(lib, T=4, o=None)) == INVALID
    assert p1(lib, io=7) == INVALID
    assert p1(lib, d=60) == INVALID                       # d % 8
    assert p1(lib, d=0) == INVALID
    assert p1(lib, T=-1) == INVALID
    assert p1(lib, n=0) == INVALID
    assert p1(lib, S=0) == INVALID
    assert p1(lib, eps=-1.0) == INVALID
    assert p1(lib, eps=float("nan")) == INVALID
    assert p1(lib, n=65) == UNSUPPORTED
    assert p1(lib, S=65) == UNSUPPORTED
    assert p1(lib, n=17, S=64) == UNSUPPORTED              # one CTA cannot hold the tile
    assert p1(lib, n=16, S=64) == OK
    assert p1(lib, n=64, S=1) == OK
    assert p1(lib, n=64, S=24) == OK
    assert p1(lib, d=16384 + 8) == UNSUPPORTED
    assert err(p1(lib, T=10, stride=8)) == INVALID         # sources would overlap
    assert err(p1(lib, T=4, reps=PM)) == MISALIGNED
    assert err(p1(lib, T=4, u=PM)) == MISALIGNED
    assert err(p1(lib, T=4, o=PM)) == MISALIGNED
    assert err(p1(lib, T=4, stride=1024 * 64 + 4)) == MISALIGNED  # source 1 misaligned
    assert err(p1(lib, T=4, us=PM)) == MISALIGNED         # split queries misaligned
    assert p1(lib, us=P) == OK
    assert p1(lib, flags=3) == OK                         # both variant flags
    assert p1(lib, flags=4) == OK                         # o stored in fp32
    assert p1(lib, flags=7) == OK
    assert p1(lib, flags=8) == INVALID                    # unknown flag
    assert p1(lib, d=128, heads=16) == OK                 # depth-attention heads of 8 columns
    assert p1(lib, d=128, heads=0) == INVALID
    assert p1(lib, d=128, heads=3) == INVALID             # d % heads
    assert p1(lib, d=96, heads=3) == OK
    assert p1(lib, d=120, heads=5) == OK                  # heads of 24 columns
    assert p1(lib, d=120, heads=10) == INVALID            # heads of 12 columns (not 8k)
    assert p1(lib, d=64, heads=16) == INVALID             # heads of 4 columns (not 8)
    assert p1(lib, d=1024, heads=65) == UNSUPPORTED


def p2(lib, o=P, lse=P, part=None, v=None, pout=None, T=0, d=64, io=1, u=P, g=None, y=P, h=None,
       flags=0, heads=1):
    return lib.attnres_phase2_merge(o, lse, part, v, pout, T, d, io, u, 1e-6, g, 1e-6, h, y, None,
                                    flags, heads, None)


def test_phase2_validation(lib):
    assert p2(lib) == OK
    assert p2(lib, o=None, y=None, u=None, lse=None) == OK
    assert p2(lib, part=P, v=P, pout=P) == OK
    assert err(p2(lib, T=4, o=None)) == INVALID
    assert err(p2(lib, T=4, y=None)) == INVALID
    assert err(p2(lib, T=4, part=P, lse=None)) == INVALID  # a partial source needs lse ...
    assert p2(lib, part=P, lse=None, flags=1) == OK       # ... except with sigmoid weights
    assert p2(lib, flags=8) == INVALID
    assert p2(lib, flags=4) == OK                         # o_l stored in fp32
    assert err(p2(lib, T=4, v=P, u=None)) == INVALID       # ... and the query
    assert err(p2(lib, T=4, pout=P)) == INVALID            # nothing to write without a partial
    assert p2(lib, d=12) == INVALID
    assert p2(lib, io=2) == INVALID
    assert err(p2(lib, T=4, o=PM)) == MISALIGNED
    assert err(p2(lib, T=4, part=PM)) == MISALIGNED
    assert err(p2(lib, T=4, v=P, g=PM)) == MISALIGNED
    assert err(p2(lib, T=4, h=PM)) == MISALIGNED
    assert p2(lib, heads=8) == OK
    assert p2(lib, heads=16) == INVALID                   # heads of 4 columns
    assert p2(lib, heads=-1) == INVALID


def test_full_and_update_validation(lib):
    import ctypes
    arr = (ctypes.c_void_p * 3)(P, P + 4096, P + 8192)
    def f(*args, heads=1):
        return lib.attnres_full_reference_path(*args[:-1], 0, heads, args[-1])
    assert f(arr, 3, 0, 64, 1, P, 1e-6, None, 1e-6, None, P, None, None) == OK
    assert err(f(None, 3, 4, 64, 1, P, 1e-6, None, 1e-6, None, P, None, None)) == INVALID
    assert f(arr, 0, 0, 64, 1, P, 1e-6, None, 1e-6, None, P, None, None) == INVALID
    assert f(arr, 65, 0, 64, 1, P, 1e-6, None, 1e-6, None, P, None, None) == UNSUPPORTED
    assert err(f(arr, 3, 4, 64, 1, P, 1e-6, None, 1e-6, None, None, None, None)) == INVALID
    bad = (ctypes.c_void_p * 2)(P, PM)
    assert err(f(bad, 2, 4, 64, 1, P, 1e-6, None, 1e-6, None, P, None, None)) == MISALIGNED
    nul = (ctypes.c_void_p * 2)(P, None)
    assert err(f(nul, 2, 4, 64, 1, P, 1e-6, None, 1e-6, None, P, None, None)) == INVALID
    assert lib.attnres_full_reference_path(arr, 3, 0, 64, 1, P, 1e-6, None, 1e-6, None, P, None,
                                           16, 1, None) == INVALID
    assert lib.attnres_full_reference_path(arr, 3, 0, 64, 1, P, 1e-6, None, 1e-6, None, P, None,
                                           4, 1, None) == INVALID  # no phase-1 output here
    assert f(arr, 3, 0, 64, 1, P, 1e-6, None, 1e-6, None, P, None, None, heads=8) == OK
    assert f(arr, 3, 0, 64, 1, P, 1e-6, None, 1e-6, None, P, None, None, heads=7) == INVALID
    up = lib.attnres_partial_update
    assert up(P, P, P, 0, 64, 1, None) == OK
    assert err(up(None, P, P, 4, 64, 1, None)) == INVALID
    assert err(up(P, P, PM, 4, 64, 1, None)) == MISALIGNED
    assert up(P, P, P, 0, 63, 1, None) == INVALID
    qp = lib.attnres_query_prep
    assert qp(P, None, P, None, 0, 64, None) == OK
    assert qp(P, None, P, P, 0, 64, None) == OK
    assert err(qp(None, None, P, None, 4, 64, None)) == INVALID
    assert err(qp(P, PM, P, None, 4, 64, None)) == MISALIGNED
    assert err(qp(P, None, P, PM, 4, 64, None)) == MISALIGNED


def test_merge_sources_validation(lib):
    import ctypes
    arr = (ctypes.c_void_p * 2)(P, P + 4096)
    ms = lib.attnres_phase2_merge_sources

    def call(o=P, lse=P, srcs=arr, k=2, T=0, d=64, u=P, h=None, y=P, flags=0, heads=1):
        return ms(o, lse, srcs, k, T, d, 1, u, 1e-6, None, 1e-6, h, y, None, flags, heads, None)
    assert call() == OK
    assert call(k=0, srcs=None) == OK
    assert call(k=-1) == INVALID
    assert call(k=65) == UNSUPPORTED
    assert err(call(T=4, o=None)) == INVALID
    assert err(call(T=4, lse=None)) == INVALID           # the history's lse is needed ...
    assert call(lse=None, flags=1) == OK                  # ... except with sigmoid weights
    assert err(call(T=4, y=None)) == INVALID              # nothing to write
    assert err(call(T=4, srcs=None)) == INVALID
    assert err(call(T=4, o=PM)) == MISALIGNED
    bad = (ctypes.c_void_p * 2)(P, PM)
    assert err(call(T=4, srcs=bad)) == MISALIGNED
    assert call(flags=4) == OK                            # o_l stored in fp32
    assert call(flags=8) == INVALID
    assert call(heads=2) == OK
    assert call(heads=128) == UNSUPPORTED


def test_backward_validation(lib):
    import ctypes
    src = (ctypes.c_void_p * 2)(P, P + 4096)
    dst = (ctypes.c_void_p * 2)(P + 8192, P + 12288)
    bw = lib.attnres_backward

    def call(srcs=src, n=2, T=0, d=64, io=1, u=P, gy=P, dsrcs=dst, du=P, dgi=None):
        return bw(srcs, n, T, d, io, u, 1e-6, None, 1e-6, gy, dsrcs, du, dgi, None)
    assert call() == OK
    assert call(n=0) == INVALID
    assert call(n=17) == UNSUPPORTED
    assert call(d=8192 + 8) == UNSUPPORTED                 # bf16 rows beyond 1024 vectors
    assert call(d=4096 + 8, io=0) == UNSUPPORTED           # fp32 rows beyond 1024 vectors
    assert err(call(T=4, du=None)) == INVALID
    assert err(call(T=4, gy=None)) == INVALID
    assert err(call(T=4, dsrcs=None)) == INVALID
    assert err(call(T=4, du=PM)) == MISALIGNED
    bad = (ctypes.c_void_p * 2)(P, PM)
    assert err(call(T=4, dsrcs=bad)) == MISALIGNED


def test_backward_block_validation(lib):
    import ctypes
    ws = lib.attnres_backward_block_workspace_size
    out = ctypes.c_uint64(0)
    assert ws(9, 24, 16, 7168, 1, ctypes.byref(out)) == OK
    n, S, T, d = 9, 24, 16, 7168
    R = (S * n + 3 * S + 3) // 4 * 4
    a256 = lambda x: (x + 255) // 256 * 256              # noqa: E731
    want = (a256(S * T * d * 4) + a256(S * T * 4) + a256(S * T * n * 4) + a256(S * T * d * 4)
            + a256(S * T * 16) + a256(T * R * 4))
    assert out.value == want                              # o, lse, alpha, q, scalars, records
    assert ws(17, 24, 16, 64, 1, ctypes.byref(out)) == UNSUPPORTED
    assert ws(9, 25, 16, 64, 1, ctypes.byref(out)) == UNSUPPORTED
    assert ws(9, 24, 16, 8192 + 8, 1, ctypes.byref(out)) == UNSUPPORTED
    assert ws(9, 24, 16, 4096 + 8, 0, ctypes.byref(out)) == UNSUPPORTED
    assert ws(0, 24, 16, 64, 1, ctypes.byref(out)) == INVALID
    assert ws(9, 24, 16, 64, 1, None) == INVALID
    bb = lib.attnres_backward_block

    def call(reps=P, n=2, v=P, S=3, T=0, d=64, u=P, gy=P, dr=P, dv=P, du=P, ws=P + 8192,
             wsb=1 << 40, vst=1 << 20, sst=1 << 20):
        return bb(reps, sst, n, v, vst, S, T, d, 1, u, None, 1e-6, None, 1e-6, gy, dr, dv, vst,
                  du, None, ws, wsb, None)
    assert call() == OK                                   # T = 0: nothing to do
    assert call(n=17) == UNSUPPORTED
    assert err(call(T=4, v=None)) == INVALID              # S > 1 needs v and d_v
    assert err(call(T=4, du=None)) == INVALID
    assert err(call(T=4, ws=None)) == INVALID
    assert err(call(T=4, wsb=16)) == INVALID              # workspace too small
    assert err(call(T=4, ws=P + 16)) == MISALIGNED        # workspace not 256-byte aligned
    assert err(call(T=4, reps=PM)) == MISALIGNED
    assert call(S=1, v=None, dv=None) == OK


def test_selftest_validation(lib):
    assert lib.attnres_selftest_wait_timeout((1 << 20) + 1, None) == INVALID


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(ar, "_lib", None)
    monkeypatch.setattr(ar, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        ar.library()
