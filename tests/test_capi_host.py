"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every entry point the header declares, and rejects bad
arguments before touching the device (every call here returns before any
CUDA call is made, so fake aligned pointers are never dereferenced)."""
import ctypes
import os
import re

import pytest

from bwd_sparse_mla_gb300 import build as B
from bwd_sparse_mla_gb300 import capi

HEADER = os.path.join(B.ROOT, "include", "sparse_mla.h")
EINVAL, ENOTSUP = -22, -95
FAKE = ctypes.c_void_p(0x10000)        # aligned, never dereferenced
MISALIGNED = ctypes.c_void_p(0x10008)


@pytest.fixture(scope="module")
def lib():
    srcs = B.sources() + [HEADER]
    stale = (not os.path.exists(B.LIB) or
             max(os.path.getmtime(s) for s in srcs + [os.path.join(B.CSRC, "smla_common.cuh")])
             > os.path.getmtime(B.LIB))
    if stale:
        B.build()
    return capi.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(sparse_mla_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert {"sparse_mla_fwd", "sparse_mla_bwd", "sparse_mla_bwd_workspace_bytes",
            "sparse_mla_check_indices", "sparse_mla_last_error", "sparse_mla_version"} <= set(syms)
    for s in syms:
        assert hasattr(lib, s), s


def test_version(lib):
    assert "sm_103a" in capi.sparse_mla_version()


def _fwd(lib, T=16, H=8, topk=64, scale=0.04, q=FAKE, kv=FAKE, idx=FAKE, out=FAKE, lse=FAKE):
    return lib.sparse_mla_fwd(q, kv, idx, None, T, H, topk, 1, scale, out, lse, None)


@pytest.mark.parametrize("kw,msg", [
    (dict(H=7), "H must be"),
    (dict(H=256), "H must be"),
    (dict(topk=100), "topk"),
    (dict(topk=0), "topk"),
    (dict(T=-1), "T must be"),
    (dict(scale=float("nan")), "scale"),
    (dict(scale=float("inf")), "scale"),
    (dict(q=None), "q must not be NULL"),
    (dict(lse=None), "lse must not be NULL"),
    (dict(kv=MISALIGNED), "kv must be 16-byte aligned"),
])
def test_fwd_rejects_bad_arguments(lib, kw, msg):
    assert _fwd(lib, **kw) == EINVAL
    assert msg in capi.sparse_mla_last_error()


def test_fwd_empty_is_a_noop(lib):
    assert _fwd(lib, T=0, q=None, kv=None, idx=None, out=None, lse=None) == 0
    assert capi.sparse_mla_last_error() == ""


def _bwd(lib, T=16, H=8, topk=64, mode=0, ws=FAKE, ws_bytes=1 << 20, dq=FAKE):
    return lib.sparse_mla_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, T, H, topk, 1, 0.04, mode,
                              dq, FAKE, None, ws, ws_bytes, None)


def test_bwd_rejects_bad_arguments(lib):
    assert _bwd(lib, mode=1, ws_bytes=4096) == EINVAL          # smaller than one token's contributions
    assert "workspace too small" in capi.sparse_mla_last_error()
    assert _bwd(lib, mode=1, T=1 << 20, topk=4096) == EINVAL   # slot ids must fit int32
    assert "T * topk" in capi.sparse_mla_last_error()
    assert _bwd(lib, mode=7) == EINVAL
    assert _bwd(lib, ws_bytes=16) == EINVAL
    assert "workspace too small" in capi.sparse_mla_last_error()
    assert _bwd(lib, ws=None) == EINVAL
    assert _bwd(lib, dq=MISALIGNED) == EINVAL
    assert _bwd(lib, H=12) == EINVAL
    assert _bwd(lib, T=0) == 0


def test_workspace_bytes(lib):
    assert capi.sparse_mla_bwd_workspace_bytes(1000, 128, 2048) >= 1000 * 128 * 4
    assert capi.sparse_mla_bwd_workspace_bytes(1000, 12, 2048) == 0
    assert capi.sparse_mla_bwd_workspace_bytes(1000, 8, 100) == 0
    # deterministic mode: Delta, the slot lists (T * topk ints and more) and one chunk of
    # per-slot contributions (all 1000 tokens fit in the default 4 GiB chunk here)
    det = capi.sparse_mla_bwd_workspace_bytes(1000, 8, 64, 1)
    assert det >= 1000 * 8 * 4 + 4 * 1000 * 64 + 1000 * 64 * 576 * 4
    # the default chunk is capped: at the headline size it is 4 GiB of contributions
    big = capi.sparse_mla_bwd_workspace_bytes(65536, 128, 2048, 1)
    assert 4 << 30 <= big <= (4 << 30) + 65536 * 128 * 4 + 4 * (3 * 65536 + 65536 * 2048) + (1 << 20)
    assert capi.sparse_mla_bwd_workspace_bytes(1 << 20, 8, 4096, 1) == 0


def test_check_indices_rejects_bad_arguments(lib):
    n = ctypes.c_int64(-1)
    assert lib.sparse_mla_check_indices(FAKE, 16, 64, FAKE, 0, ctypes.byref(n), None) == EINVAL
    assert lib.sparse_mla_check_indices(FAKE, 16, 64, None, 1, ctypes.byref(n), None) == EINVAL
    assert lib.sparse_mla_check_indices(FAKE, 16, 64, FAKE, 1, None, None) == EINVAL
    assert lib.sparse_mla_check_indices(None, 0, 64, None, 1, ctypes.byref(n), None) == 0
    assert n.value == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(capi, "_lib", None)
    monkeypatch.setattr(capi, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        capi.load()


def test_topk_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    ok = dict(ld=64, T=16, ncols=64, B=1, topk=8)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.sparse_mla_topk(FAKE, a["ld"], a["T"], a["ncols"], FAKE, a["B"], a["topk"], FAKE, None)
    assert call(ncols=65) == EINVAL                         # ncols > ld
    assert call(topk=0) == EINVAL
    assert call(topk=8193, ncols=64) == EINVAL           # the sort holds 8 pairs per thread of 1024
    assert "topk" in capi.sparse_mla_last_error()
    assert call(B=0) == EINVAL
    assert call(ld=60000, ncols=60000) == EINVAL            # beyond the shared-memory selection
    assert "shared-memory selection" in capi.sparse_mla_last_error()
    assert call(T=0) == 0
    assert lib.sparse_mla_topk(None, 64, 16, 64, FAKE, 1, 8, FAKE, None) == EINVAL



def _fwd_rows(lib, T=16, t0=0, nt=16, q=FAKE, out=FAKE):
    return lib.sparse_mla_fwd_rows(q, FAKE, FAKE, None, T, 8, 64, 1, 0.04, t0, nt, out, FAKE, None)


def _bwd_rows(lib, T=16, t0=0, nt=16, ws_bytes=1 << 20, dkv=FAKE):
    return lib.sparse_mla_bwd_rows(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, T, 8, 64, 1, 0.04, t0, nt, FAKE, dkv,
                                   FAKE, ws_bytes, None)


@pytest.mark.parametrize("call", [_fwd_rows, _bwd_rows])
@pytest.mark.parametrize("t0,nt", [(-1, 4), (0, -1), (10, 7), (16, 1), (2**31 - 1, 2)])
def test_row_ranges_outside_the_tokens_are_rejected(lib, call, t0, nt):
    assert call(lib, t0=t0, nt=nt) == EINVAL
    assert "t0" in capi.sparse_mla_last_error()


@pytest.mark.parametrize("call", [_fwd_rows, _bwd_rows])
def test_empty_row_range_is_a_noop(lib, call):
    assert call(lib, t0=16, nt=0) == 0               # the range [T, T) is empty, and valid
    assert call(lib, t0=3, nt=0) == 0
    assert capi.sparse_mla_last_error() == ""


def test_row_calls_check_pointers_and_workspace(lib):
    assert _fwd_rows(lib, q=None) == EINVAL
    assert "q must not be NULL" in capi.sparse_mla_last_error()
    assert _fwd_rows(lib, out=MISALIGNED) == EINVAL
    assert _bwd_rows(lib, dkv=None) == EINVAL
    assert "dkv_f32 must not be NULL" in capi.sparse_mla_last_error()
    assert _bwd_rows(lib, ws_bytes=16 * 8 * 4 - 1) == EINVAL     # Delta needs T * H fp32 values
    assert "workspace too small" in capi.sparse_mla_last_error()


def test_dkv_cast_checks(lib):
    assert lib.sparse_mla_dkv_cast(FAKE, FAKE, -1, None) == EINVAL
    assert lib.sparse_mla_dkv_cast(None, FAKE, 4, None) == EINVAL
    assert lib.sparse_mla_dkv_cast(FAKE, MISALIGNED, 4, None) == EINVAL
    assert lib.sparse_mla_dkv_cast(None, None, 0, None) == 0


def test_bounds_selftest_is_refused_in_the_product_build(lib):
    # the product build compiles the device bounds checks away, so it has nothing to test
    assert lib.sparse_mla_bounds_selftest(None) == -38        # -ENOSYS
    assert "debug build" in capi.sparse_mla_last_error()


def test_debug_build_compiles_and_exports_every_declared_symbol(tmp_path):
    lib_path = str(tmp_path / "libsparse_mla_debug.so")
    B.build(["-DSMLA_DEBUG"], lib=lib_path, obj=str(tmp_path / "obj"))
    dbg = ctypes.CDLL(lib_path)
    for s in declared_symbols():
        assert hasattr(dbg, s), s
