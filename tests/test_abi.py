"""The C ABI library: it loads without a GPU, exports every entry point that
include/ssd.h declares, and rejects bad arguments on the host before touching
the device (so these run on a CPU-only machine)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "ssd_chunked_scan_gb300", "_lib", "libssd.so")


def _declared():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            names |= set(re.findall(r"SSD_API\s+[\w\s\*]*?\b(ssd_\w+)\s*\(", txt))
    return names


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from ssd_chunked_scan_gb300.build import build_lib
        build_lib()
    l = ctypes.CDLL(LIB)
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    l.ssd_fwd.argtypes = [p] * 6 + [i64] * 7 + [p]
    l.ssd_bwd.argtypes = [p] * 11 + [i64] * 7 + [p]
    l.ssd_fwd_ex.argtypes = [p] * 7 + [i64] * 7 + [p]
    l.ssd_bwd_ex.argtypes = [p] * 12 + [i64] * 7 + [p]
    l.ssd_strerror.restype = ctypes.c_char_p
    sz = ctypes.POINTER(ctypes.c_size_t)
    l.ssd_fwd_workspace_bytes.argtypes = [i64] * 7 + [sz]
    l.ssd_bwd_workspace_bytes.argtypes = [i64] * 7 + [sz]
    return l


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"ssd_fwd", "ssd_bwd", "ssd_fwd_ex", "ssd_bwd_ex", "ssd_set_path",
            "ssd_strerror"} <= names
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_total(lib):
    for s in range(-1, 12):
        assert lib.ssd_strerror(s)
    assert lib.ssd_strerror(0) == b"ok"


def _fwd(lib, ptrs=(0x1000,) * 6, B=1, L=8, G=1, H=1, dk=8, dv=8, chunk=64):
    return lib.ssd_fwd(*[ctypes.c_void_p(x) for x in ptrs], B, L, G, H, dk, dv, chunk, None)


def _bwd(lib, ptrs=(0x1000,) * 11, B=1, L=8, G=1, H=1, dk=8, dv=8, chunk=64):
    return lib.ssd_bwd(*[ctypes.c_void_p(x) for x in ptrs], B, L, G, H, dk, dv, chunk, None)


def _fwd_ex(lib, ptrs=(0x1000,) * 7, B=1, L=8, G=1, H=1, dk=8, dv=8, chunk=64):
    return lib.ssd_fwd_ex(*[ctypes.c_void_p(x) for x in ptrs], B, L, G, H, dk, dv, chunk, None)


def _bwd_ex(lib, ptrs=(0x1000,) * 12, B=1, L=8, G=1, H=1, dk=8, dv=8, chunk=64):
    return lib.ssd_bwd_ex(*[ctypes.c_void_p(x) for x in ptrs], B, L, G, H, dk, dv, chunk, None)


@pytest.mark.parametrize("path", [0, 1])
def test_host_argument_checks_final_state(lib, path):
    assert lib.ssd_set_path(path) == 0
    assert _fwd_ex(lib, ptrs=(0x1000,) * 6 + (0x1004,)) == 2     # hT misaligned
    assert _bwd_ex(lib, ptrs=(0x1000,) * 6 + (0x100c,) + (0x1000,) * 5) == 2  # dhT
    assert _fwd_ex(lib, G=2, H=3) == 1
    assert _bwd_ex(lib, dv=0) == 1
    assert _fwd_ex(lib, L=0, ptrs=(0,) * 7) == 0    # empty, hT not wanted
    assert _bwd_ex(lib, L=0, ptrs=(0,) * 12) == 0   # empty, dh0 not wanted


@pytest.mark.parametrize("path", [0, 1])
def test_host_argument_checks(lib, path):
    assert lib.ssd_set_path(path) == 0
    assert _fwd(lib, G=2, H=3) == 1              # H % G != 0
    assert _fwd(lib, B=-1) == 1
    assert _fwd(lib, L=-5) == 1
    assert _fwd(lib, G=0) == 1
    assert _fwd(lib, dk=0) == 1
    assert _fwd(lib, chunk=0) == 1
    assert _fwd(lib, chunk=48) == 3              # no path takes chunk 48
    assert _fwd(lib, dk=512) == 4
    assert _fwd(lib, L=0) == 0                   # empty problem: nothing launched
    assert _fwd(lib, B=0) == 0
    assert _fwd(lib, ptrs=(0x1000, 0x1000, 0, 0x1000, 0, 0x1000)) == 1   # v NULL
    assert _fwd(lib, ptrs=(0x1000, 0x1004, 0x1000, 0x1000, 0, 0x1000)) == 2
    assert _bwd(lib, ptrs=(0x1000,) * 10 + (0x1008,)) == 2
    assert _bwd(lib, ptrs=(0x1000,) * 5 + (0,) + (0x1000,) * 5) == 1      # dout NULL
    assert _bwd(lib, L=0, ptrs=(0,) * 11) == 0   # empty, dh0 not wanted


def test_set_path(lib):
    assert lib.ssd_set_path(7) == 1
    assert lib.ssd_set_path(1) == 0 and lib.ssd_get_path() == 1
    assert lib.ssd_set_path(0) == 0 and lib.ssd_get_path() == 0


def test_version(lib):
    assert lib.ssd_version() == 400


def test_set_overlap(lib):
    first = lib.ssd_set_overlap(0)
    try:
        assert first == 1  # on by default
        assert lib.ssd_get_overlap() == 0
        assert lib.ssd_set_overlap(5) == 0 and lib.ssd_get_overlap() == 1
    finally:
        lib.ssd_set_overlap(first)


def test_set_deterministic(lib):
    first = lib.ssd_set_deterministic(1)
    try:
        assert first == 0  # off by default
        assert lib.ssd_get_deterministic() == 1
        assert lib.ssd_set_deterministic(0) == 1 and lib.ssd_get_deterministic() == 0
    finally:
        lib.ssd_set_deterministic(first)


def test_deterministic_sums_grow_the_workspace_by_the_per_head_gradients(lib):
    # tensor-core path, grouped heads: 2 * B * L * H * dk more floats (plus
    # alignment slack); ungrouped problems need no per-head buffers
    sz = lambda *a: (lambda n: (lib.ssd_bwd_workspace_bytes(*a, ctypes.byref(n)), n.value))(ctypes.c_size_t(0))
    assert lib.ssd_set_path(0) == 0
    first = lib.ssd_get_deterministic()
    try:
        lib.ssd_set_deterministic(0)
        rc0, off = sz(2, 300, 2, 8, 64, 64, 64)
        rc0b, off1 = sz(2, 300, 8, 8, 64, 64, 64)
        lib.ssd_set_deterministic(1)
        rc1, on = sz(2, 300, 2, 8, 64, 64, 64)
        rc1b, on1 = sz(2, 300, 8, 8, 64, 64, 64)
    finally:
        lib.ssd_set_deterministic(first)
    assert rc0 == rc1 == rc0b == rc1b == 0
    assert on - off == 4 * (2 * 2 * 300 * 8 * 64 + 4)
    assert on1 == off1


def test_injected_workspace_failure_is_reported_before_launch(lib, monkeypatch):
    # SSD_FAULT_ALLOC=1 makes the workspace request fail on the host; the
    # call must return SSD_ERR_ALLOC without enqueueing anything
    monkeypatch.setenv("SSD_FAULT_ALLOC", "1")
    assert lib.ssd_set_path(1) == 0
    assert _fwd(lib) == 5
    assert _bwd(lib) == 5
    assert _fwd_ex(lib) == 5
    assert _bwd_ex(lib) == 5


def _ws(lib, fn, *dims):
    n = ctypes.c_size_t(123)
    rc = getattr(lib, fn)(*dims, ctypes.byref(n))
    return rc, n.value


def test_workspace_queries(lib):
    # all-fp32 path: one state per chunk and pass, plus per-chunk decays
    assert lib.ssd_set_path(1) == 0
    B, L, G, H, dk, dv, C = 2, 1000, 2, 4, 48, 40, 64
    N = -(-L // C)
    assert _ws(lib, "ssd_fwd_workspace_bytes", B, L, G, H, dk, dv, C) == (
        0, 4 * (B * H * N * dk * dv + B * H * N))
    assert _ws(lib, "ssd_bwd_workspace_bytes", B, L, G, H, dk, dv, C) == (
        0, 4 * (2 * B * H * N * dk * dv + 2 * B * H * N + B * H * dk * dv))
    assert _ws(lib, "ssd_fwd_workspace_bytes", B, L, G, H, dk, dv, 48)[0] == 3
    assert _ws(lib, "ssd_fwd_workspace_bytes", B, 0, G, H, dk, dv, C) == (0, 0)
    assert lib.ssd_fwd_workspace_bytes(B, L, G, H, dk, dv, C, None) == 1
    # tensor-core path: the segment states do not grow with L
    assert lib.ssd_set_path(0) == 0
    rc1, a = _ws(lib, "ssd_bwd_workspace_bytes", 4, 8192, 2, 8, 128, 128, 64)
    rc2, b = _ws(lib, "ssd_bwd_workspace_bytes", 4, 8 * 8192, 2, 8, 128, 128, 64)
    assert rc1 == rc2 == 0 and 0 < a < b < 8 * a
    assert b - a == pytest.approx(4 * 3 * 4 * 7 * 8192 * 8, rel=0.05)  # per-token arrays only
    assert _ws(lib, "ssd_fwd_workspace_bytes", 1 << 16, 1 << 15, 1, 1, 8, 8, 64)[0] == 4  # B*L >= 2^31
    assert _ws(lib, "ssd_fwd_workspace_bytes", 1, 100, 1, 1, 12, 8, 64)[0] == 4          # dk % 8


@pytest.mark.parametrize("path", [0, 1])
def test_chunk_one_is_sequential_on_every_path(lib, path):
    assert lib.ssd_set_path(path) == 0
    assert _ws(lib, "ssd_fwd_workspace_bytes", 2, 100, 1, 2, 5, 3, 1) == (0, 0)
    B, L, H, dk, dv = 2, 100, 2, 5, 70
    nblk = -(-dv // 32)
    assert _ws(lib, "ssd_bwd_workspace_bytes", B, L, 1, H, dk, dv, 1) == (
        0, 4 * (2 * nblk * B * L * H + B * H * dk * dv))
    assert _ws(lib, "ssd_fwd_workspace_bytes", 2, 100, 1, 2, 129, 3, 1)[0] == 4
    assert _fwd(lib, dk=5, dv=3, chunk=1, ptrs=(0x1000, 0x1004) + (0x1000,) * 4) == 2


def test_mamba_host_checks(lib):
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.ssd_mamba_fwd.argtypes = [p] * 7 + [i64] * 4 + [p]
    lib.ssd_mamba_bwd.argtypes = [p] * 13 + [i64] * 4 + [p]
    lib.ssd_mamba_workspace_bytes.argtypes = [ctypes.c_int] + [i64] * 4 + [ctypes.POINTER(ctypes.c_size_t)]
    ok = [p(0x1000)] * 7
    assert lib.ssd_mamba_fwd(*ok, 1, 8, 4, 17, None) == 4      # N > 16
    assert lib.ssd_mamba_fwd(*ok, 1, 8, 0, 4, None) == 1       # D = 0
    assert lib.ssd_mamba_fwd(*([p(0x1000)] * 6 + [p(0x1008)]), 1, 8, 4, 4, None) == 2
    assert lib.ssd_mamba_fwd(*([p(0x1000)] * 2 + [p(0)] + [p(0x1000)] * 4), 1, 8, 4, 4, None) == 1
    assert lib.ssd_mamba_fwd(*ok, 1, 0, 4, 4, None) == 0       # empty
    n = ctypes.c_size_t(7)
    assert lib.ssd_mamba_workspace_bytes(0, 2, 0, 4, 4, ctypes.byref(n)) == 0 and n.value == 0
    assert lib.ssd_mamba_workspace_bytes(1, 4, 8192, 1024, 16, ctypes.byref(n)) == 0
    fwd_n = ctypes.c_size_t(0)
    assert lib.ssd_mamba_workspace_bytes(0, 4, 8192, 1024, 16, ctypes.byref(fwd_n)) == 0
    # forward: states + delta sums per segment; backward adds the u states
    assert 0 < fwd_n.value < n.value < 2 * fwd_n.value


def _fwd_save(lib, ptrs=(0x1000,) * 8, B=1, L=8, G=1, H=1, dk=8, dv=8, chunk=64):
    lib.ssd_fwd_save.argtypes = [ctypes.c_void_p] * 8 + [ctypes.c_int64] * 7 + [ctypes.c_void_p]
    return lib.ssd_fwd_save(*[ctypes.c_void_p(x) for x in ptrs], B, L, G, H, dk, dv, chunk, None)


def _bwd_saved(lib, ptrs=(0x1000,) * 14, B=1, L=8, G=1, H=1, dk=8, dv=8, chunk=64):
    lib.ssd_bwd_saved.argtypes = [ctypes.c_void_p] * 14 + [ctypes.c_int64] * 7 + [ctypes.c_void_p]
    return lib.ssd_bwd_saved(*[ctypes.c_void_p(x) for x in ptrs], B, L, G, H, dk, dv, chunk, None)


def _saved_bytes(lib, B=1, L=8, G=1, H=1, dk=8, dv=8, chunk=64):
    lib.ssd_saved_bytes.argtypes = [ctypes.c_int64] * 7 + [ctypes.POINTER(ctypes.c_size_t)]
    n = ctypes.c_size_t(123)
    rc = lib.ssd_saved_bytes(B, L, G, H, dk, dv, chunk, ctypes.byref(n))
    return rc, n.value


@pytest.mark.parametrize("path", [0, 1])
def test_host_argument_checks_saved_states(lib, path):
    assert lib.ssd_set_path(path) == 0
    assert _fwd_save(lib, ptrs=(0x1000,) * 7 + (0x1008,)) == 2                  # saved misaligned
    assert _bwd_saved(lib, ptrs=(0x1000,) * 8 + (0x1004,) + (0x1000,) * 5) == 2  # saved
    assert _bwd_saved(lib, ptrs=(0x1000,) * 7 + (0x100c,) + (0x1000,) * 6) == 2  # hT
    assert _fwd_save(lib, G=2, H=3) == 1
    assert _bwd_saved(lib, dk=0) == 1
    assert _fwd_save(lib, L=0, ptrs=(0,) * 8) == 0    # empty: nothing to keep
    assert _bwd_saved(lib, L=0, ptrs=(0,) * 14) == 0
    if path == 0:  # saved and dhT without the final state: refused before any launch
        assert _bwd_saved(lib, ptrs=(0x1000,) * 7 + (0,) + (0x1000,) * 6) == 1
    assert lib.ssd_set_path(0) == 0


def test_saved_bytes(lib):
    assert lib.ssd_set_path(0) == 0
    rc, n = _saved_bytes(lib, B=4, L=8192, G=2, H=8, dk=128, dv=128)
    # whole [dv x dk] states, one per (batch, head, segment), at least one segment
    unit = 4 * 8 * 128 * 128 * 4
    assert rc == 0 and n >= unit and n % unit == 0
    assert _saved_bytes(lib, L=0) == (0, 0)
    assert _saved_bytes(lib, chunk=1) == (0, 0)      # the sequential evaluation keeps none
    assert _saved_bytes(lib, G=2, H=3)[0] == 1
    assert lib.ssd_set_path(1) == 0
    assert _saved_bytes(lib) == (0, 0)               # nor does the CUDA-core path
    assert lib.ssd_set_path(0) == 0
    lib.ssd_saved_bytes.argtypes = [ctypes.c_int64] * 7 + [ctypes.c_void_p]
    assert lib.ssd_saved_bytes(1, 8, 1, 1, 8, 8, 64, None) == 1
