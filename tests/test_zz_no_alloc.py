"""The allocation-free forward, ssd_fwd_noalloc, called through the C ABI.

It serves callers that cannot allocate device memory when they call the
library (their memory is reserved up front by another allocator, they run an
allocation-free real-time loop, or they are an allocator hook).  Checked here:
its result against the float64 oracle, call after call (every call reuses the
same fixed scratch array), with and without an initial state; that a call
allocates nothing (the library's pool high-water mark and the device's free
memory are unchanged, also with tracing on); and its argument checks against
ssd_fwd's.  This file is collected last so that a stop-at-first-failure run
has already run every other test."""
import ctypes

import pytest

from ssd_chunked_scan_gb300.inputs import make_inputs

from conftest import rel_err

pytestmark = pytest.mark.gpu

TOL = 2e-5  # the all-fp32 path's tolerance


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _noalloc(lib, q, k, v, la, h0, out, chunk, stream, dims=None):
    B, L, G, dk = q.shape if dims is None else dims[:4]
    H, dv = (v.shape[2], v.shape[3]) if dims is None else dims[4:]
    return lib.ssd_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(h0), _ptr(out),
                               B, L, G, H, dk, dv, chunk, stream)


@pytest.fixture
def simt_path():
    from ssd_chunked_scan_gb300 import ssd
    old = ssd.ssd_get_path()
    ssd.ssd_set_path(ssd.SSD_PATH_SIMT)
    try:
        yield ssd
    finally:
        ssd.ssd_set_path(old)


CASES = [(2, 300, 2, 4, 64, 64, 64, 11, True), (1, 517, 1, 3, 128, 128, 32, 12, True),
         (1, 200, 1, 2, 40, 24, 16, 13, False)]


def test_noalloc_matches_oracle_on_calls_in_a_row(simt_path):
    import torch
    from oracle import ssd_fwd_ref
    ssd = simt_path
    lib = ssd.LIB
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for B, L, G, H, dk, dv, chunk, seed, with_h0 in CASES:  # different inputs each call
        q, k, v, la, h0, _ = make_inputs(B, L, G, H, dk, dv, seed=seed)
        if not with_h0:
            h0 = None
        ref = ssd_fwd_ref(q, k, v, la, h0)
        tq, tk, tv, tla, th0 = (None if x is None else torch.from_numpy(x).cuda()
                                for x in (q, k, v, la, h0))
        out = torch.full((B, L, H, dv), float("nan"), device="cuda")
        rc = _noalloc(lib, tq, tk, tv, tla, th0, out, chunk, stream)
        assert rc == 0, ssd.ssd_strerror(rc)
        torch.cuda.synchronize()
        assert ssd.ssd_last_device_error() == 0
        e = rel_err(out.cpu().numpy(), ref)
        assert e <= TOL, (B, L, G, H, dk, dv, chunk, with_h0, e)


def test_noalloc_allocates_nothing(simt_path):
    import torch
    ssd = simt_path
    lib = ssd.LIB
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    B, L, G, H, dk, dv, chunk = 2, 640, 2, 4, 64, 64, 64
    q, k, v, la, h0, _ = (torch.from_numpy(x).cuda() for x in make_inputs(B, L, G, H, dk, dv, seed=5))
    out = torch.empty(B, L, H, dv, device="cuda")
    assert _noalloc(lib, q, k, v, la, h0, out, chunk, stream) == 0  # warm-up (address lookup)
    torch.cuda.synchronize()
    for tracing in (False, True):
        ssd.ssd_trace_reset()
        ssd.ssd_trace_enable(tracing)
        try:
            ssd.ssd_pool_high_water(reset=True)
            hw0 = ssd.ssd_pool_high_water()
            launches = ssd.ssd_launch_count()
            free0, _ = torch.cuda.mem_get_info()
            for _ in range(3):
                assert _noalloc(lib, q, k, v, la, h0, out, chunk, stream) == 0
            torch.cuda.synchronize()
            free1, _ = torch.cuda.mem_get_info()
            assert ssd.ssd_pool_high_water() == hw0
            assert free1 == free0
            assert ssd.ssd_launch_count() > launches
            if tracing:
                assert ssd.ssd_trace_collect() == {}  # nothing was recorded
        finally:
            ssd.ssd_trace_enable(False)
            ssd.ssd_trace_reset()


def test_noalloc_checks_match_ssd_fwd(simt_path):
    import torch
    ssd = simt_path
    lib = ssd.LIB
    x = torch.zeros(64, device="cuda")
    p = ctypes.c_void_p(x.data_ptr())
    bad = ctypes.c_void_p(x.data_ptr() + 4)  # not 16-byte aligned

    def both(ptrs, dims, chunk):
        B, L, G, H, dk, dv = dims
        a = lib.ssd_fwd_noalloc(*ptrs, B, L, G, H, dk, dv, chunk, None)
        b = lib.ssd_fwd(*ptrs, B, L, G, H, dk, dv, chunk, None)
        return a, b

    good = (p, p, p, p, None, p)
    # misaligned pointer on an empty problem: both refuse the alignment first
    a, b = both((bad,) + good[1:], (0, 8, 1, 1, 8, 8), 64)
    assert a == b == ssd.SSD_ERR_ALIGN
    # empty problems are no-ops
    a, b = both(good, (1, 0, 1, 1, 8, 8), 64)
    assert a == b == ssd.SSD_OK
    # argument and shape errors
    for dims, chunk, want in [((1, 8, 2, 3, 8, 8), 64, ssd.SSD_ERR_ARG),
                              ((1, 8, 1, 1, 8, 8), 48, ssd.SSD_ERR_CHUNK),
                              ((1, 8, 1, 1, 136, 8), 64, ssd.SSD_ERR_UNSUPPORTED)]:
        a, b = both(good, dims, chunk)
        assert a == b == want, (dims, chunk, a, b)
    # chunk 1 is ssd_fwd's sequential evaluation; the allocation-free entry refuses it
    assert lib.ssd_fwd_noalloc(*good, 0, 8, 1, 1, 8, 8, 1, None) == ssd.SSD_ERR_CHUNK


def test_noalloc_rejects_problems_beyond_its_scratch(simt_path):
    import torch
    ssd = simt_path
    lib = ssd.LIB
    cap = lib.ssd_fwd_noalloc_scratch_bytes()
    assert cap == 32 << 20
    # B*H*ceil(L/64)*dk*dv*4 bytes above the cap; pointers are never touched
    x = torch.zeros(16, device="cuda")
    p = ctypes.c_void_p(x.data_ptr())
    rc = lib.ssd_fwd_noalloc(p, p, p, p, None, p, 4, 8192, 2, 8, 128, 128, 64, None)
    assert rc == ssd.SSD_ERR_SCRATCH
