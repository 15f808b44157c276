"""The allocation-free forward, ssd_fwd_noalloc, called through the C ABI.

It serves callers that cannot allocate device memory when they call the
library (their memory is reserved up front by another allocator, they run an
allocation-free real-time loop, or they are an allocator hook).  It must give
the same result as ssd_fwd on the all-fp32 path, call after call, although
every call reuses the same fixed scratch array.  This file is collected last
so that a stop-at-first-failure run has already run every other test."""
import ctypes

import numpy as np
import pytest

from ssd_chunked_scan_gb300.inputs import make_inputs

from conftest import rel_err

pytestmark = pytest.mark.gpu

TOL = 2e-5  # the all-fp32 path's tolerance


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _noalloc(lib, q, k, v, la, h0, out, chunk, stream):
    B, L, G, dk = q.shape
    H, dv = v.shape[2], v.shape[3]
    return lib.ssd_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(h0), _ptr(out),
                               B, L, G, H, dk, dv, chunk, stream)


def test_noalloc_matches_ssd_fwd_on_two_calls_in_a_row():
    import torch
    from ssd_chunked_scan_gb300 import ssd
    lib = ssd.LIB
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [(2, 300, 2, 4, 64, 64, 64, 11), (1, 517, 1, 3, 128, 128, 32, 12)]
    for B, L, G, H, dk, dv, chunk, seed in cases:  # two calls, different inputs
        q, k, v, la, h0, _ = (None if x is None else torch.from_numpy(x).cuda()
                              for x in make_inputs(B, L, G, H, dk, dv, seed=seed))
        ssd.ssd_set_path(ssd.SSD_PATH_SIMT)
        want = ssd.ssd_fwd(q, k, v, la, h0, chunk=chunk)
        out = torch.full_like(want, float("nan"))
        rc = _noalloc(lib, q, k, v, la, h0, out, chunk, stream)
        assert rc == 0, ssd.ssd_strerror(rc)
        torch.cuda.synchronize()
        e = rel_err(out.cpu().numpy(), want.cpu().numpy())
        assert e <= TOL, e


def test_noalloc_rejects_problems_beyond_its_scratch():
    import torch
    from ssd_chunked_scan_gb300 import ssd
    lib = ssd.LIB
    cap = lib.ssd_fwd_noalloc_scratch_bytes()
    assert cap == 32 << 20
    # B*H*ceil(L/64)*dk*dv*4 bytes above the cap; pointers are never touched
    x = torch.zeros(16, device="cuda")
    p = ctypes.c_void_p(x.data_ptr())
    rc = lib.ssd_fwd_noalloc(p, p, p, p, None, p, 4, 8192, 2, 8, 128, 128, 64, None)
    assert rc == ssd.SSD_ERR_SCRATCH
