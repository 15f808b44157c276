"""The library's two debugging aids.

* The SSD_CHECK variant (``build_lib(check=True)``): every global index of the
  tensor-core and CUDA-core kernels is tested against its buffer's size; a
  failed test sets the device check word and skips the access.  On the CPU:
  it builds and exports every entry point of include/ssd.h.  On the GPU: the
  small parity cases pass under it, with the error word clear after each call.
* The failure path of the bounded device-side waits: with the test switch
  ``ssd_test_stall_walks`` on, every tensor-core walk CTA waits on a barrier
  that nothing completes; the wait gives up after its limit, the kernel
  drains what it has in flight and returns, ``ssd_last_device_error`` reports
  SSD_ERR_TIMEOUT, and the next call (switch off) is correct again.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

from test_abi import _declared

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_check_variant_builds_and_exports():
    from ssd_chunked_scan_gb300.build import build_lib
    path = build_lib(check=True)
    assert os.path.basename(path) == "libssd_check.so"
    lib = ctypes.CDLL(path)
    for n in _declared():
        assert hasattr(lib, n), n
    lib.ssd_strerror.restype = ctypes.c_char_p
    assert b"index check" in lib.ssd_strerror(10)


@pytest.mark.gpu
def test_check_variant_small_parity():
    from ssd_chunked_scan_gb300.build import build_lib
    build_lib(check=True)
    env = dict(os.environ, SSD_LIB_VARIANT="check")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join(ROOT, "tests", "test_parity.py"),
           "-k", "small_parity or forget_everything or zero_cotangent"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                       text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:]
    assert " passed" in r.stdout


@pytest.mark.gpu
def test_bounded_wait_gives_up_and_recovers():
    import torch
    from oracle import ssd_fwd_ref
    from ssd_chunked_scan_gb300 import ssd
    from ssd_chunked_scan_gb300.inputs import make_inputs

    # 80 heads of one group: one segment per (batch, head), so every walk CTA
    # runs four chunks and the stall hits its second one, with the first
    # chunk's products done and later tiles in flight
    B, L, G, H, dk, dv = 1, 256, 1, 80, 64, 64
    q, k, v, la, h0, _ = make_inputs(B, L, G, H, dk, dv, seed=7)
    ref = ssd_fwd_ref(q, k, v, la, h0)
    t = lambda x: torch.from_numpy(x).cuda()
    tq, tk, tv, tla, th0 = map(t, (q, k, v, la, h0))
    old = ssd.ssd_get_path()
    ssd.ssd_set_path(ssd.SSD_PATH_TC)
    try:
        assert ssd.ssd_last_device_error() == ssd.SSD_OK
        ssd.ssd_test_stall_walks(True)
        try:
            ssd.ssd_fwd(tq, tk, tv, tla, th0, chunk=64)
            torch.cuda.synchronize()
            status = ssd.ssd_last_device_error()
        finally:
            ssd.ssd_test_stall_walks(False)
        assert status == ssd.SSD_ERR_TIMEOUT
        # the context is intact and the next call is correct
        out = ssd.ssd_fwd(tq, tk, tv, tla, th0, chunk=64)
        torch.cuda.synchronize()
        assert ssd.ssd_last_device_error() == ssd.SSD_OK
        x = out.cpu().numpy().astype(np.float64)
        err = float(np.max(np.abs(x - ref)) / np.max(np.abs(ref)))
        assert err <= 3e-3, err
    finally:
        ssd.ssd_set_path(old)
