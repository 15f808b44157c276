"""The tensor-core backward with its dk / dv passes on the library's side
stream (the default) against the same backward with every kernel on the
caller's stream: the same gradients (bit for bit where no float atomics are
involved; dq and dk sum a group's heads with atomic adds), and backward calls
from several host threads on their own streams at once stay correct."""
import threading

import numpy as np
import pytest

from oracle import ssd_bwd_ref
from ssd_chunked_scan_gb300.inputs import make_inputs

from gpu_common import to_dev

pytestmark = pytest.mark.gpu

CASE = dict(B=2, L=300, G=2, H=8, dk=128, dv=128)


def _inputs(seed):
    return make_inputs(CASE["B"], CASE["L"], CASE["G"], CASE["H"], CASE["dk"], CASE["dv"],
                       seed=seed, la_mu=-3.0)


def _bwd(ssd, torch, dev_in, overlap, stream=None):
    prev = ssd.ssd_set_overlap(overlap)
    try:
        g = ssd.ssd_bwd(*dev_in, chunk=64, stream=stream)
        torch.cuda.synchronize()
    finally:
        ssd.ssd_set_overlap(prev)
    assert ssd.ssd_last_device_error() == 0
    return {n: t.cpu().numpy() for n, t in g.items() if t is not None}


def test_overlap_matches_serial():
    import torch
    from ssd_chunked_scan_gb300 import ssd
    ssd.ssd_set_path(ssd.SSD_PATH_TC)
    host = _inputs(7)
    dev_in = [to_dev(x) for x in host]
    on = _bwd(ssd, torch, dev_in, True)
    off = _bwd(ssd, torch, dev_in, False)
    for n in ("dv", "dlog_alpha", "dh0"):
        assert np.array_equal(on[n], off[n]), n
    for n in ("dq", "dk"):
        scale = np.abs(off[n]).max()
        assert np.abs(on[n] - off[n]).max() <= 1e-6 * scale, n
    ref = ssd_bwd_ref(*host)
    errs = {n: np.abs(on[n] - ref[n]).max() / np.abs(ref[n]).max() for n in on}
    assert all(e <= 3e-3 for e in errs.values()), errs


def test_backward_from_several_host_threads():
    """Four host threads, each on its own stream with its own inputs, call the
    backward (overlap on) repeatedly at the same time; every result equals
    that input's serial result up to the order of the atomic adds."""
    import torch
    from ssd_chunked_scan_gb300 import ssd
    ssd.ssd_set_path(ssd.SSD_PATH_TC)
    n_thr, reps = 4, 3
    dev_ins = [[to_dev(x) for x in _inputs(100 + i)] for i in range(n_thr)]
    serial = [_bwd(ssd, torch, d, False) for d in dev_ins]
    results = [[None] * reps for _ in range(n_thr)]
    errors = []

    def work(i):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for r in range(reps):
                    g = ssd.ssd_bwd(*dev_ins[i], chunk=64, stream=st)
                    st.synchronize()
                    results[i][r] = {n: t.cpu().numpy() for n, t in g.items() if t is not None}
        except Exception as e:  # reported below, on the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(n_thr)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert ssd.ssd_last_device_error() == 0
    for i in range(n_thr):
        for r in range(reps):
            got = results[i][r]
            for n in ("dv", "dlog_alpha", "dh0"):
                assert np.array_equal(got[n], serial[i][n]), (i, r, n)
            for n in ("dq", "dk"):
                scale = np.abs(serial[i][n]).max()
                assert np.abs(got[n] - serial[i][n]).max() <= 1e-6 * scale, (i, r, n)
