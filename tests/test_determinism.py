"""Deterministic group sums (ssd_set_deterministic) on the tensor-core path:
with grouped heads (H > G) the backward's dq and dk are bitwise identical
from run to run, with overlap on and off alike, agree with the float64
oracle and with the default atomic sums to within float rounding; without
the switch every other gradient is bitwise reproducible already."""
import numpy as np
import pytest

from oracle import ssd_bwd_ref
from ssd_chunked_scan_gb300.inputs import WORKLOADS, make_inputs

from gpu_common import to_dev

pytestmark = pytest.mark.gpu


def _bwd(ssd, torch, dev_in, det, overlap=True):
    pd, po = ssd.ssd_set_deterministic(det), ssd.ssd_set_overlap(overlap)
    try:
        g = ssd.ssd_bwd(*dev_in, chunk=64)
        torch.cuda.synchronize()
    finally:
        ssd.ssd_set_deterministic(pd)
        ssd.ssd_set_overlap(po)
    assert ssd.ssd_last_device_error() == 0
    return {n: t.cpu().numpy() for n, t in g.items() if t is not None}


@pytest.mark.parametrize("shape", [(2, 300, 2, 8, 128, 128), (1, 200, 1, 24, 128, 64), (2, 129, 3, 6, 48, 40)],
                         ids=lambda s: "B{}L{}G{}H{}dk{}dv{}".format(*s))
def test_grouped_gradients_are_bitwise_reproducible(shape):
    import torch
    from ssd_chunked_scan_gb300 import ssd
    B, L, G, H, dk, dv = shape
    old = ssd.ssd_get_path()
    ssd.ssd_set_path(ssd.SSD_PATH_TC)
    try:
        host = make_inputs(B, L, G, H, dk, dv, seed=sum(shape), la_mu=-3.0)
        dev_in = [to_dev(x) for x in host]
        runs = [_bwd(ssd, torch, dev_in, True, overlap=o) for o in (True, True, False)]
        for n in runs[0]:
            for r in runs[1:]:
                assert np.array_equal(runs[0][n], r[n]), n
        atomic = _bwd(ssd, torch, dev_in, False)
        for n in ("dq", "dk"):
            scale = np.abs(atomic[n]).max()
            assert np.abs(runs[0][n] - atomic[n]).max() <= 1e-6 * scale, n
        for n in ("dv", "dlog_alpha", "dh0"):
            assert np.array_equal(runs[0][n], atomic[n]), n
        ref = ssd_bwd_ref(*host)
        errs = {n: np.abs(runs[0][n] - ref[n]).max() / np.abs(ref[n]).max() for n in runs[0]}
        assert all(e <= 3e-3 for e in errs.values()), errs
    finally:
        ssd.ssd_set_path(old)


def test_long_workload_grouped_gradients_reproducible():
    """The benchmark's long-memory workload (4 heads per group), full size."""
    import torch
    from ssd_chunked_scan_gb300 import ssd
    from ssd_chunked_scan_gb300.inputs import workload_inputs
    w = [x for x in WORKLOADS if x.name == "g2h8_d128_L8192_long"][0]
    old = ssd.ssd_get_path()
    ssd.ssd_set_path(ssd.SSD_PATH_TC)
    try:
        dev_in = [to_dev(x) for x in workload_inputs(w)]
        a = _bwd(ssd, torch, dev_in, True)
        b = _bwd(ssd, torch, dev_in, True)
        for n in ("dq", "dk"):
            assert np.array_equal(a[n], b[n]), n
    finally:
        ssd.ssd_set_path(old)
