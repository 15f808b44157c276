"""GPU parity of the Mamba-1 selective scan (include/ssd_mamba.h) against the
float64 oracle: small cases across segment and block boundaries, N < 16,
ragged channel blocks, no skip term, the empty sequence, and every Mamba
workload of the benchmark pages at full size, compared whole."""
import numpy as np
import pytest

from conftest import rel_err
from oracle import mamba_bwd_ref, mamba_fwd_ref
from ssd_chunked_scan_gb300.inputs import MAMBA_WORKLOADS, make_mamba_inputs, mamba_workload_inputs

from gpu_common import to_dev

pytestmark = pytest.mark.gpu

# fp32 throughout; the bar of the all-fp32 SSD path
TOL = 2e-5

SMALL = [
    # B, L, D, N, with_D
    (1, 1, 1, 1, True),
    (2, 37, 5, 16, True),
    (2, 100, 33, 16, False),
    (1, 300, 70, 4, True),
    (3, 64, 16, 16, True),
    (2, 1025, 48, 16, True),
    (1, 3000, 20, 7, True),
]


def run_gpu(x, dt, A, Bm, Cm, Dk, dy):
    import torch
    from ssd_chunked_scan_gb300 import ssd
    tx, tdt, tA, tB, tC, tD, tdy = map(to_dev, (x, dt, A, Bm, Cm, Dk, dy))
    y = ssd.ssd_mamba_fwd(tx, tdt, tA, tB, tC, tD)
    g = ssd.ssd_mamba_bwd(tx, tdt, tA, tB, tC, tD, tdy)
    torch.cuda.synchronize()
    return y.cpu().numpy(), {n: (None if t is None else t.cpu().numpy()) for n, t in g.items()}


def check(y, g, x, dt, A, Bm, Cm, Dk, dy, label):
    ref = mamba_fwd_ref(x, dt, A, Bm, Cm, Dk)
    rg = mamba_bwd_ref(x, dt, A, Bm, Cm, Dk, dy)
    errs = {"y": rel_err(y, ref)}
    for n in ("dx", "ddelta", "dA", "dB", "dC", "dD"):
        if rg[n] is not None:
            errs[n] = rel_err(g[n], rg[n])
    bad = {n: e for n, e in errs.items() if not e <= TOL}
    assert not bad, f"{label}: rel_err above {TOL}: {bad} (all {errs})"
    return errs


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "B{}L{}D{}N{}skip{}".format(*c))
def test_mamba_small_parity(case):
    B, L, D, N, with_D = case
    x, dt, A, Bm, Cm, Dk, dy = make_mamba_inputs(B, L, D, N, seed=5000 + SMALL.index(case),
                                                 with_D=with_D)
    y, g = run_gpu(x, dt, A, Bm, Cm, Dk, dy)
    if not with_D:
        assert g["dD"] is None
    check(y, g, x, dt, A, Bm, Cm, Dk, dy, str(case))


def test_mamba_long_memory():
    # small steps (slow decay) carry state across many segments
    x, dt, A, Bm, Cm, Dk, dy = make_mamba_inputs(2, 4000, 32, 16, seed=5100)
    dt = (dt * 0.05).astype(np.float32)
    A = (A * 0.1).astype(np.float32)
    y, g = run_gpu(x, dt, A, Bm, Cm, Dk, dy)
    check(y, g, x, dt, A, Bm, Cm, Dk, dy, "long memory")


def test_mamba_empty_and_argument_errors():
    import torch
    from ssd_chunked_scan_gb300 import ssd
    x = torch.zeros((2, 0, 8), device="cuda")
    bc = torch.zeros((2, 0, 4), device="cuda")
    A = torch.randn((8, 4), device="cuda")
    Dk = torch.randn((8,), device="cuda")
    y = ssd.ssd_mamba_fwd(x, x, A, bc, bc, Dk)
    g = ssd.ssd_mamba_bwd(x, x, A, bc, bc, Dk, x)
    torch.cuda.synchronize()
    assert y.shape == (2, 0, 8)
    assert torch.count_nonzero(g["dA"]).item() == 0 and torch.count_nonzero(g["dD"]).item() == 0
    with pytest.raises(ssd.SSDError):
        A17 = torch.randn((8, 17), device="cuda")
        ssd.ssd_mamba_fwd(torch.zeros((1, 4, 8), device="cuda"), torch.zeros((1, 4, 8), device="cuda"),
                          A17, torch.zeros((1, 4, 17), device="cuda"),
                          torch.zeros((1, 4, 17), device="cuda"))


@pytest.mark.parametrize("w", MAMBA_WORKLOADS, ids=lambda w: w.name)
def test_mamba_workload_parity(w):
    x, dt, A, Bm, Cm, Dk, dy = mamba_workload_inputs(w)
    y, g = run_gpu(x, dt, A, Bm, Cm, Dk, dy)
    check(y, g, x, dt, A, Bm, Cm, Dk, dy, w.name)
