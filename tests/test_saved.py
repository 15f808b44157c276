"""GPU parity of the saved-state entry points (ssd_fwd_save / ssd_bwd_saved)
against the float64 oracle: the backward that reads the forward's segment
states instead of recomputing them gives the same gradients (with and
without a final-state cotangent), on both paths (the CUDA-core path keeps no
states and recomputes), at small sizes spanning several segments and a
ragged last chunk, and on sampled units of the full-size benchmark workload
in the benchmark's configuration."""
import numpy as np
import pytest

from oracle import ssd_bwd_ref, ssd_fwd_ref
from ssd_chunked_scan_gb300.inputs import WORKLOADS, make_inputs, make_state_cotangent

from gpu_common import compare, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # B, L, G, H, dk, dv, chunk, la_mu, with_h0
    (2, 1, 1, 1, 16, 16, 64, 0.0, True),
    (2, 63, 2, 4, 48, 40, 64, 0.0, True),
    (1, 200, 1, 3, 64, 32, 64, -3.0, False),
    (2, 300, 2, 8, 128, 128, 64, -3.0, True),
    (1, 1000, 1, 2, 128, 64, 64, -3.0, True),
    (2, 90, 1, 2, 40, 96, 64, -3.0, True),
    (2, 50, 1, 2, 5, 3, 16, 0.0, True),
]


def _supported(path, dk, dv, chunk):
    if path == "simt":
        return chunk in (16, 32, 64) and dk <= 128 and dv <= 128
    return chunk == 64 and dk % 8 == 0 and dv % 8 == 0 and dk <= 128 and dv <= 128


def _np(d):
    return {n: (None if t is None else t.cpu().numpy()) for n, t in d.items()}


def _run(path, q, k, v, la, h0, dout, dhT, chunk):
    import torch
    from ssd_chunked_scan_gb300 import ssd
    ssd.ssd_set_path(ssd.SSD_PATH_SIMT if path == "simt" else ssd.SSD_PATH_TC)
    tq, tk, tv, tla, th0, tdo, tdh = map(to_dev, (q, k, v, la, h0, dout, dhT))
    out, hT, saved = ssd.ssd_fwd_save(tq, tk, tv, tla, th0, chunk=chunk)
    if path == "simt":
        assert saved is None
    else:
        assert saved is not None and saved.numel() % (q.shape[0] * v.shape[2] * q.shape[3] * v.shape[3]) == 0
    g = ssd.ssd_bwd_saved(tq, tk, tv, tla, th0, tdo, tdh, hT, saved, chunk=chunk)
    torch.cuda.synchronize()
    assert ssd.ssd_last_device_error() == 0
    return out.cpu().numpy(), hT.cpu().numpy(), _np(g)


@pytest.mark.parametrize("path", ["simt", "tc"])
@pytest.mark.parametrize("with_dhT", [False, True])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}L{}G{}H{}dk{}dv{}c{}mu{}h{}".format(*c))
def test_saved_parity(path, with_dhT, case):
    B, L, G, H, dk, dv, chunk, mu, with_h0 = case
    if not _supported(path, dk, dv, chunk):
        pytest.skip("shape not taken by this path")
    q, k, v, la, h0, dout = make_inputs(B, L, G, H, dk, dv, seed=hash(case) % 10000 + 7, la_mu=mu)
    if not with_h0:
        h0 = None
    dhT = make_state_cotangent(B, H, dk, dv, seed=hash(case) % 1000) if with_dhT else None
    out, hT, g = _run(path, q, k, v, la, h0, dout, dhT, chunk)
    ref_out, ref_hT = ssd_fwd_ref(q, k, v, la, h0, return_final_state=True)
    rg = ssd_bwd_ref(q, k, v, la, h0, dout, dhT=dhT)
    compare(path, out, g, ref_out, rg, label=f"saved {case} dhT={with_dhT}")
    compare(path, hT, None, ref_hT, None, label=f"saved hT {case}")


def _unit(x, b, sl):
    return np.ascontiguousarray(x[b:b + 1, :, sl])


@pytest.mark.parametrize("w", [w for w in WORKLOADS if w.dk % 8 == 0 and w.dv % 8 == 0 and w.chunk == 64],
                         ids=lambda w: w.name)
def test_saved_workload_parity(w):
    """Full-size workload on the tensor-core path; the first and last (batch,
    group) units against the oracle."""
    from ssd_chunked_scan_gb300.inputs import workload_inputs
    q, k, v, la, h0, dout = workload_inputs(w)
    out, _, g = _run("tc", q, k, v, la, h0, dout, None, w.chunk)
    hpg = w.H // w.G
    for b, gi in sorted({(0, 0), (w.B - 1, w.G - 1)}):
        gs, hs = slice(gi, gi + 1), slice(gi * hpg, (gi + 1) * hpg)
        uq, uk = _unit(q, b, gs), _unit(k, b, gs)
        uv, ula, udo = _unit(v, b, hs), _unit(la, b, hs), _unit(dout, b, hs)
        uh0 = np.ascontiguousarray(h0[b:b + 1, hs])
        ref = ssd_fwd_ref(uq, uk, uv, ula, uh0)
        rg = ssd_bwd_ref(uq, uk, uv, ula, uh0, udo)
        mine = {"dq": _unit(g["dq"], b, gs), "dk": _unit(g["dk"], b, gs),
                "dv": _unit(g["dv"], b, hs), "dlog_alpha": _unit(g["dlog_alpha"], b, hs),
                "dh0": np.ascontiguousarray(g["dh0"][b:b + 1, hs])}
        compare("tc", _unit(out, b, hs), mine, ref, rg, label=f"saved {w.name} unit b{b} g{gi}")


@pytest.mark.parametrize("shape", [(2, 300, 2, 8, 128, 128), (2, 129, 3, 6, 48, 40)],
                         ids=lambda s: "B{}L{}G{}H{}dk{}dv{}".format(*s))
def test_saved_with_every_backward_mode(shape):
    """The saved-state backward under each stream and group-sum mode: overlap
    on and off, atomic and deterministic group sums; all against the oracle,
    and the deterministic runs bitwise equal to each other."""
    import torch
    from ssd_chunked_scan_gb300 import ssd
    B, L, G, H, dk, dv = shape
    old = (ssd.ssd_get_path(), ssd.ssd_get_overlap(), ssd.ssd_get_deterministic())
    ssd.ssd_set_path(ssd.SSD_PATH_TC)
    try:
        q, k, v, la, h0, dout = make_inputs(B, L, G, H, dk, dv, seed=sum(shape) + 3, la_mu=-3.0)
        dhT = make_state_cotangent(B, H, dk, dv, seed=sum(shape))
        tq, tk, tv, tla, th0, tdo, tdh = map(to_dev, (q, k, v, la, h0, dout, dhT))
        out, hT, saved = ssd.ssd_fwd_save(tq, tk, tv, tla, th0, chunk=64)
        rg = ssd_bwd_ref(q, k, v, la, h0, dout, dhT=dhT)
        det_runs = []
        for overlap in (True, False):
            for det in (False, True):
                ssd.ssd_set_overlap(overlap)
                ssd.ssd_set_deterministic(det)
                g = ssd.ssd_bwd_saved(tq, tk, tv, tla, th0, tdo, tdh, hT, saved, chunk=64)
                torch.cuda.synchronize()
                assert ssd.ssd_last_device_error() == 0
                g = _np(g)
                compare("tc", out.cpu().numpy(), g, ssd_fwd_ref(q, k, v, la, h0), rg,
                        label=f"saved {shape} overlap={overlap} det={det}")
                if det:
                    det_runs.append(g)
        for n in det_runs[0]:
            assert np.array_equal(det_runs[0][n], det_runs[1][n]), n
    finally:
        ssd.ssd_set_path(old[0])
        ssd.ssd_set_overlap(bool(old[1]))
        ssd.ssd_set_deterministic(bool(old[2]))
