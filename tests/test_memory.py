"""GPU: memory accounting and the largest index ranges.

The workspace a call takes matches what ssd_*_workspace_bytes reports, and
the kernels address tensors beyond 2^31 elements correctly (a v / out of
2^32 elements): outputs whose dependence is local to one end of the
sequence are compared with the float64 oracle on that end alone."""
import numpy as np
import pytest

from conftest import rel_err
from oracle import ssd_bwd_ref, ssd_fwd_ref
from ssd_chunked_scan_gb300.inputs import make_inputs, make_inputs_on_device

from gpu_common import TOL, to_dev

pytestmark = pytest.mark.gpu


def _set(path):
    from ssd_chunked_scan_gb300 import ssd
    ssd.ssd_set_path(ssd.SSD_PATH_SIMT if path == "simt" else ssd.SSD_PATH_TC)
    return ssd


@pytest.mark.parametrize("path", ["simt", "tc"])
def test_pool_high_water_matches_reported_workspace(path):
    import torch
    ssd = _set(path)
    B, L, G, H, dk, dv = 2, 3000, 2, 4, 64, 64
    q, k, v, la, h0, dout = map(to_dev, make_inputs(B, L, G, H, dk, dv, seed=4300))
    torch.cuda.synchronize()
    for fn, call in (("ssd_fwd_workspace_bytes", lambda: ssd.ssd_fwd(q, k, v, la, h0)),
                     ("ssd_bwd_workspace_bytes", lambda: ssd.ssd_bwd(q, k, v, la, h0, dout))):
        ws = getattr(ssd, fn)(B, L, G, H, dk, dv, 64)
        ssd.ssd_pool_high_water(reset=True)
        call()
        torch.cuda.synchronize()
        hw = ssd.ssd_pool_high_water()
        assert ws <= hw <= ws + (64 << 20), (fn, ws, hw)


@pytest.mark.parametrize("path", ["simt", "tc"])
def test_offsets_beyond_2_to_the_31(path):
    import torch
    ssd = _set(path)
    B, L, G, H, dk, dv, P = 2, 1 << 21, 1, 8, 64, 128, 512
    assert B * L * H * dv == 1 << 32
    dev = torch.device("cuda")
    q, k, v, la, h0, dout = make_inputs_on_device(dev, B, L, G, H, dk, dv, seed=4400, la_mu=-3.0)
    out = ssd.ssd_fwd(q, k, v, la, h0)
    g = ssd.ssd_bwd(q, k, v, la, h0, dout, want_dh0=False)
    torch.cuda.synchronize()
    assert ssd.ssd_last_device_error() == 0
    b = B - 1  # the last batch entry: the largest offsets
    host = lambda t, sl: np.ascontiguousarray(t[b:b + 1, sl].cpu().numpy())
    pre, suf = slice(0, P), slice(L - P, L)
    # out[t] for t < P depends only on the first P tokens and h0
    ref = ssd_fwd_ref(*(host(x, pre) for x in (q, k, v, la)), h0[b:b + 1].cpu().numpy())
    e_out = rel_err(host(out, pre), ref)
    # dk, dv of the last P tokens depend only on the last P tokens
    rg = ssd_bwd_ref(*(host(x, suf) for x in (q, k, v, la)), None, host(dout, suf))
    e_dk = rel_err(host(g["dk"], suf), rg["dk"])
    e_dv = rel_err(host(g["dv"], suf), rg["dv"])
    finite = bool(torch.isfinite(out).all()) and all(
        bool(torch.isfinite(t).all()) for t in g.values() if t is not None)
    del q, k, v, la, h0, dout, out, g
    torch.cuda.empty_cache()
    assert max(e_out, e_dk, e_dv) <= TOL[path], (e_out, e_dk, e_dv)
    assert finite
