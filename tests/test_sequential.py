"""GPU parity of the sequential evaluation (chunk = 1: one token at a time,
state in registers) against the float64 oracle, on both path settings; token
by token decoding through the final state; and the sequential kernels as a
cross-check of the chunked ones at a size the oracle would take longer on."""
import numpy as np
import pytest

from conftest import rel_err
from oracle import ssd_bwd_ref, ssd_fwd_ref
from ssd_chunked_scan_gb300.inputs import WORKLOADS, make_inputs, make_state_cotangent

from gpu_common import TOL, compare, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # B, L, G, H, dk, dv, la_mu, with_h0
    (1, 1, 1, 1, 16, 16, 0.0, True),
    (2, 37, 1, 2, 5, 3, 0.0, True),
    (2, 63, 2, 4, 48, 40, 0.0, False),
    (1, 100, 1, 3, 100, 70, -3.0, True),
    (2, 300, 2, 8, 128, 128, -3.0, True),
    (3, 77, 3, 3, 33, 65, 0.0, True),
]


def _set(path):
    from ssd_chunked_scan_gb300 import ssd
    ssd.ssd_set_path(ssd.SSD_PATH_SIMT if path == "simt" else ssd.SSD_PATH_TC)
    return ssd


def _np(d):
    return {n: (None if t is None else t.cpu().numpy()) for n, t in d.items()}


@pytest.mark.parametrize("path", ["simt", "tc"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}L{}G{}H{}dk{}dv{}mu{}h{}".format(*c))
def test_sequential_parity(path, case):
    import torch
    B, L, G, H, dk, dv, mu, with_h0 = case
    seed = 4500 + CASES.index(case)
    q, k, v, la, h0, dout = make_inputs(B, L, G, H, dk, dv, seed=seed, la_mu=mu)
    h0 = h0 if with_h0 else None
    dhT = make_state_cotangent(B, H, dk, dv, seed)
    ssd = _set(path)
    tq, tk, tv, tla, th0, tdo, tdh = map(to_dev, (q, k, v, la, h0, dout, dhT))
    out, hT = ssd.ssd_fwd_ex(tq, tk, tv, tla, th0, chunk=1)
    g = ssd.ssd_bwd_ex(tq, tk, tv, tla, th0, tdo, tdh, chunk=1)
    torch.cuda.synchronize()
    assert ssd.ssd_last_device_error() == 0
    ref, rhT = ssd_fwd_ref(q, k, v, la, h0, return_final_state=True)
    rg = ssd_bwd_ref(q, k, v, la, h0, dout, dhT=dhT)
    compare("simt", out.cpu().numpy(), _np(g), ref, rg, label=f"seq {case}")
    assert rel_err(hT.cpu().numpy(), rhT) <= TOL["simt"]


@pytest.mark.parametrize("path", ["simt", "tc"])
def test_token_by_token_decoding(path):
    """Feeding one token per call with the state carried through h0 -> hT
    reproduces one call over the whole sequence."""
    import torch
    B, L, G, H, dk, dv = 2, 40, 2, 4, 64, 32
    q, k, v, la, h0, _ = make_inputs(B, L, G, H, dk, dv, seed=4600)
    ssd = _set(path)
    state = to_dev(h0)
    outs = []
    for t in range(L):
        sl = lambda x: to_dev(np.ascontiguousarray(x[:, t:t + 1]))
        o, state = ssd.ssd_fwd_ex(sl(q), sl(k), sl(v), sl(la), state, chunk=1)
        outs.append(o.cpu().numpy())
    torch.cuda.synchronize()
    ref, rhT = ssd_fwd_ref(q, k, v, la, h0, return_final_state=True)
    assert rel_err(np.concatenate(outs, axis=1), ref) <= TOL["simt"]
    assert rel_err(state.cpu().numpy(), rhT) <= TOL["simt"]


def _unit(x, b, sl):
    return np.ascontiguousarray(x[b:b + 1, :, sl])


def test_sequential_full_size_unit():
    """The long benchmark workload at full size, sequentially; one
    (batch, group) unit against the oracle."""
    import torch
    from ssd_chunked_scan_gb300.inputs import workload_inputs
    w = [x for x in WORKLOADS if x.L >= 8192][-1]
    q, k, v, la, h0, dout = workload_inputs(w)
    ssd = _set("simt")
    tq, tk, tv, tla, th0, tdo = map(to_dev, (q, k, v, la, h0, dout))
    out = ssd.ssd_fwd(tq, tk, tv, tla, th0, chunk=1).cpu().numpy()
    g = _np(ssd.ssd_bwd(tq, tk, tv, tla, th0, tdo, chunk=1))
    torch.cuda.synchronize()
    assert ssd.ssd_last_device_error() == 0
    hpg = w.H // w.G
    b, gi = w.B - 1, w.G - 1
    gs, hs = slice(gi, gi + 1), slice(gi * hpg, (gi + 1) * hpg)
    uq, uk = _unit(q, b, gs), _unit(k, b, gs)
    uv, ula, udo = _unit(v, b, hs), _unit(la, b, hs), _unit(dout, b, hs)
    uh0 = np.ascontiguousarray(h0[b:b + 1, hs])
    ref = ssd_fwd_ref(uq, uk, uv, ula, uh0)
    rg = ssd_bwd_ref(uq, uk, uv, ula, uh0, udo)
    mine = {"dq": _unit(g["dq"], b, gs), "dk": _unit(g["dk"], b, gs),
            "dv": _unit(g["dv"], b, hs), "dlog_alpha": _unit(g["dlog_alpha"], b, hs),
            "dh0": np.ascontiguousarray(g["dh0"][b:b + 1, hs])}
    compare("simt", _unit(out, b, hs), mine, ref, rg, label=f"{w.name} sequential")


@pytest.mark.parametrize("path", ["simt", "tc"])
def test_chunked_agrees_with_sequential(path):
    """Whole-tensor cross-check of a chunked path against the sequential
    kernels at a size where every (batch, head) is compared."""
    import torch
    B, L, G, H, dk, dv = 2, 4096, 2, 8, 128, 128
    q, k, v, la, h0, dout = map(to_dev, make_inputs(B, L, G, H, dk, dv, seed=4700, la_mu=-3.0))
    ssd = _set(path)
    o_c = ssd.ssd_fwd(q, k, v, la, h0, chunk=64)
    g_c = ssd.ssd_bwd(q, k, v, la, h0, dout, chunk=64)
    o_s = ssd.ssd_fwd(q, k, v, la, h0, chunk=1)
    g_s = ssd.ssd_bwd(q, k, v, la, h0, dout, chunk=1)
    torch.cuda.synchronize()
    errs = {"out": rel_err(o_c.cpu().numpy(), o_s.cpu().numpy())}
    for n in g_c:
        errs[n] = rel_err(g_c[n].cpu().numpy(), g_s[n].cpu().numpy())
    assert max(errs.values()) <= TOL[path], errs
