"""GPU parity of the final-state entry points (ssd_fwd_ex / ssd_bwd_ex)
against the float64 oracle: the final state hT, the gradients with a final
state cotangent dhT, sequences processed in two pieces chained through
hT / dh0, and the empty sequence."""
import numpy as np
import pytest

from conftest import rel_err
from oracle import ssd_bwd_ref, ssd_fwd_ref
from ssd_chunked_scan_gb300.inputs import WORKLOADS, make_inputs, make_state_cotangent

from gpu_common import TOL, compare, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # B, L, G, H, dk, dv, chunk, la_mu, with_h0
    (2, 1, 1, 1, 16, 16, 64, 0.0, True),
    (2, 63, 2, 4, 48, 40, 64, 0.0, True),
    (1, 200, 1, 3, 64, 32, 64, -3.0, False),
    (2, 300, 2, 8, 128, 128, 64, -3.0, True),
    (1, 1000, 1, 2, 128, 64, 64, -3.0, True),
    (2, 50, 1, 2, 5, 3, 16, 0.0, True),
    (1, 90, 1, 1, 100, 70, 32, 0.0, True),
]


def _supported(path, dk, dv, chunk):
    if path == "simt":
        return chunk in (16, 32, 64) and dk <= 128 and dv <= 128
    return chunk == 64 and dk % 8 == 0 and dv % 8 == 0 and dk <= 128 and dv <= 128


def _set(path):
    from ssd_chunked_scan_gb300 import ssd
    ssd.ssd_set_path(ssd.SSD_PATH_SIMT if path == "simt" else ssd.SSD_PATH_TC)
    return ssd


def _np(d):
    return {n: (None if t is None else t.cpu().numpy()) for n, t in d.items()}


def _run(path, q, k, v, la, h0, dout, dhT, chunk):
    import torch
    ssd = _set(path)
    tq, tk, tv, tla, th0, tdo, tdh = map(to_dev, (q, k, v, la, h0, dout, dhT))
    out, hT = ssd.ssd_fwd_ex(tq, tk, tv, tla, th0, chunk=chunk)
    g = ssd.ssd_bwd_ex(tq, tk, tv, tla, th0, tdo, tdh, chunk=chunk)
    torch.cuda.synchronize()
    assert ssd.ssd_last_device_error() == 0
    return out.cpu().numpy(), hT.cpu().numpy(), _np(g)


@pytest.mark.parametrize("path", ["simt", "tc"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}L{}G{}H{}dk{}dv{}c{}mu{}h{}".format(*c))
def test_final_state_parity(path, case):
    B, L, G, H, dk, dv, chunk, mu, with_h0 = case
    if not _supported(path, dk, dv, chunk):
        pytest.skip("shape not taken by this path")
    seed = 4000 + CASES.index(case)
    q, k, v, la, h0, dout = make_inputs(B, L, G, H, dk, dv, seed=seed, la_mu=mu)
    h0 = h0 if with_h0 else None
    dhT = make_state_cotangent(B, H, dk, dv, seed)
    out, hT, g = _run(path, q, k, v, la, h0, dout, dhT, chunk)
    ref, rhT = ssd_fwd_ref(q, k, v, la, h0, return_final_state=True)
    rg = ssd_bwd_ref(q, k, v, la, h0, dout, dhT=dhT)
    compare(path, out, g, ref, rg, label=str(case))
    assert rel_err(hT, rhT) <= TOL[path], (case, rel_err(hT, rhT))


@pytest.mark.parametrize("path", ["simt", "tc"])
def test_final_state_without_cotangent_matches_plain_entry_points(path):
    import torch
    B, L, G, H, dk, dv = 2, 333, 2, 4, 64, 64
    q, k, v, la, h0, dout = make_inputs(B, L, G, H, dk, dv, seed=4100)
    ssd = _set(path)
    tq, tk, tv, tla, th0, tdo = map(to_dev, (q, k, v, la, h0, dout))
    out_ex, _ = ssd.ssd_fwd_ex(tq, tk, tv, tla, th0)
    g_ex = ssd.ssd_bwd_ex(tq, tk, tv, tla, th0, tdo, None)
    out = ssd.ssd_fwd(tq, tk, tv, tla, th0)
    g = ssd.ssd_bwd(tq, tk, tv, tla, th0, tdo)
    torch.cuda.synchronize()
    assert torch.equal(out, out_ex)
    for n in ("dv", "dh0"):  # no atomics: bitwise equal
        assert torch.equal(g[n], g_ex[n]), n
    for n in ("dq", "dk", "dlog_alpha"):
        assert rel_err(g_ex[n].cpu().numpy(), g[n].cpu().numpy()) <= TOL[path] / 10, n


@pytest.mark.parametrize("path", ["simt", "tc"])
def test_sequence_split_chains_state_and_gradients(path):
    """Forward over [0, L1) then [L1, L) from the first piece's hT, and the
    backward of the second piece feeding its dh0 to the first as dhT, equal
    one run over [0, L) (here checked against the oracle of the whole)."""
    import torch
    B, L, G, H, dk, dv, L1 = 2, 700, 2, 4, 64, 32, 257
    q, k, v, la, h0, dout = make_inputs(B, L, G, H, dk, dv, seed=4200, la_mu=-3.0)
    ssd = _set(path)
    T = lambda x, a, b: to_dev(np.ascontiguousarray(x[:, a:b]))
    parts = [(0, L1), (L1, L)]
    th0 = to_dev(h0)
    outs, states = [], [th0]
    for a, b in parts:
        o, hT = ssd.ssd_fwd_ex(T(q, a, b), T(k, a, b), T(v, a, b), T(la, a, b), states[-1])
        outs.append(o.cpu().numpy())
        states.append(hT)
    grads = [None, None]
    dnext = None
    for i in (1, 0):
        a, b = parts[i]
        grads[i] = _np(ssd.ssd_bwd_ex(T(q, a, b), T(k, a, b), T(v, a, b), T(la, a, b), states[i],
                                      T(dout, a, b), dnext))
        dnext = to_dev(grads[i]["dh0"])
    torch.cuda.synchronize()
    assert ssd.ssd_last_device_error() == 0
    ref, rhT = ssd_fwd_ref(q, k, v, la, h0, return_final_state=True)
    rg = ssd_bwd_ref(q, k, v, la, h0, dout)
    mine = {n: np.concatenate([grads[0][n], grads[1][n]], axis=1)
            for n in ("dq", "dk", "dv", "dlog_alpha")}
    mine["dh0"] = grads[0]["dh0"]
    compare(path, np.concatenate(outs, axis=1), mine, ref, rg, label="split")
    assert rel_err(states[-1].cpu().numpy(), rhT) <= TOL[path]


@pytest.mark.parametrize("path", ["simt", "tc"])
def test_empty_sequence_passes_state_through(path):
    import torch
    ssd = _set(path)
    B, H, G, dk, dv = 2, 4, 2, 16, 8
    e = torch.zeros((B, 0, G, dk), device="cuda")
    ev = torch.zeros((B, 0, H, dv), device="cuda")
    ela = torch.zeros((B, 0, H), device="cuda")
    h0 = torch.randn((B, H, dk, dv), device="cuda")
    dhT = torch.randn((B, H, dk, dv), device="cuda")
    _, hT = ssd.ssd_fwd_ex(e, e, ev, ela, h0)
    _, hz = ssd.ssd_fwd_ex(e, e, ev, ela, None)
    g = ssd.ssd_bwd_ex(e, e, ev, ela, h0, ev, dhT)
    torch.cuda.synchronize()
    assert torch.equal(hT, h0)
    assert torch.count_nonzero(hz).item() == 0
    assert torch.equal(g["dh0"], dhT)


def _unit(x, b, sl):
    return np.ascontiguousarray(x[b:b + 1, :, sl])


@pytest.mark.parametrize("path", ["simt", "tc"])
def test_final_state_full_size_unit(path):
    """The long benchmark workload at full size with a final-state cotangent;
    one (batch, group) unit against the oracle."""
    import torch
    from ssd_chunked_scan_gb300.inputs import workload_inputs
    w = [x for x in WORKLOADS if x.L >= 8192][-1]
    q, k, v, la, h0, dout = workload_inputs(w)
    dhT = make_state_cotangent(w.B, w.H, w.dk, w.dv, w.seed)
    out, hT, g = _run(path, q, k, v, la, h0, dout, dhT, w.chunk)
    hpg = w.H // w.G
    b, gi = w.B - 1, w.G - 1
    gs, hs = slice(gi, gi + 1), slice(gi * hpg, (gi + 1) * hpg)
    uq, uk = _unit(q, b, gs), _unit(k, b, gs)
    uv, ula, udo = _unit(v, b, hs), _unit(la, b, hs), _unit(dout, b, hs)
    uh0 = np.ascontiguousarray(h0[b:b + 1, hs])
    udh = np.ascontiguousarray(dhT[b:b + 1, hs])
    ref, rhT = ssd_fwd_ref(uq, uk, uv, ula, uh0, return_final_state=True)
    rg = ssd_bwd_ref(uq, uk, uv, ula, uh0, udo, dhT=udh)
    mine = {"dq": _unit(g["dq"], b, gs), "dk": _unit(g["dk"], b, gs),
            "dv": _unit(g["dv"], b, hs), "dlog_alpha": _unit(g["dlog_alpha"], b, hs),
            "dh0": np.ascontiguousarray(g["dh0"][b:b + 1, hs])}
    compare(path, _unit(out, b, hs), mine, ref, rg, label=f"{w.name} final state")
    assert rel_err(np.ascontiguousarray(hT[b:b + 1, hs]), rhT) <= TOL[path]
