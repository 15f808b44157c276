"""GPU parity: the CUDA library (through the C ABI) against the float64 oracle,
element by element on the same seeded inputs.

Small cases span several chunks and a ragged last chunk and cover the edge
cases (L = 1, empty, h0 absent, forget-everything decay, non-power-of-two
dk / dv, every chunk length a path takes).  The benchmark workloads run at
full size in the benchmark's launch configuration and are compared on whole
(batch, group) units that the oracle recomputes from sliced inputs (the op
is independent across batch entries and across groups)."""
import numpy as np
import pytest

from oracle import ssd_bwd_ref, ssd_fwd_ref
from ssd_chunked_scan_gb300.inputs import WORKLOADS, make_inputs

from gpu_common import compare, run_gpu

pytestmark = pytest.mark.gpu

SMALL = [
    # B, L, G, H, dk, dv, chunk, la_mu, with_h0
    (2, 1, 1, 1, 16, 16, 64, 0.0, True),
    (2, 63, 2, 4, 48, 40, 64, 0.0, True),
    (1, 65, 1, 2, 128, 128, 64, 0.0, True),
    (2, 100, 2, 4, 32, 64, 32, 0.0, False),
    (1, 200, 1, 3, 64, 32, 16, -3.0, True),
    (2, 300, 2, 8, 128, 128, 64, -3.0, True),
    (1, 129, 1, 1, 128, 64, 64, 0.0, True),
    (3, 77, 3, 3, 8, 8, 64, 0.0, True),
    # one feature count a multiple of 32 and the other not (the tensor-core
    # path's tile loads take one box per tile for the first, one per 32-feature
    # block for the second), and three 32-feature blocks
    (1, 150, 1, 2, 128, 40, 64, 0.0, True),
    (2, 90, 1, 2, 40, 96, 64, -3.0, True),
]
SIMT_ONLY = [
    (2, 50, 1, 2, 5, 3, 16, 0.0, True),
    (1, 40, 2, 2, 1, 1, 32, 0.0, True),
    (1, 90, 1, 1, 100, 70, 64, 0.0, True),
]


def _supported(path, dk, dv, chunk):
    if path == "simt":
        return chunk in (16, 32, 64) and dk <= 128 and dv <= 128
    return chunk == 64 and dk % 8 == 0 and dv % 8 == 0 and dk <= 128 and dv <= 128


def _paths():
    return ["simt", "tc"]


@pytest.mark.parametrize("path", _paths())
@pytest.mark.parametrize("case", SMALL + SIMT_ONLY, ids=lambda c: "B{}L{}G{}H{}dk{}dv{}c{}mu{}h{}".format(*c))
def test_small_parity(path, case):
    B, L, G, H, dk, dv, chunk, mu, with_h0 = case
    if not _supported(path, dk, dv, chunk):
        pytest.skip("shape not taken by this path")
    q, k, v, la, h0, dout = make_inputs(B, L, G, H, dk, dv, seed=hash(case) % 10000, la_mu=mu)
    if not with_h0:
        h0 = None
    out, g = run_gpu(path, q, k, v, la, h0, dout, chunk)
    ref = ssd_fwd_ref(q, k, v, la, h0)
    rg = ssd_bwd_ref(q, k, v, la, h0, dout)
    if h0 is None:
        assert g["dh0"] is not None
    compare(path, out, g, ref, rg, label=str(case))


@pytest.mark.parametrize("path", _paths())
def test_forget_everything_decay(path):
    # log_alpha = -1e4 (finite stand-in for -inf): out_t = (q_t.k_t) v_t
    B, L, G, H, dk, dv = 2, 130, 2, 4, 32, 16
    q, k, v, la, h0, dout = make_inputs(B, L, G, H, dk, dv, seed=77)
    la = np.full_like(la, -1e4)
    out, g = run_gpu(path, q, k, v, la, h0, dout, 64)
    rep = np.repeat
    qk = np.einsum("blgd,blgd->blg", q.astype(np.float64), k.astype(np.float64))
    want = rep(qk, H // G, axis=2)[..., None] * v
    compare(path, out, None, want, None, "forget")
    compare(path, out, g, ssd_fwd_ref(q, k, v, la, h0), ssd_bwd_ref(q, k, v, la, h0, dout), "forget")


@pytest.mark.parametrize("path", _paths())
def test_zero_cotangent_and_empty(path):
    import torch
    from ssd_chunked_scan_gb300 import ssd
    q, k, v, la, h0, dout = make_inputs(1, 70, 1, 2, 16, 8, seed=5)
    _, g = run_gpu(path, q, k, v, la, h0, np.zeros_like(dout), 64)
    for n, x in g.items():
        assert not np.any(x), n
    ssd.ssd_set_path(ssd.SSD_PATH_SIMT if path == "simt" else ssd.SSD_PATH_TC)
    e = torch.zeros((2, 0, 1, 16), device="cuda")
    ev = torch.zeros((2, 0, 2, 8), device="cuda")
    out = ssd.ssd_fwd(e, e, ev, torch.zeros((2, 0, 2), device="cuda"), None, chunk=64)
    assert out.shape == (2, 0, 2, 8)
    gg = ssd.ssd_bwd(e, e, ev, torch.zeros((2, 0, 2), device="cuda"), None, ev, chunk=64)
    torch.cuda.synchronize()
    assert torch.count_nonzero(gg["dh0"]).item() == 0


def _unit(x, b, sl):
    return np.ascontiguousarray(x[b:b + 1, :, sl])


@pytest.mark.parametrize("path", _paths())
@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_workload_parity(path, w):
    """Full-size benchmark workload; sampled (batch, group) units vs the oracle."""
    if not _supported(path, w.dk, w.dv, w.chunk):
        pytest.skip("shape not taken by this path")
    from ssd_chunked_scan_gb300.inputs import workload_inputs
    q, k, v, la, h0, dout = workload_inputs(w)
    out, g = run_gpu(path, q, k, v, la, h0, dout, w.chunk)
    hpg = w.H // w.G
    # the first, a middle and the last (batch, group) unit
    units = sorted({(0, 0), (w.B // 2, w.G // 2), (w.B - 1, w.G - 1)})
    for b, gi in units:
        gs, hs = slice(gi, gi + 1), slice(gi * hpg, (gi + 1) * hpg)
        uq, uk = _unit(q, b, gs), _unit(k, b, gs)
        uv, ula, udo = _unit(v, b, hs), _unit(la, b, hs), _unit(dout, b, hs)
        uh0 = np.ascontiguousarray(h0[b:b + 1, hs])
        ref = ssd_fwd_ref(uq, uk, uv, ula, uh0)
        rg = ssd_bwd_ref(uq, uk, uv, ula, uh0, udo)
        mine = {"dq": _unit(g["dq"], b, gs), "dk": _unit(g["dk"], b, gs),
                "dv": _unit(g["dv"], b, hs), "dlog_alpha": _unit(g["dlog_alpha"], b, hs),
                "dh0": np.ascontiguousarray(g["dh0"][b:b + 1, hs])}
        compare(path, _unit(out, b, hs), mine, ref, rg, label=f"{w.name} unit b{b} g{gi}")
