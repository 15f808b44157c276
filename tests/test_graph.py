"""The library's calls under CUDA graph capture: a forward + backward step
(tensor-core path, backward passes on the library's side stream, workspace
from the stream-ordered pool) captured once into a graph and replayed gives
the eager results, on new inputs copied into the captured buffers too."""
import numpy as np
import pytest

from ssd_chunked_scan_gb300.inputs import make_inputs

from gpu_common import to_dev

pytestmark = pytest.mark.gpu

DIMS = (2, 300, 2, 8, 128, 128)  # B, L, G, H, dk, dv


def _eager(ssd, torch, dev_in):
    out = ssd.ssd_fwd(*dev_in[:5], chunk=64)
    g = ssd.ssd_bwd(*dev_in, chunk=64)
    torch.cuda.synchronize()
    return out.cpu().numpy(), {n: t.cpu().numpy() for n, t in g.items() if t is not None}


def _close(a, b, exact):
    if exact:
        return np.array_equal(a, b)
    return np.abs(a - b).max() <= 1e-6 * np.abs(b).max()


def test_fwd_bwd_step_replays_from_a_graph():
    import torch
    from ssd_chunked_scan_gb300 import ssd
    ssd.ssd_set_path(ssd.SSD_PATH_TC)
    B, L, G, H, dk, dv = DIMS
    bufs = [to_dev(x) for x in make_inputs(B, L, G, H, dk, dv, seed=11, la_mu=-3.0)]
    out = torch.empty((B, L, H, dv), device="cuda")
    grads = {"dq": torch.empty((B, L, G, dk), device="cuda"),
             "dk": torch.empty((B, L, G, dk), device="cuda"),
             "dv": torch.empty((B, L, H, dv), device="cuda"),
             "dlog_alpha": torch.empty((B, L, H), device="cuda"),
             "dh0": torch.empty((B, H, dk, dv), device="cuda")}

    def step():
        ssd.ssd_fwd(*bufs[:5], chunk=64, out=out)
        ssd.ssd_bwd(*bufs, chunk=64, grads=grads)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside capture (creates the library's side streams)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()

    for seed in (11, 12):
        new = make_inputs(B, L, G, H, dk, dv, seed=seed, la_mu=-3.0)
        for d, x in zip(bufs, new):
            d.copy_(torch.from_numpy(x))
        graph.replay()
        torch.cuda.synchronize()
        assert ssd.ssd_last_device_error() == 0
        got_out = out.cpu().numpy()
        got = {n: t.cpu().numpy() for n, t in grads.items()}
        ref_out, ref = _eager(ssd, torch, [to_dev(x) for x in new])
        assert _close(got_out, ref_out, exact=True)
        for n in ("dv", "dlog_alpha", "dh0"):
            assert _close(got[n], ref[n], exact=True), n
        for n in ("dq", "dk"):  # summed over a group's heads by atomic adds
            assert _close(got[n], ref[n], exact=False), n
