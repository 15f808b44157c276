"""The differentiable entry point ssd_scan: its forward and the gradients
autograd returns are the library's ssd_fwd_ex / ssd_bwd_ex results (with
save_states, ssd_fwd_save / ssd_bwd_saved) on the same inputs, the gradients agree with the float64 oracle, and tensors
that are not on a CUDA device are refused (there is no CPU path)."""
import os

import numpy as np
import pytest

from ssd_chunked_scan_gb300.inputs import make_inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "ssd_chunked_scan_gb300", "_lib", "libssd.so")


def _lib_built():
    if not os.path.exists(LIB):
        from ssd_chunked_scan_gb300.build import build_lib
        build_lib()


def test_cpu_tensors_are_refused():
    _lib_built()
    import torch
    from ssd_chunked_scan_gb300.autograd import ssd_scan
    q, k, v, la, h0, _ = (torch.from_numpy(x) for x in make_inputs(1, 8, 1, 1, 8, 8, seed=3))
    with pytest.raises(ValueError, match="CUDA"):
        ssd_scan(q, k, v, la, h0)


def _same(a, b, exact):
    a, b = a.detach().cpu().numpy(), b.detach().cpu().numpy()
    if exact:
        return np.array_equal(a, b)
    return np.abs(a - b).max() <= 1e-6 * np.abs(b).max()


@pytest.mark.gpu
@pytest.mark.parametrize("final", [False, True])
@pytest.mark.parametrize("with_h0", [True, False])
@pytest.mark.parametrize("save_states", [False, True])
def test_autograd_matches_library_calls(final, with_h0, save_states):
    import torch
    from oracle import ssd_bwd_ref
    from ssd_chunked_scan_gb300 import ssd
    from ssd_chunked_scan_gb300.autograd import ssd_scan
    ssd.ssd_set_path(ssd.SSD_PATH_TC)
    B, L, G, H, dk, dv = 2, 200, 2, 4, 64, 64
    host = make_inputs(B, L, G, H, dk, dv, seed=21, la_mu=-1.0)
    q, k, v, la, h0, dout = (torch.from_numpy(x).cuda() for x in host)
    if not with_h0:
        h0 = None
    dhT = torch.from_numpy(np.random.default_rng(5).standard_normal((B, H, dk, dv)).astype(np.float32)).cuda()
    leaves = [t.clone().requires_grad_(True) for t in (q, k, v, la)]
    h0_leaf = h0.clone().requires_grad_(True) if h0 is not None else None
    res = ssd_scan(*leaves, h0_leaf, chunk=64, return_final_state=final, save_states=save_states)
    if final:
        out, hT = res
        loss = (out * dout).sum() + (hT * dhT).sum()
    else:
        out = res
        loss = (out * dout).sum()
    loss.backward()
    torch.cuda.synchronize()

    if save_states:
        ref_out, ref_hT, saved = ssd.ssd_fwd_save(q, k, v, la, h0, chunk=64)
        g = ssd.ssd_bwd_saved(q, k, v, la, h0, dout, dhT if final else None, ref_hT, saved, chunk=64,
                              want_dh0=h0 is not None)
    else:
        ref_out, ref_hT = ssd.ssd_fwd_ex(q, k, v, la, h0, chunk=64)
        g = ssd.ssd_bwd_ex(q, k, v, la, h0, dout, dhT if final else None, chunk=64,
                           want_dh0=h0 is not None)
    if final:
        assert _same(hT, ref_hT, exact=True)
    torch.cuda.synchronize()
    assert _same(out, ref_out, exact=True)
    grads = dict(zip(("dq", "dk", "dv", "dlog_alpha"), (t.grad for t in leaves)))
    if h0 is not None:
        grads["dh0"] = h0_leaf.grad
    for n in ("dv", "dlog_alpha", "dh0"):
        if n in grads:
            assert _same(grads[n], g[n], exact=True), n
    for n in ("dq", "dk"):  # a group's heads are summed by atomic adds
        assert _same(grads[n], g[n], exact=False), n

    h = [x.astype(np.float64) for x in host]
    ref = ssd_bwd_ref(h[0], h[1], h[2], h[3], h[4] if with_h0 else None, h[5],
                      dhT=dhT.cpu().numpy() if final else None)
    for n, t in grads.items():
        x = t.cpu().numpy()
        err = np.abs(x - ref[n]).max() / np.abs(ref[n]).max()
        assert err <= 3e-3, (n, err)
