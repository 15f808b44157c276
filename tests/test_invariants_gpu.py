"""Identities of the exact op checked on the GPU's own outputs at the full
benchmark sizes, for every (batch, head) or (batch, group) unit (the parity
tests compare sampled units with the oracle; these cover all of them).

With loss <dout, out>, out is linear in q, jointly linear in (v, h0), and
depends on k and v only through k_s v_s^T, so in exact arithmetic:
  per (b, g):  sum q . dq                 = sum over the group's heads of <dout_h, out_h>
  per (b, h):  <dv_h, v_h> + <dh0_h, h0_h> = <dout_h, out_h>
  overall:     <dk, k>                     = <dv, v>
  per (b, h):  dlog_alpha[b, 0, h]         = <dh0_h, h0_h>      (the first decay multiplies h0)
Each computed residual is bounded by the path's element tolerance (rel_err
bar, relative to the largest element of each tensor) times the sum of the
absolute terms it multiplies, a bound that holds whenever every element is
within the bar; the dot products are formed in float64 on the host."""
import numpy as np
import pytest

from ssd_chunked_scan_gb300.inputs import WORKLOADS

from gpu_common import TOL, run_gpu


def _supported(path, w):
    if path == "simt":
        return w.chunk in (16, 32, 64) and w.dk <= 128 and w.dv <= 128
    return w.chunk == 64 and w.dk % 8 == 0 and w.dv % 8 == 0 and w.dk <= 128 and w.dv <= 128


def check_identities(q, k, v, h0, dout, out, g, eps):
    """Assert the four identities on one problem's outputs (any precision)
    within their element-tolerance bounds; returns the worst residual / bound."""
    f = lambda x: np.asarray(x, dtype=np.float64)
    q, k, v, h0, dout, out = map(f, (q, k, v, h0, dout, out))
    dq, dk, dv, dla, dh0 = (f(g[n]) for n in ("dq", "dk", "dv", "dlog_alpha", "dh0"))
    B, G, H = q.shape[0], q.shape[2], v.shape[2]
    hpg = H // G
    m_out, m_dq, m_dk, m_dv = (np.abs(x).max() for x in (out, dq, dk, dv))
    m_dh0, m_dla = np.abs(dh0).max(), np.abs(dla).max()

    # <dout_h, out_h> and its absolute-value scale, per (b, h)
    lo = np.einsum("blhd,blhd->bh", dout, out)
    lo_abs = np.einsum("blhd->bh", np.abs(dout))

    # q . dq per (b, g) against the group's heads
    qdq = np.einsum("blgd,blgd->bg", q, dq)
    lo_g = lo.reshape(B, G, hpg).sum(axis=2)
    bound = eps * (m_dq * np.einsum("blgd->bg", np.abs(q))
                   + m_out * lo_abs.reshape(B, G, hpg).sum(axis=2)) + 1e-12
    r1 = (np.abs(qdq - lo_g) / bound).max()
    assert r1 <= 1.0, f"q.dq identity off by {r1:.3g} x its bound"

    # <dv_h, v_h> + <dh0_h, h0_h> = <dout_h, out_h>, per (b, h)
    vdv = np.einsum("blhd,blhd->bh", v, dv)
    hdh = np.einsum("bhij,bhij->bh", h0, dh0)
    bound = eps * (m_dv * np.einsum("blhd->bh", np.abs(v)) + m_dh0 * np.einsum("bhij->bh", np.abs(h0))
                   + m_out * lo_abs) + 1e-12
    r3 = (np.abs(vdv + hdh - lo) / bound).max()
    assert r3 <= 1.0, f"(v, h0) identity off by {r3:.3g} x its bound"

    # <dk, k> = <dv, v>, over the whole problem
    kdk = float(np.sum(k * dk))
    bound = eps * (m_dk * np.abs(k).sum() + m_dv * np.abs(v).sum()) + 1e-12
    r2 = abs(kdk - vdv.sum()) / bound
    assert r2 <= 1.0, f"<dk,k> = <dv,v> off by {r2:.3g} x its bound"

    # dlog_alpha at t = 0 is <dh0, h0> per (b, h)
    bound = eps * (m_dla + m_dh0 * np.einsum("bhij->bh", np.abs(h0))) + 1e-12
    r4 = (np.abs(dla[:, 0, :] - hdh) / bound).max()
    assert r4 <= 1.0, f"dla[:, 0] identity off by {r4:.3g} x its bound"
    return max(r1, r2, r3, r4)


@pytest.mark.gpu
@pytest.mark.parametrize("path", ["simt", "tc"])
@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_identities_on_every_unit(path, w):
    if not _supported(path, w):
        pytest.skip("shape not taken by this path")
    from ssd_chunked_scan_gb300.inputs import workload_inputs
    q, k, v, la, h0, dout = workload_inputs(w)
    out, g = run_gpu(path, q, k, v, la, h0, dout, w.chunk)
    check_identities(q, k, v, h0, dout, out, g, TOL[path])


def test_checker_on_oracle_outputs_and_on_planted_errors():
    """The checker itself, on the CPU: the float64 oracle's outputs satisfy
    every identity far inside the bounds; outputs perturbed elementwise within
    the bar still pass; a unit whose dv is off by more than the bar fails."""
    from oracle import ssd_bwd_ref, ssd_fwd_ref
    from ssd_chunked_scan_gb300.inputs import make_inputs
    q, k, v, la, h0, dout = make_inputs(2, 130, 2, 4, 16, 8, seed=17)
    out = ssd_fwd_ref(q, k, v, la, h0)
    g = ssd_bwd_ref(q, k, v, la, h0, dout)
    assert check_identities(q, k, v, h0, dout, out, g, 2e-5) < 1e-3
    rng = np.random.default_rng(3)
    eps = 1e-3
    noisy = lambda x: x + eps * np.abs(x).max() * rng.uniform(-1, 1, x.shape)
    check_identities(q, k, v, h0, dout, noisy(out), {n: noisy(t) for n, t in g.items()}, eps)
    bad = dict(g)
    bad["dv"] = g["dv"].copy()
    bad["dv"][1, :, 2, :] *= 1.05  # one (batch, head) unit 5 % off
    with pytest.raises(AssertionError):
        check_identities(q, k, v, h0, dout, out, bad, 2e-5)
