"""Pins of the float64 Mamba-1 selective-scan oracle against things other
than itself: directly summed unrolled terms, the SSD oracle (the selective
scan with A constant over the state index is an SSD scan), closed forms of
special cases, central finite differences of every gradient, and the
linearity identities of y in x, B, C and D."""
import math

import numpy as np
import pytest

from conftest import rel_err
from oracle import mamba_bwd_ref, mamba_fwd_ref, ssd_bwd_ref, ssd_fwd_ref
from ssd_chunked_scan_gb300.inputs import make_mamba_inputs


def _f64(*xs):
    return [None if x is None else np.asarray(x, np.float64) for x in xs]


def test_matches_unrolled_sums():
    x, dt, A, Bm, Cm, Dk, _ = _f64(*make_mamba_inputs(2, 17, 3, 4, seed=1))
    dt = dt * 20  # make decays matter over a short sequence
    y = mamba_fwd_ref(x, dt, A, Bm, Cm, Dk)
    B, L, D = x.shape
    N = A.shape[1]
    want = np.zeros_like(y)
    for b in range(B):
        for d in range(D):
            for t in range(L):
                acc = 0.0
                for s in range(t + 1):
                    for n in range(N):
                        e = 0.0
                        for r in range(s + 1, t + 1):
                            e += dt[b, r, d] * A[d, n]
                        acc += Cm[b, t, n] * math.exp(e) * dt[b, s, d] * Bm[b, s, n] * x[b, s, d]
                want[b, t, d] = acc + Dk[d] * x[b, t, d]
    assert rel_err(y, want) < 1e-12


def test_constant_decay_over_state_is_an_ssd_scan():
    # A[d, n] = a_d for every n: h_t = exp(delta_t a_d) h_{t-1} + B_t (delta_t x_t),
    # i.e. the SSD scan with one head per channel, q = C, k = B, v = delta x,
    # log_alpha = delta a_d (G = 1, dk = N, dv = 1)
    x, dt, A, Bm, Cm, Dk, dy = _f64(*make_mamba_inputs(2, 150, 5, 6, seed=2))
    dt = dt * 5
    A = np.repeat(A[:, :1], A.shape[1], axis=1)
    y = mamba_fwd_ref(x, dt, A, Bm, Cm, Dk)
    q, k = Cm[:, :, None, :], Bm[:, :, None, :]
    v = (dt * x)[..., None]
    la = dt * A[None, None, :, 0]
    out = ssd_fwd_ref(q, k, v, la)
    assert rel_err(y, out[..., 0] + Dk * x) < 1e-12
    g = mamba_bwd_ref(x, dt, A, Bm, Cm, Dk, dy)
    gs = ssd_bwd_ref(q, k, v, la, None, dy[..., None])
    assert rel_err(g["dC"], gs["dq"][:, :, 0]) < 1e-12
    assert rel_err(g["dB"], gs["dk"][:, :, 0]) < 1e-12
    assert rel_err(g["dx"], gs["dv"][..., 0] * dt + Dk * dy) < 1e-12
    assert rel_err(g["ddelta"], gs["dv"][..., 0] * x + gs["dlog_alpha"] * A[:, 0]) < 1e-12
    # the SSD scan ties the N entries of A[d, :]; their sum is its gradient
    assert rel_err(g["dA"].sum(1), np.einsum("bld,bld->d", gs["dlog_alpha"], dt)) < 1e-12


def test_special_cases():
    x, dt, A, Bm, Cm, Dk, _ = _f64(*make_mamba_inputs(2, 40, 3, 4, seed=3))
    # A = 0: the state is a plain running sum
    h = np.cumsum((dt * x)[..., None] * Bm[:, :, None, :], axis=1)
    want = np.einsum("bldn,bln->bld", h, Cm) + Dk * x
    assert rel_err(mamba_fwd_ref(x, dt, np.zeros_like(A), Bm, Cm, Dk), want) < 1e-12
    # A very negative: no memory, h_t = delta_t B_t x_t
    want = dt * x * np.einsum("bln,bln->bl", Bm, Cm)[..., None] + Dk * x
    assert rel_err(mamba_fwd_ref(x, dt, A * 1e6, Bm, Cm, Dk), want) < 1e-12
    # B = 0 leaves the skip term only; D absent drops it
    assert rel_err(mamba_fwd_ref(x, dt, A, 0 * Bm, Cm, Dk), Dk * x) < 1e-15
    y0 = mamba_fwd_ref(x, dt, A, Bm, Cm, None)
    assert rel_err(mamba_fwd_ref(x, dt, A, Bm, Cm, Dk) - Dk * x, y0) < 1e-12


def test_grads_match_central_differences():
    x, dt, A, Bm, Cm, Dk, dy = _f64(*make_mamba_inputs(2, 11, 3, 4, seed=4))
    dt = dt * 10
    g = mamba_bwd_ref(x, dt, A, Bm, Cm, Dk, dy)
    loss = lambda: float(np.sum(mamba_fwd_ref(x, dt, A, Bm, Cm, Dk) * dy))
    eps = 1e-6
    rng = np.random.default_rng(0)
    for name, arr in {"dx": x, "ddelta": dt, "dA": A, "dB": Bm, "dC": Cm, "dD": Dk}.items():
        flat = arr.reshape(-1)
        for i in rng.choice(flat.size, size=min(flat.size, 12), replace=False):
            old = flat[i]
            flat[i] = old + eps
            lp = loss()
            flat[i] = old - eps
            lm = loss()
            flat[i] = old
            fd = (lp - lm) / (2 * eps)
            an = g[name].reshape(-1)[i]
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, i, fd, an)


def test_linearity_identities():
    # y - D x is linear in x, in B and in C separately; D x is linear in D
    x, dt, A, Bm, Cm, Dk, dy = _f64(*make_mamba_inputs(2, 300, 4, 16, seed=5))
    y = mamba_fwd_ref(x, dt, A, Bm, Cm, Dk)
    g = mamba_bwd_ref(x, dt, A, Bm, Cm, Dk, dy)
    scan = float(np.sum(dy * (y - Dk * x)))
    skip = float(np.sum(dy * Dk * x))
    tol = 1e-11 * (abs(scan) + abs(skip) + 1)
    assert abs(np.sum(x * g["dx"]) - (scan + skip)) < tol
    assert abs(np.sum(Bm * g["dB"]) - scan) < tol
    assert abs(np.sum(Cm * g["dC"]) - scan) < tol
    assert abs(np.sum(Dk * g["dD"]) - skip) < tol


@pytest.mark.parametrize("L", [63, 64, 65, 129])
def test_checkpoint_boundaries(L):
    # the backward recomputes states from checkpoints every 64 steps: grads of
    # a sequence and of the same sequence with an inert tail must agree
    x, dt, A, Bm, Cm, Dk, dy = _f64(*make_mamba_inputs(1, L + 3, 2, 4, seed=6))
    dy[:, L:] = 0.0
    x[:, L:] = 0.0  # the tail contributes nothing and receives no gradient flow back
    g_full = mamba_bwd_ref(x, dt, A, Bm, Cm, Dk, dy)
    g_cut = mamba_bwd_ref(x[:, :L].copy(), dt[:, :L].copy(), A, Bm[:, :L].copy(),
                          Cm[:, :L].copy(), Dk, dy[:, :L].copy())
    for n in ("dx", "ddelta", "dB", "dC"):
        assert rel_err(g_full[n][:, :L], g_cut[n]) < 1e-12, n
    for n in ("dA", "dD"):
        assert rel_err(g_full[n], g_cut[n]) < 1e-12, n
