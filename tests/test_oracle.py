"""Pins of the float64 oracle against facts fixed independently of it.

Each test would fail on a plausible slip in the oracle: a dropped decay, the
decay applied after the k v^T add, an exclusive instead of inclusive state,
the wrong head->group map, a transposed state, a missing h0 term, or a wrong
adjoint.  CPU only.
"""
import math

import numpy as np
import pytest

from oracle import ssd_bwd_ref, ssd_fwd_ref
from oracle.brute import ssd_fwd_brute
from ssd_chunked_scan_gb300.inputs import make_inputs

from conftest import rel_err


def _case(B, L, G, H, dk, dv, seed, la_mu=0.0):
    return make_inputs(B, L, G, H, dk, dv, seed, la_mu)


@pytest.mark.parametrize("shape", [(1, 1, 1, 1, 3, 2), (2, 9, 1, 1, 4, 3),
                                   (2, 17, 2, 4, 5, 3), (1, 33, 3, 6, 2, 7)])
def test_fwd_matches_unrolled_sums(shape):
    B, L, G, H, dk, dv = shape
    q, k, v, la, h0, _ = _case(B, L, G, H, dk, dv, seed=sum(shape))
    la = la * 0.3  # keep several steps of memory alive
    ref = ssd_fwd_brute(q, k, v, la, h0)
    out = ssd_fwd_ref(q, k, v, la, h0)
    assert rel_err(out, ref) < 1e-12


def test_zero_decay_is_causal_linear_attention():
    # log_alpha = 0 and h0 = 0: out = tril(Q K^T) V, a plain matmul identity
    B, L, G, H, dk, dv = 2, 40, 1, 1, 6, 5
    q, k, v, la, _, _ = _case(B, L, G, H, dk, dv, seed=3)
    la = np.zeros_like(la)
    out = ssd_fwd_ref(q, k, v, la, None)
    for b in range(B):
        Q = q[b, :, 0].astype(np.float64)
        K = k[b, :, 0].astype(np.float64)
        V = v[b, :, 0].astype(np.float64)
        want = np.tril(Q @ K.T) @ V
        np.testing.assert_allclose(out[b, :, 0], want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("la_value", [-np.inf, -1e4])
def test_infinite_decay_keeps_only_current_token(la_value):
    B, L, G, H, dk, dv = 2, 12, 2, 4, 5, 3
    q, k, v, la, h0, _ = _case(B, L, G, H, dk, dv, seed=4)
    la = np.full_like(la, la_value)
    out = ssd_fwd_ref(q, k, v, la, h0)
    for h in range(H):
        g = h // (H // G)
        qk = np.einsum("bld,bld->bl", q[:, :, g].astype(np.float64), k[:, :, g].astype(np.float64))
        np.testing.assert_allclose(out[:, :, h], qk[..., None] * v[:, :, h], rtol=1e-12, atol=1e-14)


def test_group_map_is_contiguous_split():
    # G=2, H=4: heads 0,1 read group 0 and heads 2,3 read group 1; each head
    # alone must equal a one-group one-head problem on its own slices.
    B, L, G, H, dk, dv = 2, 20, 2, 4, 4, 3
    q, k, v, la, h0, _ = _case(B, L, G, H, dk, dv, seed=5)
    out = ssd_fwd_ref(q, k, v, la, h0)
    for h in range(H):
        g = h // 2
        single = ssd_fwd_ref(q[:, :, g:g + 1], k[:, :, g:g + 1], v[:, :, h:h + 1],
                             la[:, :, h:h + 1], h0[:, h:h + 1])
        np.testing.assert_allclose(out[:, :, h:h + 1], single, rtol=0, atol=0)


def test_single_step_closed_form():
    # L=1: out = (exp(la) h0 + k v^T)^T q, written out by hand
    q, k, v, la, h0, _ = (x.astype(np.float64) for x in _case(1, 1, 1, 1, 3, 2, seed=6))
    a = math.exp(float(la[0, 0, 0]))
    S = a * h0[0, 0] + np.outer(k[0, 0, 0], v[0, 0, 0])
    np.testing.assert_allclose(ssd_fwd_ref(q, k, v, la, h0)[0, 0, 0], S.T @ q[0, 0, 0], rtol=1e-14)


def _loss(q, k, v, la, h0, dout):
    return float(np.sum(ssd_fwd_ref(q, k, v, la, h0) * dout))


def test_grads_match_central_differences():
    B, L, G, H, dk, dv = 2, 9, 2, 4, 5, 3
    q, k, v, la, h0, dout = (x.astype(np.float64) for x in _case(B, L, G, H, dk, dv, seed=7))
    g = ssd_bwd_ref(q, k, v, la, h0, dout)
    eps = 1e-6
    args = {"dq": q, "dk": k, "dv": v, "dlog_alpha": la, "dh0": h0}
    rng = np.random.default_rng(0)
    for name, x in args.items():
        flat = x.reshape(-1)
        idx = rng.choice(flat.size, size=min(flat.size, 25), replace=False)
        for i in idx:
            old = flat[i]
            flat[i] = old + eps
            lp = _loss(q, k, v, la, h0, dout)
            flat[i] = old - eps
            lm = _loss(q, k, v, la, h0, dout)
            flat[i] = old
            fd = (lp - lm) / (2 * eps)
            an = g[name].reshape(-1)[i]
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, i, fd, an)


def test_euler_identities():
    # out is homogeneous of degree 1 in q, in (v, h0) jointly, and invariant
    # under k -> c k, v -> v / c; la_0 only scales the h0 term.
    B, L, G, H, dk, dv = 2, 150, 2, 4, 6, 5
    q, k, v, la, h0, dout = _case(B, L, G, H, dk, dv, seed=8)
    out = ssd_fwd_ref(q, k, v, la, h0)
    g = ssd_bwd_ref(q, k, v, la, h0, dout)
    f = lambda x: np.asarray(x, np.float64)
    loss = float(np.sum(out * f(dout)))
    scale = float(np.sum(np.abs(out * f(dout))))
    assert abs(float(np.sum(f(q) * g["dq"])) - loss) < 1e-12 * scale
    assert abs(float(np.sum(f(k) * g["dk"])) - float(np.sum(f(v) * g["dv"]))) < 1e-12 * scale
    assert abs(float(np.sum(f(v) * g["dv"])) + float(np.sum(f(h0) * g["dh0"])) - loss) < 1e-12 * scale
    dla0 = np.einsum("bhij,bhij->bh", f(h0), g["dh0"])
    np.testing.assert_allclose(g["dlog_alpha"][:, 0, :], dla0, rtol=1e-10, atol=1e-14)


def test_dcs_reverse_cumsum_identity():
    # dla_t = sum_{t'>=t} (q_t'.dq_h[t'] - k_t'.dk_h[t']) per head -- the identity a
    # chunked backward uses; the oracle's dla is the direct adjoint.
    B, L, G, H, dk, dv = 2, 130, 2, 4, 6, 5
    q, k, v, la, h0, dout = _case(B, L, G, H, dk, dv, seed=9)
    g = ssd_bwd_ref(q, k, v, la, h0, dout, per_head=True)
    hpg = H // G
    qh = np.repeat(q.astype(np.float64), hpg, axis=2)
    kh = np.repeat(k.astype(np.float64), hpg, axis=2)
    dcs = np.sum(qh * g["dq_heads"], -1) - np.sum(kh * g["dk_heads"], -1)
    dla = np.flip(np.cumsum(np.flip(dcs, 1), 1), 1)
    assert rel_err(dla, g["dlog_alpha"]) < 1e-10
    # and the group sums of the per-head gradients are the returned dq / dk
    np.testing.assert_allclose(g["dq"], g["dq_heads"].reshape(B, L, G, hpg, dk).sum(3), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(g["dk"], g["dk_heads"].reshape(B, L, G, hpg, dk).sum(3), rtol=1e-13, atol=1e-15)


def test_zero_cotangent_gives_zero_grads():
    q, k, v, la, h0, dout = _case(1, 70, 1, 2, 4, 3, seed=10)
    g = ssd_bwd_ref(q, k, v, la, h0, np.zeros_like(dout))
    for x in g.values():
        assert not np.any(x)


def test_empty_sequence():
    q, k, v, la, h0, dout = _case(2, 0, 1, 2, 4, 3, seed=11)
    assert ssd_fwd_ref(q, k, v, la, h0).shape == (2, 0, 2, 3)
    g = ssd_bwd_ref(q, k, v, la, h0, dout)
    assert not np.any(g["dh0"])


def test_checkpoint_boundaries():
    # the backward recomputes states in 64-step segments; lengths around the
    # segment size must agree with finite differences of the forward at the
    # last and first steps
    for L in (63, 64, 65, 129):
        q, k, v, la, h0, dout = (x.astype(np.float64) for x in _case(1, L, 1, 1, 3, 2, seed=L))
        la *= 0.05
        g = ssd_bwd_ref(q, k, v, la, h0, dout)
        for t in (0, L // 2, L - 1):
            old = la[0, t, 0]
            la[0, t, 0] = old + 1e-6
            lp = _loss(q, k, v, la, h0, dout)
            la[0, t, 0] = old - 1e-6
            lm = _loss(q, k, v, la, h0, dout)
            la[0, t, 0] = old
            fd = (lp - lm) / 2e-6
            assert abs(fd - g["dlog_alpha"][0, t, 0]) <= 1e-6 * max(1.0, abs(fd))


# ---- final state hT and its cotangent dhT ---------------------------------

def test_final_state_matches_unrolled_sums():
    from oracle.brute import ssd_final_state_brute
    q, k, v, la, h0, _ = _case(2, 23, 2, 4, 5, 3, seed=31)
    la = la * 0.3
    _, hT = ssd_fwd_ref(q, k, v, la, h0, return_final_state=True)
    assert rel_err(hT, ssd_final_state_brute(k, v, la, h0)) < 1e-12


def test_sequence_split_carries_the_state():
    # running [0, L1) then [L1, L) from the first part's final state equals
    # one run over [0, L)
    q, k, v, la, h0, _ = _case(2, 150, 2, 4, 6, 5, seed=32)
    out, hT = ssd_fwd_ref(q, k, v, la, h0, return_final_state=True)
    L1 = 61
    o1, h1 = ssd_fwd_ref(q[:, :L1], k[:, :L1], v[:, :L1], la[:, :L1], h0, return_final_state=True)
    o2, h2 = ssd_fwd_ref(q[:, L1:], k[:, L1:], v[:, L1:], la[:, L1:], h1, return_final_state=True)
    np.testing.assert_allclose(np.concatenate([o1, o2], 1), out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h2, hT, rtol=1e-12, atol=1e-13)


def _loss_T(q, k, v, la, h0, dout, dhT):
    out, hT = ssd_fwd_ref(q, k, v, la, h0, return_final_state=True)
    return float(np.sum(out * dout) + np.sum(hT * dhT))


def test_grads_with_final_state_cotangent_match_central_differences():
    B, L, G, H, dk, dv = 2, 9, 2, 4, 4, 3
    q, k, v, la, h0, dout = (x.astype(np.float64) for x in _case(B, L, G, H, dk, dv, seed=33))
    dhT = np.random.default_rng(5).standard_normal((B, H, dk, dv))
    g = ssd_bwd_ref(q, k, v, la, h0, dout, dhT=dhT)
    eps = 1e-6
    rng = np.random.default_rng(1)
    for name, x in {"dq": q, "dk": k, "dv": v, "dlog_alpha": la, "dh0": h0}.items():
        flat = x.reshape(-1)
        for i in rng.choice(flat.size, size=min(flat.size, 20), replace=False):
            old = flat[i]
            flat[i] = old + eps
            lp = _loss_T(q, k, v, la, h0, dout, dhT)
            flat[i] = old - eps
            lm = _loss_T(q, k, v, la, h0, dout, dhT)
            flat[i] = old
            fd = (lp - lm) / (2 * eps)
            an = g[name].reshape(-1)[i]
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, i, fd, an)


def test_euler_identity_with_final_state():
    # out and hT are both homogeneous of degree 1 in (v, h0) jointly
    q, k, v, la, h0, dout = _case(2, 140, 2, 4, 6, 5, seed=34)
    dhT = np.random.default_rng(6).standard_normal(h0.shape)
    out, hT = ssd_fwd_ref(q, k, v, la, h0, return_final_state=True)
    g = ssd_bwd_ref(q, k, v, la, h0, dout, dhT=dhT)
    f = lambda x: np.asarray(x, np.float64)
    total = float(np.sum(out * f(dout)) + np.sum(hT * dhT))
    lhs = float(np.sum(f(v) * g["dv"]) + np.sum(f(h0) * g["dh0"]))
    assert abs(lhs - total) < 1e-11 * (abs(total) + 1.0)
    # and the dcs identity picks up the final-state term <dhT, hT>
    gh = ssd_bwd_ref(q, k, v, la, h0, dout, per_head=True, dhT=dhT)
    qh = np.repeat(q.astype(np.float64), 2, axis=2)
    kh = np.repeat(k.astype(np.float64), 2, axis=2)
    dcs = np.sum(qh * gh["dq_heads"], -1) - np.sum(kh * gh["dk_heads"], -1)
    carry = np.einsum("bhij,bhij->bh", dhT, hT)
    dla = np.flip(np.cumsum(np.flip(dcs, 1), 1), 1) + carry[:, None, :]
    assert rel_err(dla, g["dlog_alpha"]) < 1e-10


def test_empty_sequence_final_state():
    q, k, v, la, h0, dout = _case(2, 0, 1, 2, 4, 3, seed=35)
    _, hT = ssd_fwd_ref(q, k, v, la, h0, return_final_state=True)
    np.testing.assert_array_equal(hT, h0.astype(np.float64))
    dhT = np.ones(h0.shape)
    assert np.array_equal(ssd_bwd_ref(q, k, v, la, h0, dout, dhT=dhT)["dh0"], dhT)


def test_dla_from_output_and_value_gradients():
    # per head, q.dq_h - k.dk_h = out.dout - v.dv (both are <S_t, q dout^T> -
    # <G_t, k v^T>), so dla is also the reverse cumulative sum of
    # out.dout - v.dv plus <dhT, hT>
    q, k, v, la, h0, dout = _case(2, 90, 2, 4, 6, 5, seed=36)
    dhT = np.random.default_rng(7).standard_normal(h0.shape)
    out, hT = ssd_fwd_ref(q, k, v, la, h0, return_final_state=True)
    g = ssd_bwd_ref(q, k, v, la, h0, dout, dhT=dhT)
    e = np.sum(out * dout.astype(np.float64), -1) - np.sum(v.astype(np.float64) * g["dv"], -1)
    carry = np.einsum("bhij,bhij->bh", dhT, hT)
    dla = np.flip(np.cumsum(np.flip(e, 1), 1), 1) + carry[:, None, :]
    assert rel_err(dla, g["dlog_alpha"]) < 1e-10
