"""ctypes front end of the float64 C oracle (``ssd_oracle.c``).

TEST INFRASTRUCTURE ONLY -- the CUDA library is checked against this; it is
never part of the product path.

Definition followed (the op timed by the "kernel_ssd_gpu.json" and
"kernel_ssd_cpu.json" benchmark records, whose ``scan`` implementation is the
step-by-step form of the recurrence):

    S_t = exp(la_t) S_{t-1} + k_t v_t^T,  S_{-1} = h0,   out_t = S_t^T q_t

with head h reading group h // (H // G).  Gradients are the exact adjoint of
the loss <dout, out>.  Inputs are taken as stored (fp32 values widened to
float64 exactly); all arithmetic is float64.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = build_oracle()
        lib = ctypes.CDLL(path)
        d = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.ssd_oracle_fwd.argtypes = [d, d, d, d, d, d, d] + [i64] * 6
        lib.ssd_oracle_fwd.restype = ctypes.c_int
        lib.ssd_oracle_bwd.argtypes = [d] * 14 + [i64] * 6
        lib.ssd_oracle_bwd.restype = ctypes.c_int
        lib.ssd_oracle_num_threads.argtypes = []
        lib.ssd_oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def oracle_threads() -> int:
    """Threads the oracle's OpenMP loops use (1 without OpenMP)."""
    return int(_load().ssd_oracle_num_threads())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _dims(q, v, la):
    B, L, G, dk = q.shape
    H, dv = v.shape[2], v.shape[3]
    assert v.shape[:2] == (B, L) and la.shape == (B, L, H)
    assert H % G == 0, "heads must split evenly over groups"
    return B, L, G, H, dk, dv


def ssd_fwd_ref(q, k, v, log_alpha, h0=None, return_final_state=False):
    """out [B,L,H,dv] (float64) for q,k [B,L,G,dk], v [B,L,H,dv], log_alpha [B,L,H].

    With ``return_final_state`` also returns hT = S_{L-1} [B,H,dk,dv]."""
    q, k, v, la, h0 = map(_f64, (q, k, v, log_alpha, h0))
    B, L, G, H, dk, dv = _dims(q, v, la)
    assert k.shape == q.shape
    if h0 is not None:
        assert h0.shape == (B, H, dk, dv)
    out = np.zeros((B, L, H, dv), np.float64)
    hT = np.zeros((B, H, dk, dv), np.float64) if return_final_state else None
    if hT is not None and L == 0 and h0 is not None:
        hT[...] = h0
    rc = _load().ssd_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(h0), _ptr(out),
                                _ptr(hT) if L > 0 else _ptr(None), B, L, G, H, dk, dv)
    if rc:
        raise RuntimeError(f"oracle fwd failed ({rc})")
    return (out, hT) if return_final_state else out


def ssd_bwd_ref(q, k, v, log_alpha, h0, dout, per_head=False, dhT=None):
    """Gradients of <dout, out> (+ <dhT, hT> when dhT is given): dict with dq,
    dk, dv, dlog_alpha, dh0 (float64).

    With ``per_head=True`` also returns dq_heads / dk_heads [B,L,H,dk], the
    per-head contributions before the sum over the heads of each group.
    """
    q, k, v, la, h0, dout, dhT = map(_f64, (q, k, v, log_alpha, h0, dout, dhT))
    B, L, G, H, dk, dv = _dims(q, v, la)
    assert k.shape == q.shape and dout.shape == v.shape
    r = {
        "dq": np.zeros((B, L, G, dk)), "dk": np.zeros((B, L, G, dk)),
        "dv": np.zeros((B, L, H, dv)), "dlog_alpha": np.zeros((B, L, H)),
        "dh0": np.zeros((B, H, dk, dv)),
    }
    dqh = np.zeros((B, L, H, dk)) if per_head else None
    dkh = np.zeros((B, L, H, dk)) if per_head else None
    if dhT is not None:
        assert dhT.shape == (B, H, dk, dv)
    rc = _load().ssd_oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(h0), _ptr(dout),
                                _ptr(dhT), _ptr(r["dq"]), _ptr(r["dk"]), _ptr(r["dv"]),
                                _ptr(r["dlog_alpha"]), _ptr(r["dh0"]), _ptr(dqh), _ptr(dkh),
                                B, L, G, H, dk, dv)
    if rc:
        raise RuntimeError(f"oracle bwd failed ({rc})")
    if L == 0 and dhT is not None:
        r["dh0"][...] = dhT
    if per_head:
        r["dq_heads"], r["dk_heads"] = dqh, dkh
    return r


# ---- Mamba-1 selective scan ("kernel_mamba_cpu.json" records) --------------

def _load_mamba():
    lib = _load()
    if not getattr(lib, "_mamba_ready", False):
        d = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.mamba_oracle_fwd.argtypes = [d] * 7 + [i64] * 4
        lib.mamba_oracle_fwd.restype = ctypes.c_int
        lib.mamba_oracle_bwd.argtypes = [d] * 13 + [i64] * 4
        lib.mamba_oracle_bwd.restype = ctypes.c_int
        lib._mamba_ready = True
    return lib


def mamba_fwd_ref(x, delta, A, Bm, Cm, Dk=None):
    """float64 y [B,L,D] of the selective scan
    h_t[n] = exp(delta_t A[d,n]) h_{t-1}[n] + delta_t B_t[n] x_t,
    y_t = sum_n C_t[n] h_t[n] + D[d] x_t (h_{-1} = 0)."""
    x, delta, A, Bm, Cm, Dk = map(_f64, (x, delta, A, Bm, Cm, Dk))
    B, L, D = x.shape
    N = A.shape[1]
    y = np.empty((B, L, D))
    rc = _load_mamba().mamba_oracle_fwd(_ptr(x), _ptr(delta), _ptr(A), _ptr(Bm), _ptr(Cm),
                                        _ptr(Dk), _ptr(y), B, L, D, N)
    if rc:
        raise RuntimeError(f"mamba_oracle_fwd failed ({rc})")
    return y


def mamba_bwd_ref(x, delta, A, Bm, Cm, Dk, dy):
    """float64 gradients of <dy, y>: dict dx, ddelta, dA, dB, dC, dD (dD None
    when Dk is None)."""
    x, delta, A, Bm, Cm, Dk, dy = map(_f64, (x, delta, A, Bm, Cm, Dk, dy))
    B, L, D = x.shape
    N = A.shape[1]
    g = {"dx": np.empty((B, L, D)), "ddelta": np.empty((B, L, D)), "dA": np.empty((D, N)),
         "dB": np.empty((B, L, N)), "dC": np.empty((B, L, N)),
         "dD": np.empty((D,)) if Dk is not None else None}
    rc = _load_mamba().mamba_oracle_bwd(
        _ptr(x), _ptr(delta), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(Dk), _ptr(dy), _ptr(g["dx"]),
        _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]),
        B, L, D, N)
    if rc:
        raise RuntimeError(f"mamba_oracle_bwd failed ({rc})")
    return g
