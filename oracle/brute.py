"""Brute-force unrolled sums for tiny cases -- test infrastructure only.

Pins the sequential oracle to the closed form obtained by unrolling the
recurrence S_t = exp(la_t) S_{t-1} + k_t v_t^T, out_t = S_t^T q_t:

    out_t = sum_{s<=t} exp(sum_{r=s+1..t} la_r) (q_t . k_s) v_s
            + exp(sum_{r<=t} la_r) h0^T q_t

Each decay exponent is summed directly over its own index range (no
differences of running sums), in plain Python loops, float64.  Only for tiny
L (the cost is O(L^3) per head).
"""
import math

import numpy as np


def ssd_fwd_brute(q, k, v, la, h0=None):
    q, k, v, la = (np.asarray(x, np.float64) for x in (q, k, v, la))
    B, L, G, dk = q.shape
    H, dv = v.shape[2], v.shape[3]
    hpg = H // G
    out = np.zeros((B, L, H, dv))
    for b in range(B):
        for h in range(H):
            g = h // hpg
            for t in range(L):
                acc = np.zeros(dv)
                for s in range(t + 1):
                    e = 0.0
                    for r in range(s + 1, t + 1):
                        e += la[b, r, h]
                    acc += math.exp(e) * float(np.dot(q[b, t, g], k[b, s, g])) * v[b, s, h]
                if h0 is not None:
                    e = 0.0
                    for r in range(t + 1):
                        e += la[b, r, h]
                    acc += math.exp(e) * (np.asarray(h0, np.float64)[b, h].T @ q[b, t, g])
                out[b, t, h] = acc
    return out


def ssd_final_state_brute(k, v, la, h0=None):
    """hT = sum_s exp(sum_{r=s+1..L-1} la_r) k_s v_s^T + exp(sum_{r<=L-1} la_r) h0,
    per (b, h), each exponent summed directly.  [B,H,dk,dv]"""
    k, v, la = (np.asarray(x, np.float64) for x in (k, v, la))
    B, L, G, dk = k.shape
    H, dv = v.shape[2], v.shape[3]
    hpg = H // G
    hT = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            g = h // hpg
            acc = np.zeros((dk, dv))
            for s in range(L):
                e = 0.0
                for r in range(s + 1, L):
                    e += la[b, r, h]
                acc += math.exp(e) * np.outer(k[b, s, g], v[b, s, h])
            if h0 is not None:
                e = 0.0
                for r in range(L):
                    e += la[b, r, h]
                acc += math.exp(e) * np.asarray(h0, np.float64)[b, h]
            hT[b, h] = acc
    return hT
