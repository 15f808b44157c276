"""Seeded synthetic inputs for the SSD scan workloads.

Shared by the tests, the benchmark and the smoke check; it holds no part of
the scan's arithmetic -- only shapes and random draws.

Workload shapes are the [batch, groups, heads, dk, dv] tuples and sequence
lengths of the "kernel_ssd_gpu.json" benchmark page (its ``config.configs``
and ``config.seq_lens`` blocks).  Distributions (not on the pages):
q, k ~ N(0,1)/sqrt(dk); v ~ N(0,1); log_alpha = -softplus(N(mu,1)) with mu=0
(mu=-3 for the long-memory workload); h0 ~ 0.1 N(0,1); dout ~ N(0,1).
Draw order q, k, v, log_alpha, h0, dout from one PCG64 stream per workload.
"""
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    G: int
    H: int
    L: int
    dk: int
    dv: int
    chunk: int = 64
    la_mu: float = 0.0
    seed: int = 0

    @property
    def tokens(self) -> int:
        """Tokens per call as the benchmark pages count them: B * L * H."""
        return self.B * self.L * self.H


# index i gets seed 1000 + i
WORKLOADS = [
    Workload("g1h1_d128_L512", 4, 1, 1, 512, 128, 128, seed=1000),
    Workload("g2h4_dk48_dv40_L2048", 4, 2, 4, 2048, 48, 40, seed=1001),
    Workload("g2h8_d128_L2048", 4, 2, 8, 2048, 128, 128, seed=1002),
    Workload("g1h24_dk128_dv64_L8192", 2, 1, 24, 8192, 128, 64, seed=1003),
    Workload("g2h8_d128_L8192_long", 4, 2, 8, 8192, 128, 128, la_mu=-3.0, seed=1004),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def _softplus(x):
    return np.logaddexp(0.0, x)


def make_inputs(B, L, G, H, dk, dv, seed, la_mu=0.0, with_h0=True, with_dout=True):
    """float32 numpy arrays q, k, v, log_alpha, h0, dout (h0/dout None if not asked)."""
    rng = np.random.default_rng(seed)
    f32 = np.float32
    q = (rng.standard_normal((B, L, G, dk)) / np.sqrt(dk)).astype(f32)
    k = (rng.standard_normal((B, L, G, dk)) / np.sqrt(dk)).astype(f32)
    v = rng.standard_normal((B, L, H, dv)).astype(f32)
    la = (-_softplus(rng.standard_normal((B, L, H)) + la_mu)).astype(f32)
    h0 = (0.1 * rng.standard_normal((B, H, dk, dv))).astype(f32) if with_h0 else None
    dout = rng.standard_normal((B, L, H, dv)).astype(f32) if with_dout else None
    return q, k, v, la, h0, dout


def workload_inputs(w: Workload, with_h0=True, with_dout=True):
    return make_inputs(w.B, w.L, w.G, w.H, w.dk, w.dv, w.seed, w.la_mu, with_h0, with_dout)


def make_state_cotangent(B, H, dk, dv, seed):
    """float32 cotangent dhT [B,H,dk,dv] of the final state: standard normal
    scaled by 1/sqrt(dk), the size of one q_t dout_t^T term."""
    rng = np.random.default_rng(seed + 7919)
    return (rng.standard_normal((B, H, dk, dv)) / np.sqrt(dk)).astype(np.float32)


def make_inputs_on_device(device, B, L, G, H, dk, dv, seed, la_mu=0.0):
    """Seeded inputs generated on a CUDA device (for sizes too large to make
    on the host), with make_inputs' distributions but not its values:
    q, k ~ N(0,1)/sqrt(dk), v, dout ~ N(0,1), log_alpha = -softplus(N(la_mu,1)),
    h0 ~ 0.1 N(0,1), all float32 and contiguous."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    r = lambda *sh: torch.randn(sh, generator=gen, device=device)
    q = r(B, L, G, dk) / dk ** 0.5
    k = r(B, L, G, dk) / dk ** 0.5
    v = r(B, L, H, dv)
    la = -torch.nn.functional.softplus(r(B, L, H) + la_mu)
    h0 = 0.1 * r(B, H, dk, dv)
    dout = r(B, L, H, dv)
    return q, k, v, la, h0, dout


# ---- Mamba-1 selective scan ("kernel_mamba_cpu.json" records) --------------
#
# Shapes: batch 4, state 16, dim in {256, 512, 1024}, seq in {512, 2048, 8192}
# (the records' ``shape`` blocks).  Distributions (not on the pages): x, B, C,
# D, dy ~ N(0,1); delta log-uniform on [1e-3, 1e-1] (the range Mamba draws its
# step sizes from); A[d,n] = -(n+1) exp(0.5 N(0,1)) (the S4D-real
# initialisation -(n+1), perturbed per channel).  Draw order x, delta, A, B,
# C, D, dy from one PCG64 stream per workload.

@dataclass(frozen=True)
class MambaWorkload:
    name: str
    B: int
    L: int
    D: int
    N: int = 16
    seed: int = 0

    @property
    def tokens(self) -> int:
        """Channel-tokens per call: B * L * D."""
        return self.B * self.L * self.D


# index i gets seed 2000 + i
MAMBA_WORKLOADS = [
    MambaWorkload(f"mamba_d{d}_L{l}", 4, l, d, 16, seed=2000 + i)
    for i, (l, d) in enumerate([(512, 256), (2048, 256), (512, 512), (2048, 512), (512, 1024),
                                (2048, 1024), (8192, 256), (8192, 512), (8192, 1024)])
]
MAMBA_BY_NAME = {w.name: w for w in MAMBA_WORKLOADS}


def make_mamba_inputs(B, L, D, N, seed, with_D=True, with_dy=True):
    """float32 numpy arrays x, delta, A, Bm, Cm, Dk, dy (Dk / dy None if not asked)."""
    rng = np.random.default_rng(seed)
    f32 = np.float32
    x = rng.standard_normal((B, L, D)).astype(f32)
    delta = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), (B, L, D))).astype(f32)
    A = (-(np.arange(1, N + 1)[None, :]) * np.exp(0.5 * rng.standard_normal((D, N)))).astype(f32)
    Bm = rng.standard_normal((B, L, N)).astype(f32)
    Cm = rng.standard_normal((B, L, N)).astype(f32)
    Dk = rng.standard_normal((D,)).astype(f32) if with_D else None
    dy = rng.standard_normal((B, L, D)).astype(f32) if with_dy else None
    return x, delta, A, Bm, Cm, Dk, dy


def mamba_workload_inputs(w: MambaWorkload, with_D=True, with_dy=True):
    return make_mamba_inputs(w.B, w.L, w.D, w.N, w.seed, with_D, with_dy)
