"""Helpers shared by the GPU parity tests: run the CUDA library through the
binding on numpy inputs and compare with the float64 oracle."""
import numpy as np

from conftest import rel_err

# Tolerances on rel_err = max|x - ref| / max|ref|, per output and per gradient:
# the all-fp32 path must agree to 2e-5, the TF32 tensor-core path to 3e-3.
TOL = {"simt": 2e-5, "tc": 3e-3}


def to_dev(x):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_gpu(path, q, k, v, la, h0, dout, chunk, want_bwd=True):
    import torch
    from ssd_chunked_scan_gb300 import ssd
    ssd.ssd_set_path(ssd.SSD_PATH_SIMT if path == "simt" else ssd.SSD_PATH_TC)
    tq, tk, tv, tla, th0, tdo = map(to_dev, (q, k, v, la, h0, dout))
    out = ssd.ssd_fwd(tq, tk, tv, tla, th0, chunk=chunk)
    g = ssd.ssd_bwd(tq, tk, tv, tla, th0, tdo, chunk=chunk) if want_bwd else None
    torch.cuda.synchronize()
    assert ssd.ssd_last_device_error() == 0
    out = out.cpu().numpy()
    if g is not None:
        g = {n: (None if t is None else t.cpu().numpy()) for n, t in g.items()}
    return out, g


def compare(path, out, g, ref_out, ref_g, label=""):
    tol = TOL[path]
    errs = {"out": rel_err(out, ref_out)}
    if g is not None:
        for n in ("dq", "dk", "dv", "dlog_alpha", "dh0"):
            if ref_g.get(n) is not None and g.get(n) is not None:
                errs[n] = rel_err(g[n], ref_g[n])
    bad = {n: e for n, e in errs.items() if not (e <= tol)}
    assert not bad, f"{label} {path}: rel_err above {tol}: {bad} (all: {errs})"
    return errs
