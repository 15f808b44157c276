"""The tensor layout is pinned by the argument / output buffer sizes that the
benchmark pages record for every chunked run (tests/golden/page_buffer_sizes.json).

fwd:     args = q + k [B,L,G,dk] + v [B,L,H,dv] + log_alpha [B,L,H] + h0 [B,H,dk,dv],
         out  = out [B,L,H,dv]  (no final state is returned)
fwd_bwd: out  = the five gradients (same sizes as the args) + 40 bytes of scalars.
"""
import json
import os

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROWS = json.load(open(os.path.join(HERE, "golden", "page_buffer_sizes.json")))["rows"]
MB = 2.0 ** 20


def _arg_bytes(r):
    B, L, G, H, dk, dv = r["B"], r["L"], r["G"], r["H"], r["dk"], r["dv"]
    return 4 * (2 * B * L * G * dk + B * L * H * dv + B * L * H + B * H * dk * dv)


@pytest.mark.parametrize("r", ROWS, ids=lambda r: f"{r['page']}-{r['mode']}-{r['config']}-L{r['L']}")
def test_page_buffer_sizes(r):
    assert _arg_bytes(r) / MB == pytest.approx(r["xla_arg_mb"], abs=1e-9)
    if r["mode"] == "fwd":
        assert 4 * r["B"] * r["L"] * r["H"] * r["dv"] / MB == pytest.approx(r["xla_out_mb"], abs=1e-9)
    else:
        assert (_arg_bytes(r) + 40) / MB == pytest.approx(r["xla_out_mb"], abs=1e-9)


def test_workloads_use_page_shapes():
    from ssd_chunked_scan_gb300.inputs import WORKLOADS
    page = {(r["B"], r["G"], r["H"], r["dk"], r["dv"], r["L"]) for r in ROWS}
    for w in WORKLOADS:
        assert (w.B, w.G, w.H, w.dk, w.dv, w.L) in page
