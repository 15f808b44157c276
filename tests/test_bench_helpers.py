"""The benchmark's pure helpers on CPU: the roofline entry of the dominant
kernel, the per-kernel table, the algorithmic cost of every kernel the
library can launch on the benchmark workload, and the traffic table."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from ssd_chunked_scan_gb300.inputs import BY_NAME  # noqa: E402

PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "measured"}


def test_roofline_takes_the_kernel_with_most_time():
    costs = {"a": (1e9, 0.0, "hbm"), "b": (2e9, 0.0, "hbm")}
    trace = {"a": (10, 5.0), "b": (4, 6.0)}  # b: 1.5 ms per launch
    r = bench.kernel_roofline(trace, costs, PEAKS, traffic_ok=False)
    assert r["kernel"] == "b"
    assert r["kernel_ms_per_launch"] == pytest.approx(1.5)
    assert r["achieved"] == pytest.approx(2e9 / 1.5e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6800.0)
    assert r["traffic"] is None and r["bound"] == "hbm" and r["unit"] == "GB/s"


def test_roofline_tensor_and_alu_bounds():
    t = bench.kernel_roofline({"k": (1, 2.0)}, {"k": (0.0, 4e12, "tensor")}, PEAKS, False)
    assert t["unit"] == "TFLOP/s"
    assert t["achieved"] == pytest.approx(4e12 / 2e-3 / 1e12)
    assert t["peak"] == pytest.approx(1900.0 * bench.TF32_OVER_BF16)
    a = bench.kernel_roofline({"k": (1, 1.0)}, {"k": (0.0, 1e12, "alu")}, PEAKS, False)
    assert a["bound"] == "alu" and a["peak"] == pytest.approx(bench.FP32_TFLOPS)


def test_roofline_refuses_a_kernel_without_a_cost():
    with pytest.raises(KeyError):
        bench.kernel_roofline({"x": (1, 1.0)}, {}, PEAKS, False)


def test_kernel_table_shares_sum_to_one():
    tab = bench.kernel_table({"a": (2, 3.0), "b": (1, 1.0)})
    assert list(tab) == ["a", "b"]
    assert sum(v["share"] for v in tab.values()) == pytest.approx(1.0)
    assert tab["a"]["launches"] == 2


def test_every_traced_kernel_has_a_cost_and_a_traffic_figure_or_a_reason():
    w = BY_NAME[bench.WORKLOAD]
    costs = bench.kernel_costs(w, 152)
    names = ["tc.seg_state", "tc.seg_state_dq", "tc.seg_state_dk", "tc.seg_scan", "tc.walk_out",
             "tc.walk_dq", "tc.walk_dk", "tc.walk_dv", "tc.dla_intra", "tc.dla",
             "simt.chunk_state", "simt.query_state", "simt.state_scan_fwd",
             "simt.state_scan_rev", "simt.chunk_out", "simt.chunk_grad", "simt.dla_carry"]
    for n in names:
        assert n in costs, n
        kb, kf, bound = costs[n]
        assert kb > 0 and bound in ("hbm", "tensor", "alu")
        t, why = bench.traffic_of(n)
        assert why, n
        if t is not None:
            # a capture that moved far fewer bytes than the algorithmic count
            # would mean the cost model counts something the kernel never touches
            assert t >= 0.5 * kb or n in ("tc.seg_scan", "tc.dla"), n


def test_traffic_is_dropped_once_the_kernel_source_changes(monkeypatch):
    grp = dict(bench.TRAFFIC_GROUPS["tc."], sha16="0" * 16, commit="abc1234",
               bytes={"tc.walk_dq": 123})
    monkeypatch.setitem(bench.TRAFFIC_GROUPS, "tc.", grp)
    t, why = bench.traffic_of("tc.walk_dq")
    assert t is None and "changed" in why and "abc1234" in why
    monkeypatch.setitem(bench.TRAFFIC_GROUPS, "tc.", dict(grp, sha16=bench._sha16(grp["source"])))
    t, why = bench.traffic_of("tc.walk_dq")
    assert t == 123 and "unchanged" in why
    assert bench.traffic_of("tc.walk_dk")[0] is None
    assert bench.traffic_of("nothing.like.this")[0] is None


def test_step_totals_match_the_workload_sizes():
    w = BY_NAME[bench.WORKLOAD]
    bytes_fb, fl_fb, bytes_f, fl_f = bench.step_totals(w)
    mib = 2 ** 20
    # fwd: arguments (q, k, v, log_alpha, h0) + out
    args = 4 * (2 * w.B * w.L * w.G * w.dk + w.B * w.L * w.H * w.dv + w.B * w.L * w.H
                + w.B * w.H * w.dk * w.dv)
    out = 4 * w.B * w.L * w.H * w.dv
    assert bytes_f == args + out
    assert bytes_f / mib == pytest.approx(323, abs=1)
    assert bytes_fb / mib == pytest.approx(841, abs=1)
    assert fl_fb > fl_f > 0


def test_sweep_resumes_after_recorded_lines(tmp_path):
    from ssd_chunked_scan_gb300.inputs import WORKLOADS
    recs = bench.sweep_records(WORKLOADS)
    # five page workloads x two paths x two modes, each path taking all five
    assert len(recs) == 20 and len({bench.sweep_key(r) for r in recs}) == 20
    out = tmp_path / "sweep.jsonl"
    assert bench.sweep_todo(str(out), recs) == recs  # nothing recorded yet
    import json
    with open(out, "w") as f:
        f.write(json.dumps({"record": recs[0], "result": {"value": 1.0}}) + "\n")
        f.write(json.dumps({"record": recs[3], "error": "exit 1: boom"}) + "\n")
        f.write('{"record": {"workload": "g1h1')  # cut short by an interruption
    todo = bench.sweep_todo(str(out), recs)
    assert recs[0] not in todo and recs[3] not in todo
    assert len(todo) == 18 and todo[0] == recs[1]


def test_l2_note_says_whether_a_step_fits_in_l2():
    w = BY_NAME[bench.WORKLOAD]
    big = bench.resident_bytes(w.B, w.L, w.G, w.H, w.dk, w.dv, "fwd_bwd")
    assert big > bench.L2_BYTES and "exceed L2" in bench.l2_note(big)
    small = BY_NAME["g1h1_d128_L512"]
    b = bench.resident_bytes(small.B, small.L, small.G, small.H, small.dk, small.dv, "fwd")
    assert b < bench.L2_BYTES and "fit in L2" in bench.l2_note(b)
