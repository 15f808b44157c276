"""The benchmark's multi-rank path on CPU: world_size-2 gloo process groups
stand in for one process per GPU.  The op shards into independent replicas
(no collective on the data path), so what the ranks share is the timing
aggregation (max over ranks, whole-job throughput) and the rule that only
rank 0 runs and prints the oracle's reference arm."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms_local = [1.5, 2.5][rank]
        ms = bench.max_over_ranks(ms_local, "cpu")
        value = bench.job_tokens_per_s(1000, world, ms)
        # the reference arm under torchrun: only rank 0 works and prints
        os.environ["RANK"] = str(rank)
        args = type("A", (), {"steps": 1, "warmup": 0, "gpus": world})()
        from ssd_chunked_scan_gb300.inputs import Workload
        tiny = Workload("tiny", B=2, G=2, H=4, L=70, dk=8, dv=8, chunk=64, la_mu=0.0, seed=1)
        buf = io.StringIO()
        with redirect_stdout(buf):
            rc = bench.run_reference(args, tiny)
        dist.barrier()
        with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": value, "rc": rc, "stdout": buf.getvalue()}, f)
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_aggregation_and_reference_arm(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(2)]
    assert r[0]["ms"] == r[1]["ms"] == 2.5          # the slowest rank's time
    assert r[0]["value"] == pytest.approx(1000 * 2 / 2.5e-3)
    assert r[0]["rc"] == r[1]["rc"] == 0
    assert r[1]["stdout"] == ""                     # rank 1 does no work
    line = json.loads(r[0]["stdout"].strip())
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_tokens_per_s(500, 1, 2.0) == pytest.approx(250000.0)
