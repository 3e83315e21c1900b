"""Multi-rank logic of bench.py on CPU: two gloo ranks.

The bench runs one replica of the step per GPU; the job's step time is the
slowest rank's and its throughput counts the work of every rank.  This
checks that aggregation with world size 2 (no GPU), and that the oracle
reference arm runs on rank 0 only.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    local_ms = [2.0, 5.0][rank]                  # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms, ws)
    value = bench.job_throughput(1e9, ws, ms)
    out[rank] = (ms, value)
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_two_gloo_ranks():
    ws = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(ws, _free_port(), out), nprocs=ws, start_method="spawn", join=True)
    for rank in range(ws):
        ms, value = out[rank]
        assert ms == 5.0                                  # every rank sees the slowest time
        assert value == pytest.approx(2 * 1e9 / 5e-3)     # both ranks' work / that time


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_throughput(10.0, 1, 1000.0) == pytest.approx(10.0)


def test_reference_arm_runs_on_rank_zero_only():
    import sys
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup = 1, 0
    assert bench.run_reference(A, 2, 1) is None          # rank 1: no work, nothing printed


def test_reference_arm_line_has_the_contract_keys():
    """One step of the oracle reference arm (on this CPU): the JSON line it
    prints carries the base keys, a cpu_baseline describing the run and an
    e2e block with no host-device bytes."""
    import json
    import sys
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup = 1, 0
    out = bench.run_reference(A, 1, 0)
    json.dumps(out)                                       # serialisable as one line
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in out, k
    assert out["impl"] == "reference" and out["metric"] == bench.METRIC and out["unit"] == "TFLOP/s"
    assert out["value"] > 0 and out["higher_is_better"] is True and out["n_gpus"] == 1
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == out["value"]
    e2e = out["e2e"]
    assert e2e["value"] == out["value"] and e2e["unit"] == out["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
