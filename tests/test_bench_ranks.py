"""Host-side logic of bench.py's multi-rank (replica) mode, on CPU with gloo ranks: the job rate
divides the units of all ranks by the slowest rank's time, and the reference arm runs on rank 0
only.  No GPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [100.0, 250.0][rank]           # rank 1 is the slow one
    total, value = bench.job_rate(local_ms, 32 * 10, world, dist)
    out[rank] = (total, value)
    dist.barrier()
    dist.destroy_process_group()


def test_job_rate_is_max_over_ranks_world_2():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    for rank in (0, 1):
        total, value = res[rank]
        assert total == 250.0                  # both ranks see the slowest rank's time
        assert value == pytest.approx(2 * 320 / 0.25)   # all ranks' tokens / that time


def test_job_rate_single_rank():
    import bench
    total, value = bench.job_rate(50.0, 32 * 5, 1)
    assert total == 50.0 and value == pytest.approx(160 / 0.05)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import bench

    class A:
        steps, warmup = 1, 1
    bench.run_reference(A(), rank=1, world=2)   # returns at once: no oracle run, no line
    assert capsys.readouterr().out == ""


def test_reference_line_shares_the_workload_config(capsys, monkeypatch):
    """The reference arm's line carries the GPU arm's workload keys, metric and unit; the oracle
    timing is stubbed (two steps of 32 tokens in 0.5 s each: 64 tokens/s)."""
    import json
    import bench
    from attention_pre_processing_gb300 import workloads

    def fake(cfg, inp, budget_s, threads=None):
        return {"value": 64.0, "unit": "tokens/s", "cores": 2, "kind": "oracle",
                "sample": f"32 tokens of {cfg.workload} in 0.5 s (fp64 C, OpenMP over tokens)"}
    monkeypatch.setattr(bench, "cpu_baseline", fake)
    monkeypatch.setattr(workloads, "make_inputs", lambda cfg: None)

    class A:
        steps, warmup = 2, 3
    bench.run_reference(A(), rank=0, world=1)
    line = json.loads(capsys.readouterr().out)
    want = bench.workload_config(workloads.config(bench.HEADLINE), 1)
    assert {k: line["config"][k] for k in want} == want
    assert want["T"] == 32 and want["He"] == 7168 and want["N"] == 128
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["value"] == pytest.approx(64.0)
    assert line["e2e"]["value"] == line["value"] and line["cpu_baseline"]["cores"] == 2
