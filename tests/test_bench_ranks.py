"""bench.py's multi-rank logic on CPU: two gloo ranks, the max-over-ranks time, the
whole-job value and the reference arm's rank-0-only rule. No GPU is touched."""
import json
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = 10.0 + 7.5 * rank                      # rank 1 is the slowest
    total = bench.max_over_ranks(mine, "cpu")
    value = bench.job_value(world, 304, 3, total)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"mine": mine, "total": total, "value": value}, f)


def test_max_over_ranks_and_weak_scaling_value(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["total"] == 17.5                   # every rank sees the slowest rank's time
        assert r["value"] == pytest.approx(world * 304 * 3 / 0.0175)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.job_value(1, 304, 10, 1000.0) == pytest.approx(3040.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun the other ranks of the reference arm exit without work or output."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "host_samples", lambda *a, **k: called.append(1) or [])

    class Args:
        steps, warmup, gpus, ref_queries = 2, 3, 2, 1
    bench.run_reference(Args, bench.inputs.WORKLOADS["v4flash_decode"], 304)
    assert not called and capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    """Rank 0 of the reference arm times the oracle and prints one complete JSON line."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "0")

    class Args:
        steps, warmup, gpus, ref_queries = 1, 1, 1, 1
    bench.run_reference(Args, bench.inputs.WORKLOADS["v4flash_decode"], 304)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "queries/s" and line["value"] > 0
    assert line["higher_is_better"] is True and line["metric"] == bench.METRIC
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
