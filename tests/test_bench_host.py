"""Host-side logic of bench.py, on CPU: the multi-rank timing reduction (world size 2 over
gloo), the whole-job aggregation, and the reference arm's JSON line (the CPU oracle)."""

import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # each rank measured its own batch; rank 1 is the slow one
    step_seconds = 0.010 if rank == 0 else 0.025
    slowest = bench.max_over_ranks(step_seconds, world, torch.device("cpu"))
    agg = bench.aggregate(tokens_per_rank=2048, world=world, step_seconds_max=slowest, steps=5)
    bench.barrier(world)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"slowest": slowest, **agg}, f)
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["slowest"] == pytest.approx(0.025)
        # whole job: both ranks' tokens over the slowest rank's time (weak scaling)
        assert r["value"] == pytest.approx(2048 * 2 * 5 / 0.025)
        assert r["ms_per_step"] == pytest.approx(0.025 / 5 * 1e3)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(1.5, 1, torch.device("cpu")) == 1.5
    assert bench.aggregate(100, 1, 2.0, 4)["value"] == pytest.approx(200.0)


def test_reference_arm_line(capsys, monkeypatch):
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "tokens/s"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["higher_is_better"] is True


def test_reference_arm_other_ranks_print_nothing(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out.strip() == ""


def test_algorithmic_bytes_of_the_benchmark_apply():
    # x read once (2048 x 4096 bf16), y read and written once (fp32), the four adapters'
    # A and B read once, the ids and the permutation read once, the K+1 offsets
    import workloads
    wl = workloads.make("modality4")
    x = 2048 * 4096 * 2
    y = 2 * 2048 * 4096 * 4
    ab = 4 * (4096 * 16 + 16 * 4096) * 2
    idx = 2 * 2048 * 4 + 5 * 4
    assert bench.algorithmic_bytes(wl, 4) == x + y + ab + idx == 84_951_060
    # an adapter the batch does not touch costs nothing
    assert bench.algorithmic_bytes(wl, 3) == x + y + 3 * (4096 * 16 + 16 * 4096) * 2 + idx
