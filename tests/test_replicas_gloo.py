"""Multi-GPU host logic of bench.py, run as two gloo ranks on the CPU.

The decode path has no exchange step, so N GPUs run N independent replicas;
the only cross-rank work is the timing protocol: a barrier around the timed
region, the max of the per-rank times, and the whole-job value (bytes of all
ranks over the slowest rank's time)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = [3.0, 5.0][rank]
        bench.barrier(dist)
        worst = bench.max_over_ranks(my_ms, dist, "cpu")
        value = bench.aggregate_value(1_000_000_000, world, worst)
        q.put((rank, worst, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, worst, value in res:
        assert worst == 5.0                       # slowest rank's time on every rank
        assert value == pytest.approx(2 * 1e9 / 5e-3 / 1e9)  # 400 GB/s for both ranks


def test_reference_arm_only_rank0_prints(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""


def test_reference_arm_line(capsys, monkeypatch):
    """Rank 0 prints the reference arm's line: the oracle on the host cores,
    on the same workload shape as the GPU arm's config."""
    import json

    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"])
    d = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["config"] == bench.shape_config("tiny")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] == d["e2e"]["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
