"""Host logic of the multi-rank benchmark on CPU: two gloo ranks, no GPU.

Each rank runs its own tree (weak scaling, no data-path collective); the only exchange is the
max-over-ranks of the step times, and only rank 0 reports.  These tests run that exchange
over gloo between two processes and check the reference arm's rank gating.
"""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                                         world_size=world)
    try:
        # rank r: step 5 + r ms, e2e 9 - r ms -> every rank must see (5 + world - 1, 9)
        got = bench.reduce_max([5.0 + rank, 9.0 - rank], torch.device("cpu"), world)
        out_q.put((rank, got))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: [6.0, 9.0], 1: [6.0, 9.0]}


def test_single_rank_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max([1.5, 2.5], torch.device("cpu"), 1) == [1.5, 2.5]


def test_reference_arm_other_ranks_exit_quietly(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.main() == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank0(monkeypatch, capsys):
    """Rank 0 of the reference arm times the oracle on the host cores and prints one line with
    the keys the harness reads (a bounded sample per step; tiny tree keeps it short)."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setattr(bench, "cpu_baseline_sample",
                        lambda config, budget_s: dict(value=1e-3, unit=bench.UNIT, cores=1, kind="oracle",
                                                      sample="stub", seconds=0.01))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3"])
    assert bench.main() == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["unit"] == bench.UNIT and line["steps"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_profiled_traffic_is_null_for_stale_or_foreign_counters(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    prof = tmp_path / "p.md"
    digest = bench.source_digest(bench.DKDV_SOURCES)
    prof.write_text(f"- workload: rollout32k\n- source_sha1: {digest}\n- dram_bytes_per_launch: 123456\n")
    monkeypatch.setattr(bench, "DKDV_PROFILE", str(prof))
    assert bench.profiled_traffic("rollout32k") == 123456
    assert bench.profiled_traffic("forest") is None
    prof.write_text("- workload: rollout32k\n- source_sha1: 0000\n- dram_bytes_per_launch: 123456\n")
    assert bench.profiled_traffic("rollout32k") is None
