"""The N > 1 host logic of bench.py on CPU: two gloo ranks. Every rank runs
an independent replica on its own hidden vectors; the job's time is the
slowest rank's and its rate counts every rank's rows. No GPU is involved."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = 10.0 + 5.0 * rank           # rank 1 is the slow one
        ms = bench.max_over_ranks(ms_local, world, "cpu")
        rate = bench.aggregate_rate(world, 64, 100, ms)
        W = synth.make_head(96, 32, 0)
        h = bench.hidden(W, 4, rank)
        np.save(os.path.join(out_dir, f"rank{rank}.npy"), np.concatenate(
            [np.array([ms, rate]), h.astype(np.float64).ravel()]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    r0 = np.load(tmp_path / "rank0.npy")
    r1 = np.load(tmp_path / "rank1.npy")
    # both ranks agree on the slowest rank's time and on the whole-job rate
    assert r0[0] == r1[0] == 15.0
    assert r0[1] == r1[1] == pytest.approx(2 * 64 * 100 / 0.015)
    # each replica works on its own hidden vectors
    assert not np.array_equal(r0[2:], r1[2:])


def test_single_rank_is_identity():
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert bench.aggregate_rate(1, 64, 10, 1.0) == pytest.approx(640000.0)


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    # under torchrun only rank 0 times the oracle; the other ranks exit without work
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 1, 0

    assert bench.run_reference(Args()) is None
    assert capsys.readouterr().out == ""


def test_workload_config_names_the_headline_workload():
    # both arms print this dict; the candidate count is the local head's
    c = bench.workload_config(64, 2, 4)
    assert (c["n"], c["d"], c["r"], c["M"], c["tile"], c["k_tile"]) == (128256, 4096, 256, 64, 256, 2)
    assert c["candidates"] == 1002 == (128256 // 256) * 2
    assert c["parallelism"] == "replicas x2 (independent hidden vectors)"
    assert "> 2x L2" in c["l2"] and "> 2x L2" not in bench.workload_config(64, 1, 1)["l2"]


def test_pstats_percentiles():
    s = bench.pstats([float(x) for x in range(1, 102)])      # 1 .. 101
    assert (s["median"], s["p10"], s["p90"], s["calls"]) == (51.0, 11.0, 91.0, 101)


def test_dense_speedups_pair_by_head_and_M():
    rows = [{"config": 1, "head": "two_stage", "mode": "global", "M": 4, "us": 50.0},
            {"config": 2, "head": "two_stage", "mode": "local", "M": 4, "us": 25.0},
            {"config": 2, "head": "dense", "M": 4, "us": 175.0},
            {"config": 4, "head": "two_stage", "mode": "local", "M": 8, "us": 40.0},
            {"config": 4, "head": "dense", "M": 8, "us": 300.0},
            {"config": 4, "head": "pruned", "M": 8, "us": 60.0}]
    out = {(e["config"], e["M"]): e["speedup"] for e in bench.dense_speedups(rows)}
    # configurations 1 and 2 share a head, so share its dense timing
    assert out == {(1, 4): 3.5, (2, 4): 7.0, (4, 8): 7.5}


def test_config_plan_covers_every_named_configuration():
    plan = {(c, kind, mode, C, k): Ms for c, kind, mode, C, k, Ms in bench.CONFIG_PLAN}
    assert plan[(1, "two_stage", "global", 1024, 0)] == (1, 4, 8)
    assert plan[(2, "two_stage", "local", 256, 2)] == (1, 8, 16, 32, 64)
    assert {(3, "two_stage", "local", 256, 2), (3, "two_stage", "global", 1024, 0)} <= set(plan)
    assert plan[(4, "two_stage", "local", 256, 4)] == (1, 8, 32, 128, 512)
    assert plan[(4, "pruned", None, 32000, 0)] == (1, 8, 32, 128, 512)
    assert set(plan[(2, "dense", None, 0, 0)]) >= {1, 4, 8, 16, 32, 64}
