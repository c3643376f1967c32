"""Host-side logic of the multi-GPU bench path on CPU: two gloo ranks (the
replicas a torchrun launch of bench.py creates) agree on a barrier and report
the maximum of their step times, the value rank 0 prints."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    w, r, local, dist = bench.init_dist()
    assert (w, r, local) == (world, rank, rank) and dist is not None
    bench.barrier(dist)
    mine = 1.5 + rank           # this rank's "ms per step"
    results[rank] = bench.max_over_ranks(dist, mine)
    bench.barrier(dist)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(results) == {0: 2.5, 1: 2.5}


def test_single_process_needs_no_process_group():
    os.environ.pop("WORLD_SIZE", None)
    import bench
    w, r, local, dist = bench.init_dist()
    assert (w, r, dist) == (1, 0, None)
    assert bench.max_over_ranks(None, 3.0) == 3.0


def _reference_rank(rank, world, port, outdir):
    import argparse
    import contextlib
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    with open(os.path.join(outdir, "rank%d.txt" % rank), "w") as f, contextlib.redirect_stdout(f):
        bench.run_reference(argparse.Namespace(steps=1, warmup=0, gpus=world))


def test_reference_arm_under_two_ranks_prints_one_line_from_rank_zero(tmp_path):
    import json
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_reference_rank, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=600)
        assert p.exitcode == 0
    assert (tmp_path / "rank1.txt").read_text() == ""
    lines = (tmp_path / "rank0.txt").read_text().strip().splitlines()
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
