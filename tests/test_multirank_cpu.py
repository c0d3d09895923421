"""The N > 1 host logic of bench.py on CPU: two ranks over gloo (world size
2, 127.0.0.1), no GPU.  Each rank draws its own batch (the data-parallel
shard), the timed duration is the maximum over ranks on every rank, and the
job's throughput counts every rank's tokens over that slowest time."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
import nc_synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = nc_synth.WORKLOADS["tiny_f32"]
        ids, tg = bench.rank_batch(w, rank)
        shards = [None] * world
        dist.all_gather_object(shards, (ids.tolist(), tg.tolist()))
        local = 10.0 + 5.0 * rank          # this rank's "duration"
        slowest = bench.max_over_ranks(local, world)
        out[rank] = {"shards": shards, "slowest": slowest,
                     "value": bench.job_tokens_per_s(w.batch, w.seq, world, 3, slowest / 1000.0),
                     "again": bench.rank_batch(w, rank)[0].tolist()}
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_shard_time_and_throughput():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    res = dict(out)
    w = nc_synth.WORKLOADS["tiny_f32"]
    # every rank saw the same gathered shards; the shards differ between ranks
    assert res[0]["shards"] == res[1]["shards"]
    ids0, ids1 = (np.array(res[0]["shards"][r][0]) for r in range(world))
    assert ids0.shape == ids1.shape == (w.batch, w.seq)
    assert not np.array_equal(ids0, ids1)
    # a rank's shard is reproducible (same seed, same rows)
    for r in range(world):
        assert res[r]["again"] == res[r]["shards"][r][0]
    # targets are the ids shifted by one within each rank's own stream
    for r in range(world):
        ids, tg = (np.array(a) for a in res[r]["shards"][r])
        assert np.array_equal(tg[:, :-1], ids[:, 1:])
    # the slowest rank's time, on both ranks; throughput over the whole job
    assert res[0]["slowest"] == res[1]["slowest"] == 15.0
    expect = w.batch * w.seq * world * 3 / 0.015
    assert res[0]["value"] == pytest.approx(expect) and res[1]["value"] == pytest.approx(expect)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_tokens_per_s(2, 64, 1, 4, 0.5) == 2 * 64 * 4 / 0.5


def _bench_cmd(*args):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    return [sys.executable, os.path.join(root, "bench.py"), *args], env


def test_bench_gpus_flag_starts_that_many_ranks():
    """`bench.py --gpus 2` with no launcher starts two ranks itself (gloo here,
    host only: --launcher-check runs no GPU work) and reports n_gpus 2."""
    import json
    import subprocess
    cmd, env = _bench_cmd("--gpus", "2", "--launcher-check")
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = lines[0]
    assert out["n_gpus"] == 2
    assert sorted(x["rank"] for x in out["ranks"]) == [0, 1]
    assert all(x["world"] == 2 for x in out["ranks"])
    assert sorted(x["local_rank"] for x in out["ranks"]) == [0, 1]


def test_bench_refuses_a_launcher_world_that_differs_from_gpus():
    import subprocess
    cmd, env = _bench_cmd("--gpus", "4", "--launcher-check")
    env.update(RANK="0", WORLD_SIZE="2", LOCAL_RANK="0")
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 2
    assert "--gpus 4" in r.stderr
