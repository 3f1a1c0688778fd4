"""Data-parallel replicas on CPU with a world-size-2 gloo group.

The path shards by token: each rank routes and lays out its own batch, with
no exchange of data between ranks; the benchmark only uses a barrier and a
max over ranks of the step time.  These tests run that host-side logic in two
processes: per-rank inputs, the max reduction, and that a rank's result does
not depend on the other rank (the oracle stands in for the GPU work)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    import synth

    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    wl = synth.WORKLOADS[1].with_tokens(64)
    seed = bench.replica_seed(wl.seed, rank, world)
    inp = synth.make_inputs(wl, seed=seed, want=("logits", "x"))
    idx, wts = oracle.route_softmax(inp["logits"], wl.K)
    L = oracle.layout(idx, wl.E, wl.R)
    recv, _, _ = oracle.dispatch(inp["x"], L, wts)
    out = oracle.combine(recv, L, wts)
    # the step time of this rank, and the max over ranks that the bench reports
    local_ms = 1.0 + rank
    bench.barrier(world)
    mx = bench.reduce_max(local_ms, world)
    np.savez(os.path.join(out_dir, "rank%d.npz" % rank), seed=seed, idx=idx, out=out,
             max_ms=mx, tokens=wl.T)
    dist.destroy_process_group()


def test_world2_replicas_route_independently_and_reduce_the_max(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [np.load(os.path.join(tmp_path, "rank%d.npz" % r)) for r in range(world)]
    # each rank drew its own batch
    assert int(res[0]["seed"]) != int(res[1]["seed"])
    assert not np.array_equal(res[0]["idx"], res[1]["idx"])
    # both ranks report the max step time, as the benchmark's line does
    assert float(res[0]["max_ms"]) == float(res[1]["max_ms"]) == 2.0
    # a rank's result is the single-process result for its own seed: no exchange
    import oracle
    import synth
    wl = synth.WORKLOADS[1].with_tokens(64)
    for r in range(world):
        inp = synth.make_inputs(wl, seed=int(res[r]["seed"]), want=("logits", "x"))
        idx, wts = oracle.route_softmax(inp["logits"], wl.K)
        L = oracle.layout(idx, wl.E, wl.R)
        recv, _, _ = oracle.dispatch(inp["x"], L, wts)
        assert np.array_equal(oracle.combine(recv, L, wts), res[r]["out"])
    # whole-job throughput counts every rank's tokens
    assert sum(int(r["tokens"]) for r in res) == world * wl.T


def test_replica_seeds_are_deterministic_and_single_rank_keeps_the_base_seed():
    import bench
    assert bench.replica_seed(0, 0, 1) == 0
    assert bench.replica_seed(0, 1, 4) == bench.replica_seed(0, 1, 4)
    seeds = {bench.replica_seed(0, r, 8) for r in range(8)}
    assert len(seeds) == 8


def test_reduce_max_is_identity_for_one_rank():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5


def _env_without_ranks():
    drop = ("RANK", "WORLD_SIZE", "LOCAL_RANK", "LOCAL_WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT")
    return {k: v for k, v in os.environ.items() if k not in drop}


def test_bench_gpus_flag_starts_one_rank_per_gpu():
    """`bench.py --gpus 2` started as a plain process runs itself again as two
    ranks under torch.distributed.run.  The reference arm (the CPU oracle on
    rank 0; the other ranks exit at once) needs no GPU, so the launch path is
    exercised here: one JSON line, reporting both ranks."""
    import json
    import subprocess
    import sys
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3", "--workload", "1", "--ref-tokens", "16"]
    r = subprocess.run(cmd, capture_output=True, text=True, env=_env_without_ranks(), timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2


def test_bench_rejects_a_rank_count_that_differs_from_gpus():
    import subprocess
    import sys
    env = dict(_env_without_ranks(), WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 2 and "ranks were started" in r.stderr
