"""The replica harness of bench.py over two processes on the CPU (gloo):
rendezvous on 127.0.0.1, the barrier, the max-over-ranks time and the
whole-job value; and the reference arm's rank rule (rank 0 alone runs)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    ws, r = bench.dist_setup()
    assert dist.get_backend() == "gloo"
    bench.barrier(ws)
    elapsed = bench.max_over_ranks(10.0 + 5.0 * rank, ws)        # rank 1 is the slower one
    value = bench.aggregate(ws, 60, 4, elapsed)
    bench.barrier(ws)
    q.put((r, ws, elapsed, value))
    dist.destroy_process_group()


def test_two_replicas_rendezvous_barrier_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    # both ranks see the slowest rank's time; value = all ranks' rows over it
    assert got == [(0, 2, 15.0, 2 * 60 * 4 / 0.015), (1, 2, 15.0, 2 * 60 * 4 / 0.015)]


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_runs_on_rank_zero_only(rank):
    env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--config", "1", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank == 1:
        assert lines == []
    else:
        d = json.loads(lines[-1])
        assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
        assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
        # the same workload description as the GPU arm prints, every tree row timed
        assert d["config"]["workload"] == "tiny-fp32-d256-p24-tree8"
        assert d["config"]["tree_rows"] == 8 and d["config"]["paged"] is False
        assert d["rows_timed_per_step"] == 8


def _shard_worker(rank, port, q, logits, cuts):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from oracle import argmax_rows
    from speculative_decoding_tree_gb300.dist import allreduce_argmax
    dist.init_process_group("gloo", rank=rank, world_size=2)
    lo, hi = cuts[rank], cuts[rank + 1]
    shard = logits[:, lo:hi]
    # the rank's local result, as tv_lm_head_argmax gives it for its slice
    am = torch.from_numpy(argmax_rows(shard)).to(torch.int32)
    mx = torch.tensor([float(shard[r, am[r]]) if not all(x != x for x in shard[r]) else float("nan")
                       for r in range(shard.shape[0])], dtype=torch.float32)
    v, i = allreduce_argmax(mx, am, lo)
    q.put((rank, v.tolist(), i.tolist()))
    dist.destroy_process_group()


def test_vocab_sharded_argmax_allreduce():
    import numpy as np
    from oracle import argmax_rows
    g = np.random.default_rng(0)
    logits = g.normal(size=(6, 40)).astype(np.float32)
    logits[1, 5] = logits[1, 30] = 9.0            # a tie across the two shards: the smaller token wins
    logits[2, 12] = logits[2, 13] = 9.5           # a tie inside one shard
    logits[3, :] = np.nan                         # no valid entry anywhere
    logits[4, :20] = np.nan                       # no valid entry on rank 0
    cuts = [0, 20, 40]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, port, q, logits, cuts)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    ref = argmax_rows(logits)
    for rank, vals, idx in got:
        assert idx == ref.tolist()
        for r in range(6):
            if r == 3:
                assert vals[r] != vals[r]
            else:
                assert vals[r] == float(logits[r, ref[r]])
