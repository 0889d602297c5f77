"""Data-parallel replicas (CPU, gloo, world size 2): whole packed sequences are
load-balanced across ranks longest-first, with no exchange of attention data.

Each rank computes its shard from the same global batch; the ranks then
all-gather their shard lists and check that the shards partition the batch,
that every rank derived the same assignment, and that the most loaded rank is
within one sequence of the mean (the list-scheduling bound)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from diffusion_lm_block_bda_b300 import sharding, workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, n_seq, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        gen = torch.Generator().manual_seed(0)
        lens = W.packed_lengths(gen, n=n_seq)
        full = W.Workload("batch", W.BLOCK_CAUSAL, 32, 32, 8, 128, lens, list(lens))
        costs = sharding.sequence_costs(full)
        shards = sharding.lpt_shard(costs, world)
        mine = shards[rank]
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        sub = sharding.subset(full, mine)
        load = torch.tensor([sum(costs[i] for i in mine)], dtype=torch.float64)
        loads = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(loads, load)
        if rank == 0:
            out.put((gathered, shards, [float(x) for x in loads], costs, sub.seqlens_q,
                     [lens[i] for i in mine]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("n_seq", [16, 33])
def test_lpt_sharding_two_gloo_ranks(n_seq):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n_seq, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    gathered, shards, loads, costs, sub_lens, want_lens = q.get()
    assert gathered == shards  # every rank derived the same assignment
    flat = sorted(i for s in gathered for i in s)
    assert flat == list(range(n_seq))
    assert sum(loads) == sum(costs)
    assert max(loads) <= sum(costs) / world + max(costs)
    assert sub_lens == want_lens


def test_lpt_shard_single_rank_and_errors():
    assert sharding.lpt_shard([5, 1, 3], 1) == [[0, 1, 2]]
    assert sharding.lpt_shard([], 3) == [[], [], []]
    with pytest.raises(ValueError):
        sharding.lpt_shard([1], 0)


def test_bench_launches_its_own_ranks_and_shards_the_batch():
    """`bench.py --gpus 2` without an outer launcher starts two ranks itself
    (torch.distributed.run; here with gloo and no kernel, --stub): both ranks
    start, and their shards partition the 32-sequence global batch."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--stub"],
                         capture_output=True, text=True, timeout=300, env=env, cwd=root)
    assert res.returncode == 0, res.stderr[-2000:]
    line = [ln for ln in res.stdout.splitlines() if ln.startswith("{")][-1]
    out = json.loads(line)
    assert out["n_gpus"] == 2 and out["gpus_active"] == 2
    shards = out["shards"]
    assert len(shards) == 2 and all(shards)
    assert sorted(i for sh in shards for i in sh) == list(range(32))
    loads = out["shard_pairs"]
    assert max(loads) - min(loads) <= max(loads) * 0.25


def test_bench_refuses_a_world_size_that_differs_from_gpus():
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="3", RANK="0", LOCAL_RANK="0")
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--stub"],
                         capture_output=True, text=True, timeout=120, env=env, cwd=root)
    assert res.returncode != 0 and "WORLD_SIZE=3" in res.stderr
