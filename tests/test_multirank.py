"""Multi-rank paths on the CPU with the gloo backend (world size 2).

* bench.py's job time is the maximum over ranks;
* the sharded quantization design: each rank owns a range of 16-row stripes,
  the two amax values are combined with an all-reduce(MAX), and stochastic
  rounding counters are offset by first_row * N -- the gathered shards equal
  the unsharded result bit for bit (checked with the CPU oracle).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _max_worker(rank, world, port, q):
    _init(rank, world, port)
    import bench
    q.put((rank, bench.max_over_ranks(10.0 + 5 * rank, world)))
    dist.destroy_process_group()


def _shard_worker(rank, world, port, q):
    _init(rank, world, port)
    import oracle
    import synthetic
    flags = 1 | 2 | 16 | 32  # both copies, Hadamard on the columnwise copy, stochastic rounding
    full = synthetic.gradient(64, 48, 7)
    M, N = full.shape
    rows = M // world
    mine = full[rank * rows:(rank + 1) * rows]
    st, am = oracle.amax(mine, flags, rht_seed=11)
    t = torch.from_numpy(am.copy())
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    out = oracle.quantize(mine, N, t.numpy(), flags, sr_seed=5, rht_seed=11, counter_offset=rank * rows * N)
    q.put((rank, {k: v for k, v in out.items() if k != "status"}, out["status"]))
    dist.destroy_process_group()


def _run(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=fn, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(results, key=lambda r: r[0])


def test_job_time_is_the_max_over_ranks():
    res = _run(_max_worker)
    assert [v for _, v in res] == [15.0, 15.0]


def test_row_shards_with_amax_allreduce_reproduce_the_whole_tensor():
    import oracle
    import synthetic
    res = _run(_shard_worker)
    assert all(st == 0 for _, _, st in res)
    full = synthetic.gradient(64, 48, 7)
    flags = 1 | 2 | 16 | 32
    st, am = oracle.amax(full, flags, rht_seed=11)
    whole = oracle.quantize(full, 48, am, flags, sr_seed=5, rht_seed=11)
    shards = [o for _, o, _ in res]
    assert np.array_equal(np.concatenate([o["q_row"] for o in shards]), whole["q_row"])
    assert np.array_equal(np.concatenate([o["s_row"] for o in shards]), whole["s_row"])
    assert np.array_equal(np.concatenate([o["q_col"] for o in shards], axis=1), whole["q_col"])
    assert np.array_equal(np.concatenate([o["s_col"] for o in shards], axis=1), whole["s_col"])
    for o in shards:
        assert np.array_equal(o["alpha"], whole["alpha"])
