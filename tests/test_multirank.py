"""Host logic of the multi-GPU bench path on CPU: two gloo ranks draw
independent batches (weak scaling, no collective on the data path) and the
step time reported is the maximum over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from paged_latent_attention_cache_gb300 import workloads as W
        seed = bench.rank_seed(5, rank)
        w = W.make_workload("r", q_lens=[1, 3], past_lens=[10, 4], num_heads=2, **W.GLM,
                            block_size=16, seed=seed)
        mine = float(10 + rank)                       # this rank's step time
        worst = bench.reduce_max(mine)
        bench.barrier()
        q.put((rank, seed, worst, float(w.query.float().sum())))
    finally:
        dist.destroy_process_group()


def test_two_ranks_reduce_max_and_independent_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, w0, q0), (r1, s1, w1, q1) = out
    assert (r0, r1) == (0, 1)
    assert w0 == w1 == 11.0          # max over ranks
    assert s0 != s1 and q0 != q1     # each rank draws its own batch


def test_algorithmic_work_counts_each_row_once():
    from paged_latent_attention_cache_gb300 import workloads as W
    w = W.make_workload("a", q_lens=[1, 4], past_lens=[9, 3], num_heads=2, **W.GLM,
                        block_size=16, seed=1)
    a = bench.algorithmic_work(w)
    # seq 0 sees rows 0..9 (10 rows), seq 1 sees rows 0..6 (7 rows)
    assert a["cache_rows"] == 17
    # flops: seq0 10 keys; seq1 tokens at pos 3..6 see 4+5+6+7 keys
    assert a["flops"] == (10 + 22) * 2 * (2 * 192 + 2 * 128)
