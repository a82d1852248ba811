"""Multi-process host logic on the CPU: world_size 2 over gloo.

Each rank runs the fp64 oracle on its share of a packed batch; gathered, the
shares must equal the whole batch computed in one process, and the timing
reduction must take the max over ranks and the sum of units.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from linear_attention_prefill_gb300.sharding import partition_sequences, rank_seed, reduce_timing


def test_partition_covers_every_sequence_once():
    lens = [512, 2048, 1000, 7, 0, 1999, 640, 1280, 3]
    for world in (1, 2, 3, 8, 16):
        parts = partition_sequences(lens, world)
        assert len(parts) == world
        flat = sorted(i for p in parts for i in p)
        assert flat == list(range(len(lens)))
    loads = [sum(lens[i] for i in p) for p in partition_sequences(lens, 2)]
    assert max(loads) - min(loads) <= max(lens)


def test_rank_seeds_differ():
    assert len({rank_seed(4, r) for r in range(8)}) == 8


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    from oracle import gdn_recurrent
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(0)
    lens = [5, 9, 3, 12, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    q_ = rng.standard_normal((1, T, 1, 6)); q_ /= np.linalg.norm(q_, axis=-1, keepdims=True)
    k_ = rng.standard_normal((1, T, 1, 6)); k_ /= np.linalg.norm(k_, axis=-1, keepdims=True)
    v_ = rng.standard_normal((1, T, 2, 4))
    g_ = -rng.random((1, T, 2))
    b_ = rng.random((1, T, 2))
    h0 = rng.standard_normal((5, 2, 6, 4))
    mine = partition_sequences(lens, world)[rank]
    res = {}
    for n in mine:
        a, b = cu[n], cu[n + 1]
        o, hT = gdn_recurrent(q_[:, a:b], k_[:, a:b], v_[:, a:b], g_[:, a:b], b_[:, a:b], 0.4,
                              h0[n:n + 1])
        res[n] = (o, hT)
    gathered = [None] * world
    dist.all_gather_object(gathered, res)
    ms, units = reduce_timing(1.0 + rank, float(sum(lens[n] for n in mine)))
    if rank == 0:
        o_all, h_all = gdn_recurrent(q_, k_, v_, g_, b_, 0.4, h0, cu)
        merged = {}
        for d in gathered:
            merged.update(d)
        ok = sorted(merged) == list(range(5))
        for n, (o, hT) in merged.items():
            ok &= np.allclose(o[0], o_all[0, cu[n]:cu[n + 1]], atol=1e-13)
            ok &= np.allclose(hT[0], h_all[n], atol=1e-13)
        q.put((ok, ms, units))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_gloo_shards_equal_whole_batch():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    ok, ms, units = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert ok
    assert ms == 2.0 and units == 30.0
