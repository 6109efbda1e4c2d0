"""The multi-GPU path on CPU: two gloo ranks run the replica bookkeeping the
benchmark uses (balanced shards, slowest-rank time, whole-job throughput), and
each rank runs the oracle on its own shard; the shards reassemble the
single-process result exactly (tokens are independent, so sharding by whole
sequences changes nothing)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from hashed_gram_memory_gb300.replicas import shard_range, whole_job_throughput


def test_shard_range_partitions_exactly():
    for n in (0, 1, 7, 64, 65, 1000):
        for world in (1, 2, 3, 8):
            got = [shard_range(n, r, world) for r in range(world)]
            assert got[0][0] == 0 and got[-1][1] == n
            for (a, b), (c, d) in zip(got, got[1:]):
                assert b == c
            sizes = [b - a for a, b in got]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_range(5, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import oracle
    import workloads as W
    from hashed_gram_memory_gb300.replicas import max_over_ranks, shard_range, sum_over_ranks
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    cfg = W.by_name("tiny_fp8_d256").scaled(B=5, S=24)
    ids = W.token_ids(cfg)
    b0, b1 = shard_range(cfg.B, rank, world)
    e, _ = oracle.compress(ids[b0:b1], W.tid2eid(cfg), cfg.n_eids)
    rows, _ = oracle.hash_ids(e, cfg.H, cfg.rows)
    slowest = max_over_ranks(1.0 + rank)          # per-rank "step time"
    tokens = sum_over_ranks(rows.shape[0] * rows.shape[1])
    dist.barrier()
    out[rank] = (b0, b1, rows.tobytes(), slowest, tokens)
    dist.destroy_process_group()


def test_two_gloo_ranks_reassemble_the_batch():
    import oracle
    import workloads as W
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()   # no fork of this (threaded) process
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    cfg = W.by_name("tiny_fp8_d256").scaled(B=5, S=24)
    e, _ = oracle.compress(W.token_ids(cfg), W.tid2eid(cfg), cfg.n_eids)
    full, _ = oracle.hash_ids(e, cfg.H, cfg.rows)
    parts = []
    for r in range(world):
        b0, b1, raw, slowest, tokens = out[r]
        parts.append(np.frombuffer(raw, np.int32).reshape(b1 - b0, cfg.S, 3, cfg.H))
        assert slowest == 2.0 and tokens == cfg.T
    assert np.array_equal(np.concatenate(parts), full)
    assert whole_job_throughput(2 * cfg.T, 0.5) == 4 * cfg.T
