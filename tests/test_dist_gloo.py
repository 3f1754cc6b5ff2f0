"""Multi-rank host logic on CPU (gloo, world size 2): sequence sharding and meter-count reduction.

The decode path needs no collective (sequences are independent); these tests
cover what ranks do share: a deterministic, balanced assignment of sequences
and the host-side sum of the meter counters.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from quantized_kv_cache_kvq_gb300.dist import reduce_meter_counts, shard_sequences


def test_shard_sequences_partition_and_balance():
    rng = np.random.default_rng(3)
    lens = np.floor(np.exp(rng.uniform(np.log(1024), np.log(131072), 128))).astype(int)
    for ws in (1, 2, 4, 8):
        shards = shard_sequences(lens, ws, prefix_len=632)
        allidx = np.sort(np.concatenate(shards))
        assert np.array_equal(allidx, np.arange(128))               # a partition
        loads = [int((lens[s] + 632).sum()) for s in shards]
        assert max(loads) - min(loads) <= int(lens.max()) + 632     # greedy bound
        again = shard_sequences(lens, ws, prefix_len=632)
        assert all(np.array_equal(a, b) for a, b in zip(shards, again))  # deterministic


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    lens = np.arange(1, 17) * 100
    mine = shard_sequences(lens, world)[rank]
    # each rank's counters: covered = its sequences with even index, cells = its sequences * 32 heads
    counts = [int(np.sum(mine % 2 == 0)), 0, rank, len(mine) * 32]
    tot = reduce_meter_counts(counts)
    q.put((rank, mine.tolist(), tot.tolist()))
    dist.destroy_process_group()


def test_two_rank_gloo_reduce():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    shards = [r[1] for r in res]
    assert sorted(shards[0] + shards[1]) == list(range(16))
    for _, _, tot in res:
        assert tot == [8, 0, 1, 16 * 32]


def _bench_rank(rank, world, port, q):
    """One rank of bench.py's multi-GPU path, host side: its share of the global batch and the job totals."""
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = bench.W.WORKLOADS["ragged_paged"]
    wr, lens, idx = bench.rank_share(w, rank, world)
    step = bench.step_bytes(wr, lens)
    counts = [rank, 0, 0, int(wr.batch) * w.n_layers * w.n_q_heads]
    (tot_bytes, tot_tokens), tot_counts = bench.job_totals([step, float(lens.sum())], counts, world)
    q.put((rank, idx.tolist(), step, tot_bytes, tot_tokens, tot_counts))
    dist.destroy_process_group()


def test_two_rank_bench_path():
    """bench.py --gpus 2 on CPU ranks: the global batch is split by shard_sequences, the step bytes and meter
    counters are summed over the ranks, and the totals equal those of the whole global batch."""
    import bench

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_bench_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = bench.W.WORKLOADS["ragged_paged"]
    wg = bench.W.reduced(w, batch=2 * w.batch)
    lens_g = bench.W.seq_lengths(wg)
    assert sorted(res[0][1] + res[1][1]) == list(range(2 * w.batch))
    for _, _, _, tot_bytes, tot_tokens, tot_counts in res:
        assert tot_bytes == res[0][2] + res[1][2] == bench.step_bytes(wg, lens_g)
        assert tot_tokens == float(lens_g.sum())
        assert tot_counts == [1, 0, 0, 2 * w.batch * w.n_layers * w.n_q_heads]
