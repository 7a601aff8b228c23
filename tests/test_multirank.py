"""The N>1 paths on CPU with gloo, world size 2: replica batches reduced the way
bench.py reports them, and the exact merge of per-shard top-k lists for a row
whose pages are split across ranks (checked against the oracle)."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _replicas(rank, world, port, out):
    _init(rank, world, port)
    from sparse_attention_kv_e4m3_gb300 import synth

    w = synth.make_workload("rep", num_q=3, history=lambda g, n: g.integers(100, 500, size=n), seed=rank)
    keys = int(w.visible_counts().sum())
    ms = 1.0 + rank  # rank 1 is the slower one
    k_all, m_max = bench.reduce_over_ranks(keys, ms, dist, "cpu")
    out[rank] = (keys, k_all, m_max)
    dist.destroy_process_group()


def test_replica_reduction_gloo():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_replicas, args=(2, port, out), nprocs=2, join=True)
    assert out[0][1] == out[1][1] == out[0][0] + out[1][0]  # keys summed over ranks
    assert out[0][2] == out[1][2] == 2.0                     # time = the slowest rank


def _shards(rank, world, port, out):
    _init(rank, world, port)
    import torch

    from sparse_attention_kv_e4m3_gb300 import synth
    import oracle

    w = synth.make_workload("cp", num_q=1, history=[64 * 23 + 9], seed=5)
    npages = 24
    mine = np.arange(rank, npages, world, dtype=np.int32)   # this rank's pages
    shard = synth.Workload(name="cp_shard", q=w.q, fused_w=w.fused_w, kv=w.kv, page_table=w.page_table,
                           q_len=w.q_len, resident=mine.reshape(1, -1),
                           n_resident=np.array([len(mine)], dtype=np.int32))
    k = 100
    idx, _, lg, _ = oracle.topk(oracle.Problem(shard), k)
    t_idx = torch.from_numpy(idx[0].astype(np.int64))
    t_lg = torch.from_numpy(lg[0])
    g_idx = [torch.zeros_like(t_idx) for _ in range(world)]
    g_lg = [torch.zeros_like(t_lg) for _ in range(world)]
    dist.all_gather(g_idx, t_idx)
    dist.all_gather(g_lg, t_lg)
    merged, _ = bench.merge_shard_topk([(a.numpy(), b.numpy()) for a, b in zip(g_idx, g_lg)], k)
    full_idx = oracle.topk(oracle.Problem(w), k)[0][0]
    out[rank] = bool(np.array_equal(merged, full_idx))
    dist.destroy_process_group()


def test_context_parallel_merge_gloo():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_shards, args=(2, port, out), nprocs=2, join=True)
    assert out[0] and out[1]
