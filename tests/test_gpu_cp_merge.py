"""csa_index_merge_topk: the exact merge of G per-shard top-k lists on the device.

Context-parallel scoring splits one request's pages across G GPUs; each shard
returns its rows' local top-k and the lists are gathered to one device ("Two-
level recall algorithm", Level 2: the top-512 over the scored history). Here the
shards are resident page subsets scored by the fused path on this one GPU, and
their lists are merged by the new entry point; the result must be the oracle's
top-k of the whole history (band rule), and on random lists it must equal a
plain sort of their union exactly.
"""
import os
import socket

import numpy as np
import pytest
import torch

import _parity
import bench
from sparse_attention_kv_e4m3_gb300 import native, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_kv_e4m3_gb300 import build

    build.build()
    native.load()


@pytest.mark.parametrize("g,nq,k_in,k", [(2, 3, 512, 512), (8, 5, 512, 512), (3, 4, 100, 40), (6, 2, 1024, 1024),
                                         (1, 3, 64, 128)])
def test_equals_a_sort_of_the_union(g, nq, k_in, k):
    rng = np.random.default_rng(g * 100 + k_in)
    idx = np.full((g, nq, k_in), -1, dtype=np.int32)
    vals = np.zeros((g, nq, k_in), dtype=np.float32)
    for b in range(nq):
        pos = rng.permutation(200000)[: g * k_in].reshape(g, k_in).astype(np.int32)
        v = rng.standard_normal((g, k_in)).astype(np.float32)
        v[:, ::7] = np.round(v[:, ::7], 1)  # ties in value: broken by position
        fill = rng.integers(k_in // 2, k_in + 1, size=g)  # some lists padded
        for s in range(g):
            idx[s, b, : fill[s]] = pos[s, : fill[s]]
            vals[s, b, : fill[s]] = v[s, : fill[s]]
    oi, ov = native.csa_index_merge_topk(torch.from_numpy(idx).cuda(), torch.from_numpy(vals).cuda(), k)
    torch.cuda.synchronize()
    oi, ov = oi.cpu().numpy(), ov.cpu().numpy()
    for b in range(nq):
        want_p, want_v = bench.merge_shard_topk([(idx[s, b], vals[s, b]) for s in range(g)], k)
        assert np.array_equal(oi[b], want_p.astype(np.int32)), b
        got_v = np.where(oi[b] >= 0, ov[b], -np.inf)
        assert np.array_equal(got_v.astype(np.float64), want_v), b


def _shard_workload(w, shard: int, count: int) -> synth.Workload:
    """The pages of every request that shard `shard` of `count` holds (every count-th page)."""
    lens = np.asarray(w.q_len)
    pages = [np.arange(shard, (int(L) + 63) // 64, count, dtype=np.int32) for L in lens]
    stride = max(1, max(len(p) for p in pages))
    res = np.full((w.num_req, stride), -1, dtype=np.int32)
    for r, p in enumerate(pages):
        res[r, : len(p)] = p
    return synth.Workload(name=f"{w.name}_shard{shard}", q=w.q, fused_w=w.fused_w, kv=w.kv, page_table=w.page_table,
                          q_len=w.q_len, q_req=w.q_req, resident=res,
                          n_resident=np.array([len(p) for p in pages], dtype=np.int32))


@pytest.mark.parametrize("count", [2, 4])
def test_context_parallel_shards_merge_to_the_whole_history(count):
    k = 512
    w = synth.make_workload("cpw", num_q=3, history=[40000, 9000, 70000], outlier_frac=0.05, seed=81)
    lists_i, lists_v = [], []
    for s in range(count):
        prob = native.Problem.from_workload(_shard_workload(w, s, count))
        i, v = native.csa_index_score_topk_fused(prob, k)
        torch.cuda.synchronize()
        assert int(prob.dev_status.item()) == 0
        lists_i.append(i)
        lists_v.append(v)
    oi, ov = native.csa_index_merge_topk(torch.stack(lists_i), torch.stack(lists_v), k)
    torch.cuda.synchronize()
    _parity.check_topk(w, oi.cpu().numpy(), ov.cpu().numpy(), k, ranked_by_logit=False)
    # and the same set as the single-device fused call, but for ties in the scores
    full_i, _ = native.csa_index_score_topk_fused(native.Problem.from_workload(w), k)
    a, b = oi.cpu().numpy(), full_i.cpu().numpy()
    for r in range(w.num_q):
        assert len(set(a[r]) ^ set(b[r])) <= 8, r


# ------------------------------------------------------------------ two ranks (gloo), one GPU

def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from sparse_attention_kv_e4m3_gb300 import native as nat, synth as syn

    nat.load()
    k = 256
    w = syn.make_workload("cpg", num_q=2, history=[30000, 12000], seed=83)
    prob = nat.Problem.from_workload(_shard_workload(w, rank, world))
    i, v = nat.csa_index_score_topk_fused(prob, k)
    torch.cuda.synchronize()
    gi = [torch.zeros_like(i.cpu()) for _ in range(world)]
    gv = [torch.zeros_like(v.cpu()) for _ in range(world)]
    dist.all_gather(gi, i.cpu())
    dist.all_gather(gv, v.cpu())
    if rank == 0:
        oi, ov = nat.csa_index_merge_topk(torch.stack(gi).cuda(), torch.stack(gv).cuda(), k)
        torch.cuda.synchronize()
        try:
            _parity.check_topk(w, oi.cpu().numpy(), ov.cpu().numpy(), k, ranked_by_logit=False)
            out[0] = "ok"
        except AssertionError as e:
            out[0] = str(e)
    dist.destroy_process_group()


def test_two_ranks_gather_and_merge_on_the_device():
    """The N>1 exchange step as a run would do it: each rank scores its shard,
    the lists are all-gathered (gloo here, on host copies) and rank 0 merges them
    on its GPU. Both ranks share this one GPU; their kernels never wait on each
    other."""
    import torch.multiprocessing as mp

    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()  # no fork after CUDA is initialised here
    mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == "ok", out[0]
