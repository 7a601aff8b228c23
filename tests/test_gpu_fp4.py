"""The MXFP4 indexer (record_format = CSA_RECORD_MXFP4) against the oracle.

68-byte records (64 bytes of e2m1 codes, then the UE8M0 scales of the four
32-element blocks) and a query MXFP4-rounded per head (the published model
FP4-rounds the index key and query alike: the BatchGen #153 commit log's indexer
quantisation notes, "DeepSeek-V4.1 native paged runtime"; the block format is the
OCP MXFP4 reading the oracle states). The kernel converts each record and query
block to e4m3 exactly while the block exponents of a record (or of a head) span at
most 14, so scores are held to the same bars as the e4m3 path.
"""
import numpy as np
import pytest
import torch

import _parity
import oracle
from sparse_attention_kv_e4m3_gb300 import native, synth

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_kv_e4m3_gb300 import build

    build.build()
    native.load()


def fp4(w, seed=7):
    return synth.mxfp4_cache(w, seed)


def run(w, k, unfused=True):
    prob = native.Problem.from_workload(w)
    assert prob.record_format == native.RECORD_MXFP4
    out = {"scores": native.csa_index_score(prob)}
    out["idx"], out["vals"] = native.csa_index_score_topk_fused(prob, k)
    if unfused:
        out["tidx"], out["tvals"] = native.csa_index_topk(out["scores"], prob, k)
    torch.cuda.synchronize()
    out = {a: v.cpu().numpy() for a, v in out.items()}
    out["status"] = int(prob.dev_status.item())
    return out


def check_all(w, k, score_rows=None, unfused=True):
    r = run(w, k, unfused)
    assert r["status"] == 0, r["status"]
    _parity.check_scores(w, r["scores"], rows=score_rows)
    ora = oracle.topk(oracle.Problem(w), k)
    _parity.check_topk(w, r["idx"], r["vals"], k, oracle_result=ora)
    if unfused:
        _parity.check_topk(w, r["tidx"], r["tvals"], k, ranked_by_logit=False, oracle_result=ora)
    return r


def test_every_code_at_every_block_offset():
    """Record i holds code i % 16 in every element of block (i // 16) % 4, the
    other blocks zero, that block's exponent i // 64 (0..14) below the record's
    largest: each record's logit is the code's value times its block scale times
    the block's summed query (heads 0 and 1: q = +1 and -1), which the conversion
    to e4m3 must keep exactly, subnormal e4m3 values included."""
    n = 16 * 4 * 15
    recs = np.zeros((n, 68), dtype=np.uint8)
    for i in range(n):
        code, blk, span = i % 16, (i // 16) % 4, i // 64
        recs[i, 16 * blk: 16 * blk + 16] = code | (code << 4)
        recs[i, 64:68] = 127 + 3          # block scales 2^3 ...
        recs[i, 64 + blk] = 127 + 3 - span  # ... and the coded block 2^-span below them
    page = 64 * 68
    pages = (n + 63) // 64
    kv = np.zeros((pages, page), dtype=np.uint8)
    kv.reshape(-1)[: n * 68] = recs.reshape(-1)
    q = np.zeros((1, 64, D), dtype=np.float32)
    q[0, 0, :] = 1.0      # block-rounded exactly: 1.0 = 4 * 2^-2
    q[0, 1, :] = -1.0
    wv = np.zeros((1, 64), dtype=np.float32)
    wv[0, 0], wv[0, 1] = 2.0 ** -8, -(2.0 ** -8)
    from _pins import bf16_bits

    w = synth.Workload(name="fp4codes", q=bf16_bits(q), fused_w=wv, kv=kv,
                       page_table=np.arange(pages, dtype=np.int32).reshape(1, -1),
                       q_len=np.array([n], dtype=np.int32), record_format="mxfp4")
    prob = native.Problem.from_workload(w)
    lg = native.csa_index_logits(prob).cpu().numpy()[0, :n].astype(np.float64)
    torch.cuda.synchronize()
    assert int(prob.dev_status.item()) == 0
    o, valid, _ = oracle.logits(oracle.Problem(w), lg.shape[0])
    assert np.array_equal(lg, o[0, :n]), np.argmax(np.abs(lg - o[0, :n]))
    # and the exact value: 32 elements of code c, times 2^(3 - span), times sum(q) = 32, relu'd and weighted
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6] * 2) * np.repeat([1, -1], 8)
    want = np.array([max(vals[i % 16] * 2.0 ** (3 - i // 64) * 32, 0) * 2.0 ** -8
                     + max(-vals[i % 16] * 2.0 ** (3 - i // 64) * 32, 0) * -(2.0 ** -8) for i in range(n)])
    assert np.array_equal(lg, want)


SMALL = {
    "ragged_multi_tile": dict(num_q=5, history=[3000, 1000, 129, 64, 1], seed=31),
    "resident_partial_tail": dict(num_q=3, history=[64 * 40 + 17, 64 * 9, 64 * 30], resident_pages=7, seed=33),
    "prefill_rows": dict(num_q=40, history=[3000], single_request=True,
                         q_len=lambda h, n: np.minimum(3000, np.arange(n) * 70 + 1), seed=34),
    "charged_split": dict(num_q=7, history=[20000, 0, 256, 0, 50000, 64, 4096], seed=37),
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("k", [40, 512])
def test_small_workloads(name, k):
    check_all(fp4(synth.make_workload(name, **SMALL[name])), k)


def test_query_rounding_spans_the_block_exponents():
    """Query heads whose blocks differ by up to 10 binades (plus the blocks' own
    spread), and a block whose elements sit on the e2m1 midpoints (ties to the even
    code): the rounding matches the oracle and one e4m3 term stays exact."""
    w = fp4(synth.make_workload("fp4q", num_q=2, history=[700, 300], seed=41))
    rng = np.random.default_rng(9)
    qf = rng.standard_normal((2, 64, D)).astype(np.float32)
    qf *= np.float32(2.0) ** rng.integers(-5, 6, size=(2, 64, 4, 1)).repeat(32, axis=3).reshape(2, 64, D)
    qf[0, 3, :32] = 0.0  # block 0 of head 3: amax 5 gives the block scale 1, so these are the midpoints
    qf[0, 3, :8] = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 4.5], dtype=np.float32)
    from _pins import bf16_bits

    w.q[:] = bf16_bits(qf)
    check_all(w, 64)


@pytest.mark.parametrize("name", ["tiny_decode", "decode_batch", "long_ragged_decode", "resident_1m",
                                  "prefill_chunk"])
def test_named_workload(name):
    w = fp4(synth.config(name))
    rows = None if w.num_q <= 64 else list(range(0, w.num_q, 97)) + [w.num_q - 1]
    if w.num_q > 64:  # the oracle on a sample of rows for the 4096-row batch
        r = run(w, 512, unfused=False)
        assert r["status"] == 0
        _parity.check_scores(w, r["scores"], rows=rows)
        sub = synth.Workload(name="fp4_rows", q=w.q[rows], fused_w=w.fused_w[rows], kv=w.kv,
                             page_table=w.page_table, q_len=w.q_len[rows], q_req=w.q_req[rows],
                             record_format="mxfp4")
        _parity.check_topk(sub, r["idx"][rows], r["vals"][rows], 512)
    else:
        check_all(w, 512, score_rows=rows)


def test_wide_block_span_and_nan_scale_are_flagged():
    w = fp4(synth.make_workload("fp4bad", num_q=1, history=[640], seed=43))
    recs = w.kv.reshape(w.kv.shape[0], 64, 68)

    def rec(pos):  # the record of logical position pos (the page table is shuffled)
        return recs[w.page_table[0, pos // 64], pos % 64]

    rec(5)[64:68] = [127, 127, 127, 100]   # a block 27 binades below the record's largest
    rec(9)[64:68] = [127, 255, 127, 127]   # a NaN scale byte: the record is left out
    prob = native.Problem.from_workload(w)
    idx, _ = native.csa_index_score_topk_fused(prob, 512)
    sc = native.csa_index_score(prob)
    torch.cuda.synchronize()
    assert int(prob.dev_status.item()) & 4  # CSA_DEV_RANGE
    assert 9 not in set(idx.cpu().numpy()[0].tolist())
    assert np.isnan(sc.cpu().numpy()[0, 9])


def test_fp4_rejects_128_heads_and_short_pages():
    import ctypes

    w = fp4(synth.make_workload("fp4args", num_q=1, history=[64], seed=44))
    prob = native.Problem.from_workload(w)
    lib = native.load()
    ws = native.alloc_workspace(prob, 8)
    a = prob.args()
    a.page_stride_bytes = 4336  # less than 64 records of 68 bytes
    assert lib.csa_index_score_topk_fused(ctypes.byref(a), 8, 0x1000, 0x2000, ws.data_ptr(), ws.numel(), None) == 1
    a = prob.args()
    a.num_heads = 128  # MXFP4 records: the 64-head indexer only
    assert lib.csa_index_score(ctypes.byref(a), 0x1000, 256, None) == 2
    a = prob.args()
    a.record_format = 2
    assert lib.csa_index_score(ctypes.byref(a), 0x1000, 256, None) == 1
