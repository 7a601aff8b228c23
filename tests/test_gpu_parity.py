"""CUDA path vs the oracle, through the C ABI, on seeded inputs."""
import struct

import numpy as np
import pytest
import torch

import _parity
import _pins
import oracle
from sparse_attention_kv_e4m3_gb300 import native, synth

pytestmark = pytest.mark.gpu
PAGE, REC, D = 64, 132, 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_kv_e4m3_gb300 import build

    build.build()
    native.load()


def run(w, k, score=True, unfused=True):
    prob = native.Problem.from_workload(w)
    out = {"prob": prob}
    if score:
        out["scores"] = native.csa_index_score(prob)
    out["idx"], out["vals"] = native.csa_index_score_topk_fused(prob, k)
    if unfused:
        sc = out["scores"] if score else native.csa_index_score(prob)
        out["tidx"], out["tvals"] = native.csa_index_topk(sc, prob, k)
    torch.cuda.synchronize()
    out = {k2: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k2, v in out.items()}
    out["status"] = int(prob.dev_status.item())
    return out


def check_all(w, k, score_rows=None):
    r = run(w, k)
    assert r["status"] == 0, r["status"]
    _parity.check_scores(w, r["scores"], rows=score_rows)
    ora = oracle.topk(oracle.Problem(w), k)
    _parity.check_topk(w, r["idx"], r["vals"], k, oracle_result=ora)
    _parity.check_topk(w, r["tidx"], r["tvals"], k, ranked_by_logit=False, oracle_result=ora)
    return r


# ------------------------------------------------------------------ exact arithmetic

def test_every_e4m3_byte_through_the_tensor_core():
    """Record i holds byte i at d = i % 128 (NaN codes left out). Head 0 reads
    q = +1, head 1 q = -1, w = (2^-6, -2^-6): logit = 2^-6 * e4m3(byte) exactly,
    subnormals included."""
    codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
    recs = np.stack([_pins.record({i % D: c}, 1.0) for i, c in enumerate(codes)])
    q = np.zeros((64, D), dtype=np.float32)
    q[0, :] = 1.0
    q[1, :] = -1.0
    wv = np.zeros(64, dtype=np.float32)
    wv[0], wv[1] = 2.0 ** -6, -(2.0 ** -6)
    w = _pins.hand_workload(recs, q, wv)
    r = run(w, len(codes))
    assert r["status"] == 0
    table = {c: oracle.e4m3(c) for c in codes}
    want = _parity.sigmoid(np.array([table[c] * 2.0 ** -6 for c in codes]))
    got = r["scores"][0, : len(codes)].astype(np.float64)
    assert np.max(np.abs(got - want)) <= 1e-6, np.argmax(np.abs(got - want))
    _parity.check_topk(w, r["idx"], r["vals"], len(codes))


def test_query_split_is_exact_for_large_dynamic_range():
    """q rows mixing magnitudes from 2^-20 to 2^20 (per-head scaling)."""
    w = synth.make_workload("dyn", num_q=2, history=[300, 200], seed=21)
    rng = np.random.default_rng(3)
    qf = rng.standard_normal((2, 64, D)).astype(np.float32)
    qf *= np.float32(2.0) ** rng.integers(-20, 21, size=(2, 64, 1)).astype(np.float32)
    w.q[:] = _pins.bf16_bits(qf)
    w.fused_w[:] *= np.float32(2.0) ** rng.integers(-6, 7, size=(2, 64)).astype(np.float32)
    check_all(w, 100)


def test_query_heads_at_the_bottom_of_bf16():
    """Heads whose largest |q| lies between bf16's smallest subnormal (2^-133)
    and 2^-126: their power-of-two scale exceeds 2^126 (two factors in the
    kernel) and the folded weight 2^-e is an fp32 subnormal. With weights of
    2^100 the logits are of order 2^-20; they must match the oracle to fp32
    accumulation accuracy, which a split that lost the small heads' low bits
    (or their subnormal elements) would not."""
    w = synth.make_workload("tinyq", num_q=2, history=[300, 200], seed=22)
    rng = np.random.default_rng(5)
    qf = rng.standard_normal((2, 64, D)).astype(np.float64)
    top = rng.integers(-133, -125, size=(2, 64, 1)).astype(np.float64)  # each head's largest |q|: 2^top
    qf = qf / np.abs(qf).max(axis=2, keepdims=True) * 2.0 ** top
    qf[0, 0, :] = 0.0
    qf[0, 0, 5] = 2.0 ** -133  # one head holding a single smallest subnormal
    w.q[:] = _pins.bf16_bits(qf.astype(np.float32))
    w.fused_w[:] = np.float32(2.0 ** 100) * np.sign(rng.standard_normal((2, 64))).astype(np.float32)
    prob = native.Problem.from_workload(w)
    lg = native.csa_index_logits(prob).cpu().numpy().astype(np.float64)
    torch.cuda.synchronize()
    assert int(prob.dev_status.item()) == 0
    o_lg, valid, _ = oracle.logits(oracle.Problem(w), lg.shape[1])
    for b in range(w.num_q):
        v = valid[b]
        ref = o_lg[b, v]
        scale = np.abs(ref).max()
        assert scale > 2.0 ** -40, "the test must produce visible logits"
        assert np.max(np.abs(lg[b, v] - ref)) <= 2.0 ** -16 * scale, np.max(np.abs(lg[b, v] - ref)) / scale
    r = run(w, 64, score=False, unfused=False)
    _parity.check_topk(w, r["idx"], r["vals"], 64)


# ------------------------------------------------------------------ small workloads

SMALL = {
    "ragged_multi_tile": dict(num_q=5, history=[3000, 1000, 129, 64, 1], seed=31),
    "outliers": dict(num_q=3, history=[5000, 2600, 777], outlier_frac=0.05, seed=32),
    "resident_partial_tail": dict(num_q=3, history=[64 * 40 + 17, 64 * 9, 64 * 30], resident_pages=7, seed=33),
    "prefill_rows": dict(num_q=40, history=[3000], single_request=True,
                         q_len=lambda h, n: np.minimum(3000, np.arange(n) * 70 + 1), seed=34),
    "padded_pages": dict(num_q=2, history=[1500, 900], page_pad=112, seed=35),
    "contiguous": dict(num_q=2, history=[4096, 4000], shuffle=False, seed=36),
    # long rows on average (the plan charges each row start extra tiles) mixed with
    # empty and one-tile rows, so that some CTA ranges hold only a row's charge
    "charged_split": dict(num_q=7, history=[20000, 0, 256, 0, 50000, 64, 4096], seed=37),
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("k", [40, 512])
def test_small_workloads(name, k):
    check_all(synth.make_workload(name, **SMALL[name]), k)


def test_tiny_pin_workloads():
    for w in _pins.tiny_workloads():
        check_all(w, 64)


def test_k_extremes():
    w = synth.make_workload("kx", num_q=3, history=[9000, 1030, 5], seed=37)
    for k in (1, 2, 1023, 1024):
        check_all(w, k)


def test_zero_weights_rank_by_position():
    w = synth.make_workload("zw", num_q=2, history=[2000, 300], seed=38)
    w.fused_w[:] = 0.0
    r = run(w, 512)
    assert r["status"] == 0
    assert np.array_equal(r["idx"][0], np.arange(512))
    assert np.array_equal(r["idx"][1], np.concatenate([np.arange(300), -np.ones(212, dtype=np.int64)]))
    assert np.all(r["vals"][0] == 0.5) and np.all(r["scores"][0, :2000] == 0.5)
    assert np.array_equal(r["tidx"], r["idx"])


def test_negative_and_zero_scales():
    w = synth.make_workload("neg", num_q=2, history=[700, 400], seed=39)
    recs = w.kv[:, : PAGE * REC].reshape(-1, REC)
    sc = recs[:, D:].copy().view("<f4").reshape(-1)
    rng = np.random.default_rng(5)
    sc[rng.random(sc.shape[0]) < 0.3] *= -1.0
    sc[rng.random(sc.shape[0]) < 0.05] = 0.0
    recs[:, D:] = sc.view(np.uint8).reshape(-1, 4)
    check_all(w, 128)


def test_empty_rows_and_padding():
    w = synth.make_workload("empty", num_q=4, history=[0, 10, 0, 600], seed=40)
    r = check_all(w, 64)
    assert np.all(r["idx"][0] == -1) and np.all(r["vals"][0] == 0.0)
    assert np.all(r["idx"][1, 10:] == -1)


def test_all_rows_empty():
    w = synth.make_workload("allempty", num_q=3, history=[64, 64, 64], seed=41, q_len=lambda h, n: np.zeros(n))
    r = run(w, 16)
    assert r["status"] == 0 and np.all(r["idx"] == -1) and np.all(r["vals"] == 0.0)
    assert np.all(np.isnan(r["scores"]))


def test_more_rows_than_sms():
    w = synth.make_workload("many", num_q=700, history=[300], single_request=True,
                            q_len=lambda h, n: 1 + (np.arange(n) * 37) % 300, seed=42)
    check_all(w, 32)


# Batches of 512 rows and more take the short-row scorer: a whole row inside a CTA
# that fits its candidate buffer (up to 2048 records) is written to its slot uncut
# and the merge cuts it. The rows here hold 1024..2047 visible records, more than
# a cut segment keeps, and the mixed batch adds long rows split across CTAs.
SHORT_ROWS = {
    "prefill_like": dict(num_q=600, history=[2100], single_request=True,
                         q_len=lambda h, n: 1024 + (np.arange(n) * 97) % 1024, seed=43),
    "mixed_long": dict(num_q=560, history=lambda rng, n: np.where(np.arange(n) % 70 == 0, 30000, 1800),
                       q_len=lambda h, n: np.where(np.arange(n) % 70 == 0, h, 700 + (np.arange(n) * 53) % 1100),
                       seed=44),
    # resident mode: rows of up to 30 resident pages of a longer history (whole rows in a CTA,
    # written uncut through the selector)
    "resident_short": dict(num_q=520, history=lambda rng, n: np.full(n, 64 * 40), resident_pages=30, seed=45),
}


@pytest.mark.parametrize("name", sorted(SHORT_ROWS))
@pytest.mark.parametrize("k", [40, 512])
def test_short_row_scorer(name, k):
    w = synth.make_workload(name, **SHORT_ROWS[name])
    assert w.num_q >= 512
    r = run(w, k, score=False, unfused=False)
    assert r["status"] == 0, r["status"]
    _parity.check_topk(w, r["idx"], r["vals"], k)


def test_short_row_scorer_edges():
    """Exactly 512 rows (the short-row scorer's threshold): empty rows, rows shorter
    than k (padding), rows of exactly four tiles (the whole buffer), and a page out
    of range inside a short row (flagged; its records left out, the rest ranked)."""
    lens = np.array([0, 5, 2048, 2047, 1, 513, 1536, 700] * 64)
    w = synth.make_workload("edges512", num_q=512, history=lambda rng, n: np.full(n, 2048),
                            q_len=lambda h, n: lens[:n], seed=46)
    w.page_table[10, 20] = w.num_pages + 1  # row 10: 2048 records, one page out of range
    r = run(w, 512, score=False, unfused=False)
    assert r["status"] & native.DEV_PAGE_OOB
    assert np.all(r["idx"][0] == -1) and np.all(r["vals"][0] == 0.0)
    assert np.all(r["idx"][1, 5:] == -1)
    _parity.check_topk(w, r["idx"], r["vals"], 512)


def test_invalid_geometry_is_flagged_not_fatal():
    w = synth.make_workload("bad", num_q=4, history=[900, 900, 900, 900], seed=43)
    w.page_table[0, 2] = w.num_pages + 3      # page out of range
    w.page_table[1, 0] = -1
    w.q_len[2] = -5                           # negative length
    r = run(w, 128)
    assert r["status"] & native.DEV_PAGE_OOB and r["status"] & native.DEV_LEN_OOB
    _parity.check_scores(w, r["scores"])
    _parity.check_topk(w, r["idx"], r["vals"], 128)
    _parity.check_topk(w, r["tidx"], r["tvals"], 128, ranked_by_logit=False)
    # a request id out of range: the row is empty
    w2 = synth.make_workload("badreq", num_q=2, history=[300], single_request=True, seed=44)
    w2.q_req[1] = 9
    r2 = run(w2, 32)
    assert r2["status"] & native.DEV_BAD_REQUEST and np.all(r2["idx"][1] == -1)
    # resident page past the row's length
    w3 = synth.make_workload("badres", num_q=1, history=[640], resident_pages=4, seed=45)
    w3.resident[0, 1] = 10
    r3 = run(w3, 64)
    assert r3["status"] & native.DEV_RESIDENT_OOB
    _parity.check_topk(w3, r3["idx"], r3["vals"], 64)


def test_deterministic():
    w = synth.make_workload("det", num_q=6, history=[20000, 7000, 300, 64, 12000, 9000], seed=46)
    a, b = run(w, 512), run(w, 512)
    for key in ("idx", "vals", "tidx", "tvals"):
        assert np.array_equal(a[key], b[key]), key
    assert np.array_equal(a["scores"], b["scores"], equal_nan=True)


def test_prepared_call_repeats_the_plain_call():
    """native.PreparedFused marshals the arguments once; each call (plain or with
    the event between the kernels) must write what the plain binding writes,
    also after the inputs' contents change in place between calls."""
    w = synth.make_workload("prep", num_q=5, history=[9000, 300, 0, 20000, 4100], seed=49)
    prob = native.Problem.from_workload(w)
    ws = native.alloc_workspace(prob, 256, "cuda")
    idx = torch.empty((5, 256), dtype=torch.int32, device="cuda")
    vals = torch.empty((5, 256), dtype=torch.float32, device="cuda")
    call = native.PreparedFused(prob, 256, ws, idx, vals)
    for step in range(3):
        if step == 2:  # new lengths in the same buffer
            prob.q_len.copy_(torch.tensor([4000, 200, 0, 19000, 4100], dtype=torch.int32))
        want_i, want_v = native.csa_index_score_topk_fused(prob, 256)
        idx.fill_(7)
        vals.fill_(7.0)
        call(mark=torch.cuda.Event(enable_timing=True) if step == 1 else None)
        torch.cuda.synchronize()
        assert torch.equal(idx, want_i) and torch.equal(vals, want_v), step
    assert int(prob.dev_status.item()) == 0
    with pytest.raises(ValueError):
        native.PreparedFused(prob, 128, ws, idx, vals)


def test_dev_status_optional():
    w = synth.make_workload("nostat", num_q=1, history=[500], seed=47)
    prob = native.Problem.from_workload(w, dev_status=False)
    idx, vals = native.csa_index_score_topk_fused(prob, 32)
    torch.cuda.synchronize()
    _parity.check_topk(w, idx.cpu().numpy(), vals.cpu().numpy(), 32)


def test_misaligned_device_pointer_rejected():
    w = synth.make_workload("mis", num_q=1, history=[100], seed=48)
    prob = native.Problem.from_workload(w)
    raw = torch.empty(prob.kv.numel() + 16, dtype=torch.uint8, device="cuda")
    prob.kv = raw[4: 4 + prob.kv.numel()].view(prob.kv.shape)
    with pytest.raises(native.CsaError) as e:
        native.csa_index_score_topk_fused(prob, 8)
    assert e.value.status == 3


# ------------------------------------------------------------------ the five named workloads

@pytest.mark.parametrize("name", ["tiny_decode", "decode_batch", "long_ragged_decode", "resident_1m",
                                  "prefill_chunk"])
def test_named_workload(name):
    w = synth.config(name)
    rows = None if w.num_q <= 64 else list(range(0, w.num_q, 97)) + [w.num_q - 1]
    check_all(w, 512, score_rows=rows)


def test_prefill_chunk_tail_reading():
    w = synth.config("prefill_chunk_tail")
    r = run(w, 512, score=False, unfused=False)
    assert r["status"] == 0
    # oracle on a sample of rows (each row sees 15361..16384 records)
    rows = list(range(0, w.num_q, 257)) + [w.num_q - 1]
    sub = synth.Workload(name="tail_rows", q=w.q[rows], fused_w=w.fused_w[rows], kv=w.kv,
                         page_table=w.page_table, q_len=w.q_len[rows], q_req=w.q_req[rows])
    _parity.check_topk(sub, r["idx"][rows], r["vals"][rows], 512)
