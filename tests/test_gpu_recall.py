"""Level-1 recall and the raw-logit scorer on the GPU, through the C ABI, against
the oracle (FlashMemory-DeepSeek-V4, "Two-level recall algorithm", Level 1, and
"Joint checkpoint + ensemble").

The combined scores are floating point: within the strict score bar. The keep
decision is an integer the kernel takes in fp32: it must follow from the GPU's
own scores exactly, and may differ from the oracle's only for chunks whose
oracle score lies within the score bar of the threshold. The page lists must be
exactly the pages of the GPU's kept chunks."""
import dataclasses

import numpy as np
import pytest
import torch

import _parity
import _pins
import oracle
from sparse_attention_kv_e4m3_gb300 import native, synth

pytestmark = pytest.mark.gpu
PAGE = 64
TOL = _parity.STRICT_SCORE_TOL


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_kv_e4m3_gb300 import build

    build.build()
    native.load()


def _dev(w):
    return torch.from_numpy(w.q.view("int16")).cuda().view(torch.bfloat16), torch.from_numpy(w.fused_w).cuda()


def gpu_layers(layers):
    """Device Problems; layers that share a cache (synth.level1_layers) share its copy."""
    p0 = native.Problem.from_workload(layers[0])
    out = [p0]
    for w in layers[1:]:
        if w.kv is layers[0].kv and w.page_table is layers[0].page_table:
            q, fw = _dev(w)
            out.append(dataclasses.replace(p0, q=q, fused_w=fw, dev_status=None))
        else:
            out.append(native.Problem.from_workload(w))
    return out


def row_length(w, b):
    req = b if w.q_req is None else int(w.q_req[b])
    if req < 0 or req >= w.page_table.shape[0]:
        return 0
    return int(min(max(int(w.q_len[b]), 0), PAGE * w.page_table.shape[1]))


def run_gpu(layers, mean, threshold, sink, recent, problems=None):
    P = problems or gpu_layers(layers)
    num_q, pts = P[0].num_q, int(P[0].page_table.shape[1])
    stride = PAGE * pts + 64  # wider than needed: the extra columns must stay untouched
    keep = torch.full((num_q, stride), 7, dtype=torch.uint8, device="cuda")
    sc = torch.full((num_q, stride), float("nan"), dtype=torch.float32, device="cuda")
    pages = torch.full((num_q, pts + 3), -5, dtype=torch.int32, device="cuda")
    npg = torch.full((num_q,), -9, dtype=torch.int32, device="cuda")
    native.csa_recall_level1(P, mean, threshold, sink, recent, out=(keep, pages, npg, sc))
    torch.cuda.synchronize()
    st = int(P[0].dev_status.item()) if P[0].dev_status is not None else 0
    return keep.cpu().numpy(), pages.cpu().numpy(), npg.cpu().numpy(), sc.cpu().numpy(), st


def check(layers, mean, threshold, sink, recent, rows=None, expect_flags=0, problems=None):
    """GPU recall over all rows of `layers`; the oracle over `rows` (all by default)."""
    keep, pages, npg, sc, st = run_gpu(layers, mean, threshold, sink, recent, problems)
    w0 = layers[0]
    rows = list(range(w0.num_q)) if rows is None else list(rows)
    if len(rows) == w0.num_q:
        ora_layers = layers
    else:  # the sampled rows as a problem of their own: row i reads request rows[i]
        req = np.array([b if w0.q_req is None else w0.q_req[b] for b in rows], np.int32)
        ora_layers = [synth.Workload(name=w.name, q=w.q[rows], fused_w=w.fused_w[rows], kv=w.kv,
                                     page_table=w.page_table, q_len=w.q_len[rows], q_req=req) for w in layers]
    okeep, osc, opages, oflags = oracle.recall([oracle.Problem(w) for w in ora_layers], mean, threshold, sink,
                                               recent)
    assert st == oflags == expect_flags, (st, oflags)
    thr = np.float32(threshold)
    for i, b in enumerate(rows):
        L = row_length(w0, b)
        g, k = sc[b].astype(np.float64), keep[b]
        assert np.all(k[L:] == 7) and np.all(np.isnan(g[L:])), f"row {b}: columns past the length written"
        assert not np.any(np.isnan(g[:L])), f"row {b}: a column below the length left unwritten"
        d = np.abs(g[:L] - osc[i, :L])
        assert d.max(initial=0.0) <= TOL, f"row {b}: max |dscore| {d.max()}"
        n = np.arange(L)
        own = (sc[b, :L] >= thr) | (n < sink) | (n >= L - recent)
        assert np.array_equal(k[:L], own.astype(np.uint8)), f"row {b}: keep does not follow the scores"
        flip = np.nonzero(k[:L] != okeep[i, :L])[0]
        assert np.all(np.abs(osc[i, flip] - threshold) <= TOL), f"row {b}: keep differs outside the band"
        want_pages = np.unique(np.nonzero(k[:L])[0] // PAGE).astype(np.int32)
        m = int(npg[b])
        assert m == len(want_pages) and np.array_equal(pages[b, :m], want_pages), f"row {b}: page list"
        assert np.all(pages[b, m:] == -5), f"row {b}: page list overran its count"
        for p in set(want_pages.tolist()) ^ set(opages[i].tolist()):
            assert np.any((flip >= p * PAGE) & (flip < (p + 1) * PAGE)), f"row {b}: page {p} differs"
    return keep, sc, osc


def mid_threshold(osc, L):
    """A threshold halfway between two adjacent distinct oracle scores near the median."""
    v = np.unique(osc[:L])
    j = len(v) // 2
    return float((v[j - 1] + v[j]) / 2)


# ------------------------------------------------------------------ raw logits

@pytest.mark.parametrize("heads", [64, 128])
def test_logits_match_the_oracle(heads):
    """Both head counts of the scorer, against the oracle's logits; 128 heads also
    through csa_index_score."""
    w = synth.make_workload("lg", num_q=4, history=[3000, 700, 64, 1], seed=61)
    if heads == 128:
        w = synth.level1_layers(w, 1, seed=62)[0]
    prob = native.Problem.from_workload(w)
    lg = native.csa_index_logits(prob)
    torch.cuda.synchronize()
    lg = lg.cpu().numpy().astype(np.float64)
    olg, valid, _ = oracle.logits(oracle.Problem(w), lg.shape[1])
    assert np.all(np.isnan(lg[~valid])) and not np.any(np.isnan(lg[valid]))
    d = np.abs(lg[valid] - olg[valid])
    assert np.all(d <= _parity.STRICT_LOGIT_TOL * (1.0 + np.abs(olg[valid]))), d.max()
    # and the sigmoid of them is what csa_index_score writes
    s = native.csa_index_score(prob).cpu().numpy().astype(np.float64)
    assert np.max(np.abs(_parity.sigmoid(lg[valid]) - s[valid])) <= 1e-6


def test_128_head_logits_large_dynamic_range_and_bad_pages():
    """128-head queries whose heads span 2^-20..2^20, weights scaled by 2^-6..2^6,
    one page out of range (flagged, its records not written)."""
    w = synth.level1_layers(synth.make_workload("dr", num_q=3, history=[2500, 900, 130], seed=64), 1, seed=65)[0]
    rng = np.random.default_rng(66)
    qf = rng.standard_normal((3, 128, 128)).astype(np.float32)
    qf *= np.float32(2.0) ** rng.integers(-20, 21, size=(3, 128, 1)).astype(np.float32)
    w.q = _pins.bf16_bits(qf).reshape(3, 128, 128)
    w.fused_w = w.fused_w * (np.float32(2.0) ** rng.integers(-6, 7, size=(3, 128)).astype(np.float32))
    w.page_table = w.page_table.copy()
    w.page_table[1, 3] = w.num_pages + 5
    prob = native.Problem.from_workload(w)
    lg = native.csa_index_logits(prob)
    torch.cuda.synchronize()
    assert int(prob.dev_status.item()) == native.DEV_PAGE_OOB
    lg = lg.cpu().numpy().astype(np.float64)
    olg, valid, flags = oracle.logits(oracle.Problem(w), lg.shape[1])
    assert flags == oracle.PAGE_OOB
    assert np.all(np.isnan(lg[~valid])) and not np.any(np.isnan(lg[valid]))
    # weights of both signs make terms near 1e6 cancel: fp32 error scales with
    # sum_h relu(k . q_h) |w_h|, which is the oracle's logit with |w|
    mag = synth.Workload(name="mag", q=w.q, fused_w=np.abs(w.fused_w), kv=w.kv, page_table=w.page_table,
                         q_len=w.q_len)
    scale, _, _ = oracle.logits(oracle.Problem(mag), lg.shape[1])
    d = np.abs(lg[valid] - olg[valid])
    assert np.all(d <= _parity.STRICT_LOGIT_TOL * (1.0 + scale[valid])), (d / (1.0 + scale[valid])).max()


# ------------------------------------------------------------------ recall against the oracle

@pytest.mark.parametrize("mean", [False, True], ids=["max", "mean"])
def test_recall_separate_caches(mean):
    """Three layers, each with its own cache of the same lengths; ragged rows, an
    empty row, a one-record row."""
    layers = _pins.recall_layers(3, 6, [5000, 1300, 129, 64, 1, 0], seed=63)
    _, osc, _, _ = oracle.recall([oracle.Problem(w) for w in layers], mean, 2.0, 0, 0)
    check(layers, mean, mid_threshold(osc[0], 5000), sink=3, recent=70)


def test_recall_one_layer_is_the_sigmoid_of_its_logit():
    layers = _pins.recall_layers(1, 3, [2000, 777, 64], seed=64)
    _, osc, _, _ = oracle.recall([oracle.Problem(layers[0])], False, 2.0, 0, 0)
    for mean in (False, True):
        check(layers, mean, mid_threshold(osc[0], 2000), sink=0, recent=0)


def test_recall_sink_and_tail_edges():
    layers = _pins.recall_layers(2, 4, [300, 70, 65, 5], seed=65)
    for thr, sink, recent in ((2.0, 0, 0), (2.0, 1, 1), (2.0, 64, 64), (2.0, 400, 0), (2.0, 0, 400),
                              (-1.0, 0, 0), (0.0, 0, 0)):
        keep, _, _ = check(layers, False, thr, sink, recent)
        if thr < 0:
            assert np.all(keep[0, :300] == 1)


def test_recall_zero_weights():
    """Every score is exactly 0.5: threshold 0.5 keeps all, the next float up
    keeps the sink and the tail alone."""
    layers = _pins.recall_layers(3, 2, [400, 90], seed=66, zero_weights=(0, 1, 2))
    for mean in (False, True):
        keep, sc, _ = check(layers, mean, 0.5, 2, 64)
        assert np.all(sc[0, :400] == 0.5) and np.all(keep[0, :400] == 1)
        keep, _, _ = check(layers, mean, float(np.nextafter(np.float32(0.5), np.float32(1))), 2, 64)
        assert np.array_equal(np.nonzero(keep[0, :400])[0], np.r_[0:2, 336:400])


def test_recall_prefill_rows():
    """Rows of one request with growing lengths (q_req given), several tiles each."""
    layers = _pins.recall_layers(2, 24, [3000], seed=67, single_request=True,
                                 q_len=lambda h, n: np.minimum(3000, 1 + np.arange(n) * 131))
    _, osc, _, _ = oracle.recall([oracle.Problem(w) for w in layers], True, 2.0, 0, 0)
    check(layers, True, mid_threshold(osc[-1], 3000), sink=4, recent=128)


def test_recall_invalid_geometry_is_flagged_not_fatal():
    """A page out of range in one layer scores 0 there; a request id out of range
    makes its row empty; other layers' q_len and q_req are not read."""
    layers = _pins.recall_layers(2, 3, [300, 300, 300], seed=68)
    layers[1].page_table = layers[1].page_table.copy()
    layers[1].page_table[0, 2] = layers[1].num_pages + 1
    layers[0].q_req = np.array([0, 1, 7], np.int32)
    layers[1].q_req = np.array([0, 1, 2], np.int32)
    layers[1].q_len = np.array([5, 5, 5], np.int32)
    for mean in (False, True):
        keep, _, _ = check(layers, mean, 0.3, 0, 0, expect_flags=oracle.PAGE_OOB | oracle.BAD_REQUEST)
        assert np.all(keep[2] == 7)


def test_recall_long_ragged_geometry_sampled_rows():
    """Three target layers over the 64-row ragged decode cache (64K..128K records
    per row), checked on sampled rows."""
    w = synth.config("long_ragged_decode")
    layers = synth.level1_layers(w, 3, seed=69)
    rows = [0, 31, 63]
    sub = [synth.Workload(name="s", q=l.q[rows[:1]], fused_w=l.fused_w[rows[:1]], kv=l.kv, page_table=l.page_table,
                          q_len=l.q_len[rows[:1]], q_req=np.array(rows[:1], np.int32)) for l in layers]
    _, osc, _, _ = oracle.recall([oracle.Problem(x) for x in sub], False, 2.0, 0, 0)
    thr = mid_threshold(osc[0], int(w.q_len[0]))
    check(layers, False, thr, sink=4, recent=512, rows=rows)


def test_recall_deterministic():
    layers = _pins.recall_layers(3, 4, [9000, 3000, 100, 0], seed=70)
    P = gpu_layers(layers)
    a = run_gpu(layers, True, 0.5, 2, 100, problems=P)
    b = run_gpu(layers, True, 0.5, 2, 100, problems=P)
    for x, y in zip(a, b):
        assert np.array_equal(x, y, equal_nan=True)


def test_128_head_scores_resident_mode():
    """The 128-head scorer over a resident page list (csa_index_score), against the
    oracle's scores in the resident column layout."""
    w = synth.make_workload("r128", num_q=3, history=[64 * 40 + 17, 64 * 9, 64 * 30], resident_pages=7, seed=71)
    w = dataclasses.replace(synth.level1_layers(w, 1, seed=72)[0], resident=w.resident, n_resident=w.n_resident)
    prob = native.Problem.from_workload(w)
    sc = native.csa_index_score(prob)
    torch.cuda.synchronize()
    assert int(prob.dev_status.item()) == 0
    _parity.check_scores(w, sc.cpu().numpy())


def test_recall_eight_layers_mean():
    """The largest layer count, mean ensemble, threshold between two oracle scores."""
    layers = _pins.recall_layers(8, 2, [1500, 700], seed=73)
    _, osc, _, _ = oracle.recall([oracle.Problem(w) for w in layers], True, 2.0, 0, 0)
    check(layers, True, mid_threshold(osc[0], 1500), sink=1, recent=33)
