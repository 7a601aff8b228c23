"""The seeded workloads: determinism, shapes and the recipe's properties."""
import numpy as np
import torch

from sparse_attention_kv_e4m3_gb300 import synth

REC, D, PAGE = 132, 128, 64


def _records(w):
    return w.kv[:, : PAGE * REC].reshape(-1, REC)


def test_deterministic():
    a = synth.make_workload("a", num_q=3, history=lambda g, n: g.integers(100, 300, size=n),
                            outlier_frac=0.1, resident_pages=2, seed=5, threads=1)
    b = synth.make_workload("b", num_q=3, history=lambda g, n: g.integers(100, 300, size=n),
                            outlier_frac=0.1, resident_pages=2, seed=5, threads=4)
    for f in ("q", "fused_w", "kv", "page_table", "q_len", "resident", "n_resident"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    c = synth.make_workload("c", num_q=3, history=[200] * 3, seed=6)
    assert not np.array_equal(a.q, c.q)


def test_record_recipe():
    w = synth.make_workload("r", num_q=2, history=[3000, 2000], seed=1)
    recs = _records(w)
    codes = recs[:, :D]
    # no NaN codes (S.1111.111) ever; the largest magnitude of each row is 448 (0x7e / 0xfe)
    assert not np.any((codes & 0x7F) == 0x7F)
    assert np.all(((codes & 0x7F) == 0x7E).any(axis=1))
    s = recs[:, D:].copy().view("<f4").reshape(-1)
    assert np.all(s > 0) and np.all(s < 6.5 / 448)
    vals = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy() * s[:, None]
    assert abs(vals.mean()) < 0.02 and abs(vals.std() - 1.0) < 0.02


def test_outliers_and_permutation():
    w = synth.make_workload("o", num_q=4, history=[6400] * 4, outlier_frac=0.05, seed=2)
    base = synth.make_workload("o", num_q=4, history=[6400] * 4, outlier_frac=0.0, seed=2)
    s1 = _records(w)[:, D:].copy().view("<f4").reshape(-1)
    s0 = _records(base)[:, D:].copy().view("<f4").reshape(-1)
    ratio = s1 / s0
    assert set(np.unique(ratio)) <= {1.0, 8.0}
    assert 0.04 < (ratio == 8.0).mean() < 0.06
    assert np.array_equal(_records(w)[:, :D], _records(base)[:, :D])
    assert sorted(w.page_table.reshape(-1).tolist()) == list(range(w.num_pages))


def test_resident_lists_distinct():
    w = synth.make_workload("res", num_q=3, history=[64 * 50] * 3, resident_pages=20, seed=3)
    for r in range(3):
        row = w.resident[r, : w.n_resident[r]]
        assert len(set(row.tolist())) == 20 and row.min() >= 0 and row.max() < 50


def test_named_config_shapes():
    t = synth.config("tiny_decode")
    assert t.num_q == 1 and t.num_pages == 64 and np.array_equal(t.page_table[0], np.arange(64))
    assert int(t.visible_counts().sum()) == 4096
    p = synth.config("prefill_chunk")
    assert p.num_q == 4096 and p.num_req == 1 and p.num_pages == 256
    assert p.q_len.min() == 1024 and p.q_len.max() == 2047
    assert int(p.visible_counts().sum()) == 6289408
    pt = synth.config("prefill_chunk_tail")
    assert pt.q_len.min() == 15361 and pt.q_len.max() == 16384
    assert int(pt.visible_counts().sum()) == 65013760


def test_fused_weight_recipe():
    w = synth.make_workload("w", num_q=64, history=[64] * 64, seed=4)
    x = w.fused_w.astype(np.float64) * np.sqrt(128.0) * np.sqrt(64.0)
    assert abs(x.std() - 1.0) < 0.03


def test_mxfp4_cache_shape_and_determinism():
    """68-byte records drawn directly (codes and block-scale bytes), same geometry
    and rows as the workload it is made from, identical for the same seed."""
    base = synth.make_workload("mx", num_q=2, history=[700, 130], seed=5, threads=1)
    a, b = synth.mxfp4_cache(base, seed=9), synth.mxfp4_cache(base, seed=9)
    assert a.record_format == "mxfp4" and a.kv.shape == (base.kv.shape[0], 64 * 68)
    assert np.array_equal(a.kv, b.kv) and not np.array_equal(a.kv, synth.mxfp4_cache(base, seed=10).kv)
    scales = a.kv.reshape(-1, 64, 68)[..., 64:]
    assert scales.min() >= 124 and scales.max() <= 128
    assert np.array_equal(a.page_table, base.page_table) and np.array_equal(a.q, base.q)
    assert a.k_bytes() == int(a.visible_counts().sum()) * 68
