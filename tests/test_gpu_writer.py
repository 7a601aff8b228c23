"""The compressed-K writer on the GPU, through the C ABI, against the oracle.

Every comparison is of whole cache buffers, byte for byte: the writer decides
integer codes, so the bar is bit-exact."""
import numpy as np
import pytest
import torch

import _parity
import oracle
from sparse_attention_kv_e4m3_gb300 import native, synth

pytestmark = pytest.mark.gpu
D, PAGE, REC = 128, 64, 132


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_kv_e4m3_gb300 import build

    build.build()
    native.load()


def _cache(num_req, pages_per_req, pad=0, seed=0, extra_pages=3):
    """A cache filled with 0xA5 and a shuffled page table (spare pages stay untouched)."""
    rng = np.random.default_rng(seed)
    num_pages = num_req * pages_per_req + extra_pages
    pt = rng.permutation(num_pages)[: num_req * pages_per_req].reshape(num_req, pages_per_req).astype(np.int32)
    kv = np.full((num_pages, PAGE * REC + pad), 0xA5, dtype=np.uint8)
    return kv, pt


def _rows(n, seed):
    """Rows of varied magnitude: N(0,1) times a per-row 10^U(-6, 6)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, D)).astype(np.float32)
    x *= (10.0 ** rng.uniform(-6, 6, (n, 1))).astype(np.float32)
    return x


def _distinct_positions(num_req, pages_per_req, n, seed):
    rng = np.random.default_rng(seed)
    slots = rng.choice(num_req * pages_per_req * PAGE, size=n, replace=False)
    return (slots // (pages_per_req * PAGE)).astype(np.int32), (slots % (pages_per_req * PAGE)).astype(np.int32)


def _write_gpu(keys, req, pos, kv, pt):
    kv_d = torch.from_numpy(kv).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    native.csa_index_write_keys(torch.from_numpy(keys).cuda(), torch.from_numpy(pos).cuda(), kv_d,
                                torch.from_numpy(pt).cuda(),
                                row_req=None if req is None else torch.from_numpy(req).cuda(), dev_status=status)
    torch.cuda.synchronize()
    return kv_d.cpu().numpy(), int(status.item())


def _bf16_as_f32(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float32).numpy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bit_exact_against_the_oracle(dtype):
    kv, pt = _cache(num_req=5, pages_per_req=7, pad=32, seed=1)
    n = 5 * 7 * PAGE // 2
    req, pos = _distinct_positions(5, 7, n, seed=2)
    x = _rows(n, seed=3)
    if dtype == "bf16":
        xt = torch.from_numpy(x).to(torch.bfloat16)
        keys_gpu = xt
        x_oracle = _bf16_as_f32(xt)
    else:
        keys_gpu = torch.from_numpy(x)
        x_oracle = x
    want = kv.copy()
    assert oracle.write_keys(x_oracle, req, pos, want, pt) == 0
    kv_d = torch.from_numpy(kv).cuda()
    native.csa_index_write_keys(keys_gpu.cuda(), torch.from_numpy(pos).cuda(), kv_d, torch.from_numpy(pt).cuda(),
                                row_req=torch.from_numpy(req).cuda())
    torch.cuda.synchronize()
    got = kv_d.cpu().numpy()
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]


def test_special_rows():
    """Zero and underflowing rows, a row on the e4m3 grid, signed zeros, exact
    e4m3 midpoints (ties), values past 448 after scaling, subnormal inputs."""
    grid = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    rows = []
    rows.append(np.zeros(D, np.float32))
    tiny = np.zeros(D, np.float32)
    tiny[[1, 90]] = [1e-44, -3e-45]
    rows.append(tiny)
    on_grid = grid[np.random.default_rng(0).integers(0, 127, D)].astype(np.float32)
    on_grid[5] = 448.0
    on_grid[::4] *= -1
    rows.append(on_grid)
    signed_zero = np.zeros(D, np.float32)
    signed_zero[::2] = -0.0
    signed_zero[7] = 3.0
    rows.append(signed_zero)
    mids = ((grid[:-1].astype(np.float64) + grid[1:]) / 2).astype(np.float32)
    tie = np.resize(mids, D).astype(np.float32)
    tie[0] = 448.0  # scale exactly 1, so x / scale are the midpoints themselves
    rows.append(tie)
    rows.append(-tie)
    sub = (np.random.default_rng(1).standard_normal(D) * 1e-39).astype(np.float32)  # subnormal inputs
    rows.append(sub)
    big = np.full(D, 3.0e38, np.float32)
    big[::3] = -1.0e-30
    rows.append(big)
    x = np.stack(rows).astype(np.float32)
    n = x.shape[0]
    kv, pt = _cache(num_req=1, pages_per_req=1, seed=4)
    pos = np.arange(n, dtype=np.int32) * 3
    want = kv.copy()
    assert oracle.write_keys(x, np.zeros(n, np.int32), pos, want, pt) == 0
    got, status = _write_gpu(x, np.zeros(n, np.int32), pos, kv, pt)
    assert status == 0
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]


def _scales_with_all_ones_significand(rng, count):
    """amax values whose scale RN(amax / 448) has the all-ones significand
    (2 - 2^-23) 2^e, the hardest divisor for a reciprocal-based quotient."""
    out = []
    while len(out) < count:
        e = int(rng.integers(-88, 100))
        target = np.float32(np.ldexp(2.0 - 2.0 ** -23, e))
        a = np.float32(np.float64(target) * 448.0)
        for _ in range(8):
            if np.float32(a / np.float32(448.0)) == target:
                out.append(a)
                break
            a = np.nextafter(a, np.float32(np.inf) if a / np.float32(448.0) < target else np.float32(0))
    return np.array(out, dtype=np.float32)


def test_quotients_at_code_boundaries():
    """x / scale within a few binary32 ulps of every e4m3 rounding boundary
    (midpoints between codes, the 448/464 saturation edge, the 2^-10 edge of
    the smallest code), at scales from 2^-96 to 2^110 (both sides of the
    writer's 2^-90 switch from reciprocal-based quotients to the division) and
    at divisors with an all-ones significand: the codes must be the oracle's,
    whose quotients are IEEE binary32 divisions."""
    rng = np.random.default_rng(11)
    grid = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    grid = grid.astype(np.float64)
    bounds = np.concatenate([(grid[:-1] + grid[1:]) / 2, grid[1:], [2.0 ** -10, 2.0 ** -9, 440.0]])
    bounds = bounds[bounds <= 440.0]
    n = 8192
    amax = np.ldexp(rng.uniform(1.0, 2.0, n), rng.integers(-87, 118, n)).astype(np.float32)
    amax[: n // 8] = _scales_with_all_ones_significand(rng, n // 8)
    # scales around 2^-90, the switch: amax = 448 scale
    amax[n // 8: n // 8 + 256] = np.ldexp(rng.uniform(1.0, 2.0, 256), rng.integers(-84, -78, 256)).astype(np.float32)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    m = rng.choice(bounds, size=(n, D))
    sign = np.where(rng.random((n, D)) < 0.5, -1.0, 1.0)
    ulps = rng.integers(-3, 4, size=(n, D))
    x = (sign * m * scale[:, None].astype(np.float64)).astype(np.float32)
    up, down = np.float32(np.inf), np.float32(-np.inf)
    for _ in range(3):  # up to three ulps away in either direction
        x = np.where(ulps > 0, np.nextafter(x, up), np.where(ulps < 0, np.nextafter(x, down), x))
        ulps = ulps - np.sign(ulps)
    x[:, 0] = amax  # the largest magnitude of each row, so its scale is the one above
    kv, pt = _cache(num_req=8, pages_per_req=16, seed=12)
    req, pos = _distinct_positions(8, 16, n, seed=13)
    want = kv.copy()
    assert oracle.write_keys(x, req, pos, want, pt) == 0
    got, status = _write_gpu(x, req, pos, kv, pt)
    assert status == 0
    bad = np.argwhere(got != want)
    assert len(bad) == 0, bad[:5]


def test_invalid_rows_are_flagged_and_skipped():
    kv, pt = _cache(num_req=2, pages_per_req=2, seed=5)
    pt[1, 1] = kv.shape[0] + 4  # a page id out of range
    x = _rows(7, seed=6)
    x[5, 9] = np.nan
    x[6, 0] = -np.inf
    req = np.array([0, 1, 2, -1, 1, 0, 1], np.int32)
    pos = np.array([3, 70, 0, 1, 130, 100, 5], np.int32)
    want = kv.copy()
    flags = oracle.write_keys(x, req, pos, want, pt)
    got, status = _write_gpu(x, req, pos, kv, pt)
    assert flags == oracle.BAD_REQUEST | oracle.PAGE_OOB | oracle.LEN_OOB | oracle.RANGE
    assert status == native.DEV_BAD_REQUEST | native.DEV_PAGE_OOB | native.DEV_LEN_OOB | native.DEV_RANGE
    assert np.array_equal(got, want)


def test_identity_requests_and_many_rows():
    """row_req NULL maps row i to request i; more rows than one grid pass."""
    num_req = 4096
    kv, pt = _cache(num_req=num_req, pages_per_req=1, seed=7)
    x = _rows(num_req, seed=8)
    pos = np.random.default_rng(9).integers(0, PAGE, num_req).astype(np.int32)
    want = kv.copy()
    assert oracle.write_keys(x, None, pos, want, pt) == 0
    got, status = _write_gpu(x, None, pos, kv, pt)
    assert status == 0 and np.array_equal(got, want)


def test_reproduces_the_generator_cache():
    """The workload generator's pages come from rows drawn per physical page and
    quantised with numpy and torch; writing those rows reproduces its bytes."""
    pages = 40
    w = synth.make_workload("wr", num_q=1, history=[pages * PAGE], shuffle=False, seed=12)
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(12, spawn_key=(1, 0))))
    x = g.standard_normal((pages, PAGE, D), dtype=np.float32).reshape(-1, D)
    kv = np.zeros_like(w.kv)
    got, status = _write_gpu(x, np.zeros(pages * PAGE, np.int32), np.arange(pages * PAGE, dtype=np.int32), kv,
                             w.page_table)
    assert status == 0
    assert np.array_equal(got[:, : PAGE * REC], w.kv[:, : PAGE * REC])


def test_written_cache_scores_like_the_oracle():
    """Keys written by the writer feed the indexer: its top-k over them matches the
    oracle's on the same bytes."""
    w = synth.make_workload("ws", num_q=3, history=[3000, 1500, 700], seed=13)
    n_req, pts = w.page_table.shape
    rows_per_req = [int(L) for L in w.q_len]
    req = np.concatenate([np.full(L, r, np.int32) for r, L in enumerate(rows_per_req)])
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in rows_per_req])
    x = _rows(len(req), seed=14) * np.float32(1e-3)
    kv, status = _write_gpu(x, req, pos, np.zeros_like(w.kv), w.page_table)
    assert status == 0
    want = np.zeros_like(w.kv)
    assert oracle.write_keys(x, req, pos, want, w.page_table) == 0
    assert np.array_equal(kv, want)
    w.kv = kv
    prob = native.Problem.from_workload(w)
    idx, vals = native.csa_index_score_topk_fused(prob, 256)
    torch.cuda.synchronize()
    _parity.check_topk(w, idx.cpu().numpy(), vals.cpu().numpy(), 256)
