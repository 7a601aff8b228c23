"""Checks that pin the oracle to things other than itself.

Each `pin_*` function takes an `oracle.Oracle` and raises AssertionError when
the oracle disagrees with an outside fact: a library routine (torch's fp8 and
bf16 casts, numpy's float64 matmul and lexsort), the format definition, a
closed form, a hand-worked example or an invariant of the method. The same
functions run against the real oracle (all must pass) and against builds of
the oracle with a mistake planted in them (at least one must fail).
"""
from __future__ import annotations

import math
import os
import struct

import numpy as np
import torch

from sparse_attention_kv_e4m3_gb300 import synth
import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
H, D, PAGE, REC = 64, 128, 64, 132


# ---------------------------------------------------------------- helpers

def e4m3_code(x: float) -> int:
    """The e4m3 byte of x by torch's cast (round to nearest even)."""
    return int(torch.tensor([x], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).item())


def bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def hand_workload(records: np.ndarray, q: np.ndarray, w: np.ndarray, q_len=None,
                  num_q: int = 1) -> synth.Workload:
    """One request whose history is `records` ([n, 132] uint8), identity pages."""
    n = records.shape[0]
    pages = max(1, (n + PAGE - 1) // PAGE)
    kv = np.zeros((pages, PAGE * REC), dtype=np.uint8)
    kv.reshape(-1, REC)[:n] = records
    qb = np.broadcast_to(bf16_bits(q), (num_q, H, D)).copy()
    wb = np.broadcast_to(np.asarray(w, dtype=np.float32), (num_q, H)).copy()
    return synth.Workload(
        name="hand", q=qb, fused_w=wb, kv=kv,
        page_table=np.arange(pages, dtype=np.int32).reshape(1, pages),
        q_len=np.full(num_q, n if q_len is None else q_len, dtype=np.int32),
        q_req=np.zeros(num_q, dtype=np.int32))


def record(values: dict, scale: float) -> np.ndarray:
    """A 132-byte record: e4m3 bytes given as {d: byte}, then the fp32 scale."""
    r = np.zeros(REC, dtype=np.uint8)
    for d, b in values.items():
        r[d] = b
    r[D:] = np.frombuffer(struct.pack("<f", scale), dtype=np.uint8)
    return r


def tiny_workloads():
    """Small seeded workloads spanning partial pages, shuffled pages, several rows,
    resident subsets and shared-request rows."""
    yield synth.make_workload("t_full", num_q=3, history=[130, 70, 1], seed=11)
    yield synth.make_workload("t_out", num_q=2, history=[200, 64], outlier_frac=0.2, seed=12)
    yield synth.make_workload("t_res", num_q=2, history=[600, 333], resident_pages=3, seed=13)
    yield synth.make_workload("t_pre", num_q=5, history=[300], single_request=True,
                              q_len=lambda h, n: np.array([1, 64, 65, 250, 300]), seed=14)
    yield synth.make_workload("t_pad", num_q=2, history=[100, 129], page_pad=48, seed=15)


def brute_logits(w: synth.Workload):
    """Independent float64 restatement with library primitives: torch's e4m3 and
    bf16 decodes, numpy's matmul. Returns {(b, position): (logit, column)}."""
    table = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    table = table.to(torch.float64).numpy()
    out = {}
    for b in range(w.num_q):
        req = int(w.q_req[b]) if w.q_req is not None else b
        L = min(max(int(w.q_len[b]), 0), PAGE * w.pt_stride)
        qf = torch.from_numpy(w.q[b].view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
        wf = w.fused_w[b].astype(np.float64)
        npages = (L + PAGE - 1) // PAGE
        if w.resident is None:
            plist = [(p, p) for p in range(npages)]
        else:
            plist = [(int(p), j) for j, p in enumerate(w.resident[req, : int(w.n_resident[req])])]
        for p, j in plist:
            if not (0 <= p < npages):
                continue
            phys = int(w.page_table[req, p])
            if not (0 <= phys < w.num_pages):
                continue
            for r in range(PAGE):
                pos = p * PAGE + r
                if pos >= L:
                    break
                rec = w.kv[phys, r * REC:(r + 1) * REC]
                s = float(np.frombuffer(rec[D:].tobytes(), dtype="<f4")[0])
                k = table[rec[:D]] * s
                dots = qf @ k
                logit = float(np.maximum(dots, 0.0) @ wf)
                out[(b, pos)] = (logit, j * PAGE + r)
    return out


def brute_topk(w: synth.Workload, k: int):
    lg = brute_logits(w)
    idx = np.full((w.num_q, k), -1, dtype=np.int64)
    val = np.full((w.num_q, k), -np.inf)
    for b in range(w.num_q):
        items = [(pos, v[0]) for (bb, pos), v in lg.items() if bb == b]
        if not items:
            continue
        pos = np.array([i[0] for i in items])
        lv = np.array([i[1] for i in items])
        order = np.lexsort((pos, -lv))[:k]
        idx[b, : len(order)] = pos[order]
        val[b, : len(order)] = lv[order]
    return idx, val


# ---------------------------------------------------------------- pins

def pin_e4m3_vs_torch(o: O.Oracle):
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for b in range(256):
        got, want = o.e4m3(b), float(lib[b])
        if math.isnan(want):
            assert math.isnan(got), f"byte {b:#04x}: want NaN, got {got}"
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), \
                f"byte {b:#04x}: {got} != {want}"


def pin_e4m3_spec_golden(o: O.Oracle):
    with open(os.path.join(GOLDEN, "e4m3_ocp_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if not line:
                continue
            b, v = int(line[0], 16), float(line[1])
            got = o.e4m3(b)
            if math.isnan(v):
                assert math.isnan(got), f"{b:#04x}"
            else:
                assert got == v and math.copysign(1, got) == math.copysign(1, v), f"{b:#04x}: {got} != {v}"


def pin_bf16_vs_torch(o: O.Oracle):
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, size=4000).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite values only
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([o.bf16(int(x)) for x in bits])
    assert np.array_equal(got, want)


def pin_scale_little_endian(o: O.Oracle):
    for s in (2.5, -0.75, 1e-3, 3.0e5):
        r = record({}, s)
        assert o.scale(r) == struct.unpack("<f", struct.pack("<f", s))[0]


def pin_sigmoid_closed_form(o: O.Oracle):
    assert o.sigmoid(0.0) == 0.5
    assert abs(o.sigmoid(math.log(3.0)) - 0.75) < 1e-15
    assert abs(o.sigmoid(-math.log(3.0)) - 0.25) < 1e-15


def pin_worked_example(o: O.Oracle):
    vals = {}
    with open(os.path.join(GOLDEN, "worked_example.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if line:
                vals[line[0]] = line[1:]
    rec = record({d: int(x, 16) for d, x in enumerate(vals["bytes"])}, float(vals["scale"][0]))
    q = np.zeros((H, D), dtype=np.float32)
    for h in range(3):
        q[h, :3] = [float(x) for x in vals[f"q{h}"]]
    w = np.zeros(H, dtype=np.float32)
    w[:3] = [float(x) for x in vals["w"]]
    P = O.Problem(hand_workload(rec[None, :], q, w))
    lg = o.logit(P, 0, 0)
    assert lg == float(vals["logit"][0]), lg
    idx, sc, lgk, _ = o.topk(P, 4)
    assert idx[0, 0] == 0 and list(idx[0, 1:]) == [-1, -1, -1]
    assert abs(sc[0, 0] - float(vals["score"][0])) < 1e-15
    assert list(sc[0, 1:]) == [0.0, 0.0, 0.0]


def pin_zero_weights_half(o: O.Oracle):
    w = synth.make_workload("zw", num_q=2, history=[150, 90], seed=3)
    w.fused_w[:] = 0.0
    P = O.Problem(w)
    sc, valid, _ = o.scores(P)
    assert valid.sum() == 240 and np.all(sc[valid] == 0.5)
    idx, s, _, _ = o.topk(P, 100)
    # equal logits everywhere: the lower position wins every tie
    assert np.array_equal(idx[0], np.arange(100)) and np.array_equal(idx[1], np.arange(90).tolist() + [-1] * 10)
    assert np.all(s[0] == 0.5)


def pin_zero_query_half(o: O.Oracle):
    w = synth.make_workload("zq", num_q=1, history=[70], seed=4)
    w.q[:] = 0
    sc, valid, _ = o.scores(O.Problem(w))
    assert np.all(sc[valid] == 0.5)


def pin_one_hot(o: O.Oracle):
    """One head, w = 1, q one-hot at d0: score = sigmoid(max(0, s * e4m3(byte[d0])))."""
    w = synth.make_workload("oh", num_q=1, history=[128], seed=5)
    d0 = 37
    q = np.zeros((H, D), dtype=np.float32)
    q[9, d0] = 1.0
    w.q[0] = bf16_bits(q)
    w.fused_w[0] = 0.0
    w.fused_w[0, 9] = 1.0
    P = O.Problem(w)
    table = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for pos in (0, 5, 63, 64, 127):
        phys = int(w.page_table[0, pos // PAGE])
        rec = w.kv[phys, (pos % PAGE) * REC:(pos % PAGE + 1) * REC]
        s = float(np.frombuffer(rec[D:].tobytes(), dtype="<f4")[0])
        want = max(0.0, s * table[rec[d0]])
        assert o.logit(P, 0, pos) == want


def pin_relu_before_sum(o: O.Oracle):
    """relu comes before the head-weighted sum (BatchGen #153 commit log): record A
    has head dots (+3, -5), record B (+1, +1); with w = (1, 1) A scores 3 and B 2,
    so A ranks first; summing before relu would rank B first (-2 < 2)."""
    q = np.zeros((H, D), dtype=np.float32)
    q[0, 0] = 1.0
    q[1, 1] = 1.0
    w = np.zeros(H, dtype=np.float32)
    w[:2] = 1.0
    A = record({0: e4m3_code(3.0), 1: e4m3_code(-5.0)}, 1.0)
    B = record({0: e4m3_code(1.0), 1: e4m3_code(1.0)}, 1.0)
    P = O.Problem(hand_workload(np.stack([B, A]), q, w))
    assert o.logit(P, 0, 0) == 2.0 and o.logit(P, 0, 1) == 3.0
    idx, _, _, _ = o.topk(P, 1)
    assert idx[0, 0] == 1


def pin_negative_scale(o: O.Oracle):
    """relu acts on the dequantised k . q, so a negative scale flips which heads pass:
    x = (+3, -5), s = -1 -> relu(s*x) = (0, 5) -> logit 5 with w = (1, 1)."""
    q = np.zeros((H, D), dtype=np.float32)
    q[0, 0] = 1.0
    q[1, 1] = 1.0
    w = np.zeros(H, dtype=np.float32)
    w[:2] = 1.0
    A = record({0: e4m3_code(3.0), 1: e4m3_code(-5.0)}, -1.0)
    P = O.Problem(hand_workload(A[None, :], q, w))
    assert o.logit(P, 0, 0) == 5.0


def pin_padding(o: O.Oracle):
    w = synth.make_workload("pad", num_q=2, history=[10, 0], seed=6)
    idx, sc, lg, _ = o.topk(O.Problem(w), 16)
    assert np.all(idx[0, 10:] == -1) and np.all(sc[0, 10:] == 0.0) and np.all(np.isneginf(lg[0, 10:]))
    assert sorted(idx[0, :10]) == list(range(10))
    assert np.all(idx[1] == -1) and np.all(sc[1] == 0.0)


def pin_brute_force(o: O.Oracle):
    for w in tiny_workloads():
        P = O.Problem(w)
        want = brute_logits(w)
        lg, valid, flags = o.logits(P)
        assert flags == 0, (w.name, flags)
        assert int(valid.sum()) == len(want), (w.name, int(valid.sum()), len(want))
        for (b, pos), (v, col) in want.items():
            assert valid[b, col], (w.name, b, pos)
            assert abs(lg[b, col] - v) <= 1e-12 * (1.0 + abs(v)), (w.name, b, pos, lg[b, col], v)
        k = 40
        bi, bv = brute_topk(w, k)
        idx, sc, lgk, _ = o.topk(P, k)
        assert np.array_equal(idx, bi), w.name
        fin = np.isfinite(bv)
        assert np.allclose(lgk[fin], bv[fin], rtol=1e-12, atol=1e-12)
        with np.errstate(over="ignore"):
            assert np.allclose(sc[fin], 1.0 / (1.0 + np.exp(-bv[fin])), rtol=1e-12, atol=1e-15)


def pin_scores_in_unit_interval(o: O.Oracle):
    w = synth.make_workload("u", num_q=2, history=[300, 77], outlier_frac=0.3, seed=7)
    sc, valid, _ = o.scores(O.Problem(w))
    assert np.all((sc[valid] >= 0.0) & (sc[valid] <= 1.0))


def pin_resident_is_masked_full(o: O.Oracle):
    """Resident mode = full mode with non-resident logits at -inf
    ("Two-level recall algorithm", Level 2)."""
    w = synth.make_workload("rm", num_q=2, history=[700, 450], resident_pages=4, seed=8)
    k = 50
    idx_r, sc_r, _, _ = o.topk(O.Problem(w), k)
    full = synth.Workload(name="rf", q=w.q, fused_w=w.fused_w, kv=w.kv, page_table=w.page_table,
                          q_len=w.q_len)
    lg, valid, _ = o.logits(O.Problem(full))
    for b in range(2):
        pages = set(int(p) for p in w.resident[b, : int(w.n_resident[b])])
        pos = np.array([n for n in range(int(w.q_len[b])) if n // PAGE in pages])
        order = np.lexsort((pos, -lg[b, pos]))[:k]
        want = np.full(k, -1)
        want[: len(order)] = pos[order]
        assert np.array_equal(idx_r[b], want), b


def pin_physical_relayout(o: O.Oracle):
    """Moving pages to other physical slots (and updating the page table) changes nothing."""
    w = synth.make_workload("pr", num_q=2, history=[256, 190], seed=9)
    idx0, sc0, _, _ = o.topk(O.Problem(w), 64)
    perm = np.random.default_rng(2).permutation(w.num_pages)
    kv2 = np.empty_like(w.kv)
    kv2[perm] = w.kv
    w2 = synth.Workload(name="pr2", q=w.q, fused_w=w.fused_w, kv=kv2, page_table=perm[w.page_table].astype(np.int32),
                        q_len=w.q_len)
    idx1, sc1, _, _ = o.topk(O.Problem(w2), 64)
    assert np.array_equal(idx0, idx1) and np.array_equal(sc0, sc1)


def pin_logical_permutation(o: O.Oracle):
    """Permuting a request's logical pages permutes the returned positions."""
    w = synth.make_workload("lp", num_q=1, history=[320], seed=10)
    idx0, sc0, _, _ = o.topk(O.Problem(w), 80)
    pi = np.array([3, 0, 4, 1, 2])  # new logical page p reads old logical page pi[p]
    w2 = synth.Workload(name="lp2", q=w.q, fused_w=w.fused_w, kv=w.kv,
                        page_table=w.page_table[:, pi].copy(), q_len=w.q_len)
    idx1, sc1, _, _ = o.topk(O.Problem(w2), 80)
    inv = np.argsort(pi)
    mapped = inv[idx0[0] // PAGE] * PAGE + idx0[0] % PAGE
    assert np.array_equal(np.sort(mapped), np.sort(idx1[0])) and np.array_equal(sc0, sc1)


def pin_positive_rescaling(o: O.Oracle):
    """Scaling every fused_w by c > 0, or every record scale by c > 0 when w >= 0,
    keeps the top-k (sigmoid and relu are monotone / positively homogeneous)."""
    w = synth.make_workload("sc", num_q=2, history=[260, 140], seed=16)
    idx0, _, _, _ = o.topk(O.Problem(w), 60)
    w.fused_w *= np.float32(4.0)
    idx1, _, _, _ = o.topk(O.Problem(w), 60)
    assert np.array_equal(idx0, idx1)
    w.fused_w[:] = np.abs(w.fused_w)
    idx2, _, _, _ = o.topk(O.Problem(w), 60)
    recs = w.kv[:, : PAGE * REC].reshape(-1, REC)
    sc = recs[:, D:].copy().view("<f4") * np.float32(8.0)
    recs[:, D:] = sc.view(np.uint8)
    idx3, _, _, _ = o.topk(O.Problem(w), 60)
    assert np.array_equal(idx2, idx3)


def pin_invalid_geometry(o: O.Oracle):
    w = synth.make_workload("bad", num_q=3, history=[200, 200, 200], seed=17)
    w.page_table[0, 1] = w.num_pages + 5        # page 1 of row 0 out of range
    w.q_req = np.array([0, 1, 7], dtype=np.int32)  # row 2 names a missing request
    P = O.Problem(w)
    pos0, _, f0 = o.visible(P, 0)
    assert f0 & O.PAGE_OOB and len(pos0) == 200 - 64 and not np.any((pos0 >= 64) & (pos0 < 128))
    pos2, _, f2 = o.visible(P, 2)
    assert f2 & O.BAD_REQUEST and len(pos2) == 0
    r = synth.make_workload("badr", num_q=1, history=[300], resident_pages=2, seed=18)
    r.resident[0, 1] = 5                         # == ceil(300/64): first page past the end
    posr, _, fr = o.visible(O.Problem(r), 0)
    assert fr & O.RESIDENT_OOB and len(posr) == min(64, 300 - 64 * int(r.resident[0, 0]))


# ---------------------------------------------------------------- compressed-K writer
#
# The writer quantises key rows into records (scale = amax/448 in binary32, codes
# = nearest e4m3 of x / scale, ties to even). Its pins tie it to torch's e4m3 cast,
# to the workload generator's own records, to closed forms and to the geometry.

def _torch_decode(codes) -> np.ndarray:
    t = torch.as_tensor(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float32).numpy()


def _torch_encode(v) -> np.ndarray:
    t = torch.as_tensor(np.ascontiguousarray(v, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def pin_writer_encode_round_trip(o: O.Oracle):
    """Every finite e4m3 value encodes back to its own byte (signed zero too)."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    got = o.e4m3_encode(_torch_decode(codes))
    assert np.array_equal(got, codes), codes[got != codes]


def pin_writer_encode_vs_torch(o: O.Oracle):
    """Nearest with ties to even, as torch's cast: at every midpoint between
    neighbouring values, one binary32 step to either side of it, and on random
    values from the subnormal range to 448."""
    vals = np.sort(_torch_decode(np.arange(0, 127, dtype=np.uint8)))
    mid = ((vals[:-1].astype(np.float64) + vals[1:]) / 2).astype(np.float32)
    probes = np.concatenate([mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9))])
    rng = np.random.default_rng(11)
    rnd = (2.0 ** rng.uniform(-12, np.log2(448.0), 20000)).astype(np.float32)
    probes = np.concatenate([probes, rnd, vals])
    probes = np.concatenate([probes, -probes])
    assert np.array_equal(o.e4m3_encode(probes), _torch_encode(probes))


def pin_writer_matches_generator(o: O.Oracle):
    """The workload generator quantises its keys with numpy and torch; quantising
    the same drawn rows with the oracle gives the same 132-byte records."""
    w = synth.make_workload("wgen", num_q=1, history=[2 * PAGE], shuffle=False, seed=5, threads=1)
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(5, spawn_key=(1, 0))))
    x = g.standard_normal((2, PAGE, D), dtype=np.float32)
    for p in range(2):
        for r in range(PAGE):
            rec, flags = o.quantise_row(x[p, r])
            assert flags == 0
            assert np.array_equal(rec, w.kv[p, r * REC:(r + 1) * REC]), (p, r)


def pin_writer_closed_forms(o: O.Oracle):
    # zero row, and a row whose scale amax / 448 underflows: zero codes and zero scale
    rec, _ = o.quantise_row(np.zeros(D, np.float32))
    assert not rec.any()
    tiny = np.zeros(D, np.float32)
    tiny[[3, 40]] = np.array([1e-44, -3e-45], np.float32)  # subnormal; 1e-44 / 448 rounds to 0
    rec, _ = o.quantise_row(tiny)
    assert not rec.any()
    assert o.e4m3_encode(np.array([np.inf, -np.inf, 1e30], np.float32)).tolist() == [0x7E, 0xFE, 0x7E]
    # a row on the e4m3 grid whose largest magnitude is 448: scale 1, exact codes
    codes = np.random.default_rng(3).integers(0, 126, D).astype(np.uint8)
    codes[7] = 0x7E
    codes[::3] |= 0x80
    x = _torch_decode(codes)
    rec, _ = o.quantise_row(x)
    assert struct.unpack("<f", rec[D:].tobytes())[0] == 1.0 and np.array_equal(rec[:D], codes)
    # scaling by a power of two keeps the codes and scales the scale
    for e in (-20, -3, 5, 30):
        rec2, _ = o.quantise_row((x * np.float32(2.0 ** e)).astype(np.float32))
        assert np.array_equal(rec2[:D], codes)
        assert struct.unpack("<f", rec2[D:].tobytes())[0] == 2.0 ** e
    # a single nonzero value v: code +-448 and scale |v| / 448 in binary32
    for v in (3.0, -0.015625, 1234.5):
        row = np.zeros(D, np.float32)
        row[17] = v
        rec, _ = o.quantise_row(row)
        assert rec[17] == (0xFE if v < 0 else 0x7E) and not np.delete(rec[:D], 17).any()
        assert struct.unpack("<f", rec[D:].tobytes())[0] == np.float32(abs(v)) / np.float32(448.0)


def pin_writer_error_bound(o: O.Oracle):
    """decode(code) * scale is within half a code step of x / scale, times scale."""
    x = np.random.default_rng(8).standard_normal((40, D)).astype(np.float32) * np.float32(7.0)
    for row in x:
        rec, _ = o.quantise_row(row)
        s = struct.unpack("<f", rec[D:].tobytes())[0]
        y = row.astype(np.float64) / s
        back = _torch_decode(rec[:D]).astype(np.float64)
        step = np.where(np.abs(y) >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(y), 1e-30))) - 3), 2.0 ** -9)
        assert np.all(np.abs(back - y) <= step / 2 * (1 + 1e-6))


def pin_writer_geometry(o: O.Oracle):
    """Rows land at page_table[req][pos // 64], record pos % 64; nothing else is
    touched; invalid rows are skipped and flagged."""
    kv = np.full((4, PAGE * REC + 16), 0xA5, dtype=np.uint8)
    pt = np.array([[2, 0], [3, 1]], dtype=np.int32)
    rows = np.random.default_rng(4).standard_normal((6, D)).astype(np.float32)
    rows[5, 3] = np.nan
    req = np.array([0, 1, 7, 0, 1, 1], dtype=np.int32)
    pos = np.array([70, 5, 0, 128, 64, 9], dtype=np.int32)
    flags = o.write_keys(rows, req, pos, kv, pt)
    assert flags == O.BAD_REQUEST | O.LEN_OOB | O.RANGE, flags
    want = np.full_like(kv, 0xA5)
    for i, (page, r) in ((0, (0, 6)), (1, (3, 5)), (4, (1, 0))):
        want[page, r * REC:(r + 1) * REC] = o.quantise_row(rows[i])[0]
    assert np.array_equal(kv, want)
    # identity request map; a page id out of range
    kv2 = np.full_like(kv, 0xA5)
    pt2 = np.array([[1], [9]], dtype=np.int32)
    flags = o.write_keys(rows[:2], None, np.array([3, 2], np.int32), kv2, pt2)
    assert flags == O.PAGE_OOB
    want = np.full_like(kv, 0xA5)
    want[1, 3 * REC:4 * REC] = o.quantise_row(rows[0])[0]
    assert np.array_equal(kv2, want)


# ---------------------------------------------------------------- Level-1 recall

H1 = 128  # heads of the Memory Indexer's query


def recall_layers(n_layers: int, num_q: int, history, seed: int, zero_weights=(), **kw):
    """Target layers of a Level-1 problem: one generated cache per layer (same
    lengths, its own keys and page table) with a 128-head bf16 query and weights
    N(0,1) * 128^-0.5 * 128^-0.5."""
    layers = []
    for l in range(n_layers):
        w = synth.make_workload(f"l1_{l}", num_q=num_q, history=list(history), seed=seed + 17 * l, threads=1, **kw)
        rng = np.random.default_rng(seed + 101 * l)
        w.q = bf16_bits(rng.standard_normal((num_q, H1, D))).reshape(num_q, H1, D)
        w.fused_w = (rng.standard_normal((num_q, H1)) / np.sqrt(D) / np.sqrt(H1)).astype(np.float32)
        if l in zero_weights:
            w.fused_w[:] = 0.0
        layers.append(w)
    return layers


def _kept_tail_and_sink(L: int, sink: int, recent: int) -> np.ndarray:
    n = np.arange(L)
    return ((n < sink) | (n >= L - recent)).astype(np.uint8)


def pin_recall_zero_weights(o: O.Oracle):
    """With every weight 0 each layer scores 0.5 everywhere: a threshold of 0.5
    keeps every chunk, one just above keeps exactly the sink and the tail."""
    layers = recall_layers(2, 2, [200, 70], seed=31, zero_weights=(0, 1))
    P = [O.Problem(w) for w in layers]
    for mean in (False, True):
        keep, sc, pages, _ = o.recall(P, mean, 0.5, 3, 70)
        for b, L in enumerate((200, 70)):
            assert np.all(sc[b, :L] == 0.5) and np.all(keep[b, :L] == 1)
            assert list(pages[b]) == list(range((L + PAGE - 1) // PAGE))
        keep, sc, pages, _ = o.recall(P, mean, 0.5000001, 3, 70)
        assert np.array_equal(keep[0, :200], _kept_tail_and_sink(200, 3, 70))
        assert list(pages[0]) == [0, 2, 3]   # n < 3 and 130 <= n < 200
        assert np.all(keep[1, :70] == 1)   # the tail covers the whole row
    keep, sc, pages, _ = o.recall(P, False, 2.0, 0, 0)
    assert not keep[0, :200].any() and len(pages[0]) == 0


def pin_recall_matches_brute_force(o: O.Oracle):
    """Per-layer 128-head logits of an independent numpy restatement, sigmoid,
    then max or mean across three layers; the keep rule at the median score."""
    layers = recall_layers(3, 2, [130, 77], seed=32)
    brute = [brute_logits(w) for w in layers]
    P = [O.Problem(w) for w in layers]
    for mean in (False, True):
        want = {}
        for key in brute[0]:
            s = [1.0 / (1.0 + math.exp(-bl[key][0])) for bl in brute]
            want[key] = sum(s) / len(s) if mean else max(s)
        v = np.sort(np.array(list(want.values())))
        m = len(v) // 2
        while v[m + 1] - v[m] < 1e-9:  # a threshold between two scores, not on one
            m += 1
        thr = float((v[m] + v[m + 1]) / 2)
        keep, sc, pages, _ = o.recall(P, mean, thr, 2, 5)
        for (b, pos), e in want.items():
            assert abs(sc[b, pos] - e) <= 1e-12, (b, pos)
            L = int(layers[0].q_len[b])
            assert keep[b, pos] == int(e >= thr or pos < 2 or pos >= L - 5), (b, pos)
        for b in range(2):
            L = int(layers[0].q_len[b])
            kept_pages = sorted({p // PAGE for p in range(L) if keep[b, p]})
            assert list(pages[b]) == kept_pages


def pin_recall_ensemble_closed_form(o: O.Oracle):
    """Layer A has zero weights (0.5 everywhere); layer B a one-hot query on one
    head: its score is sigmoid(max(0, s * e4m3(byte[d0])) * w). Max and mean of the
    two follow in closed form."""
    layers = recall_layers(2, 1, [64], seed=33, zero_weights=(0,))
    wB = layers[1]
    q = np.zeros((1, H1, D), np.float32)
    q[0, 5, 9] = 1.0
    wB.q = bf16_bits(q).reshape(1, H1, D)
    wB.fused_w[:] = 0.0
    wB.fused_w[0, 5] = 0.75
    P = [O.Problem(w) for w in layers]
    phys = int(wB.page_table[0, 0])
    for mean in (False, True):
        _, sc, _, _ = o.recall(P, mean, 0.9, 0, 0)
        for r in range(PAGE):
            rec = wB.kv[phys, r * REC:(r + 1) * REC]
            s = struct.unpack("<f", rec[D:].tobytes())[0]
            x = float(torch.tensor([int(rec[9])], dtype=torch.uint8).view(torch.float8_e4m3fn).double().item())
            sB = 1.0 / (1.0 + math.exp(-max(0.0, s * x) * 0.75))
            want = (0.5 + sB) / 2 if mean else max(0.5, sB)
            assert abs(sc[0, r] - want) <= 1e-12


def pin_recall_rows_and_unreadable_pages(o: O.Oracle):
    """Rows come from layer 0 (another layer's q_len is ignored); a chunk on a page
    that a layer maps out of range scores 0 in that layer; a row with a request id
    out of range is empty. One layer: a threshold just above 0 keeps every readable
    chunk and no unreadable one outside the tail. Two layers, mean: the chunks of
    the unreadable page score half of the other layer's score."""
    layers = recall_layers(2, 3, [300, 300, 300], seed=34)
    layers[1].page_table = layers[1].page_table.copy()
    layers[1].page_table[0, 2] = layers[1].num_pages + 1   # row 0, positions 128..191
    keep1, sc1, pages1, f1 = o.recall([O.Problem(layers[1])], False, 1e-300, 0, 10)
    assert f1 & O.PAGE_OOB
    assert np.all(sc1[0, 128:192] == 0.0) and np.all(keep1[0, 128:192] == 0)
    assert np.all(keep1[0, :128] == 1) and np.all(keep1[0, 192:300] == 1)
    assert list(pages1[0]) == [0, 1, 3, 4]
    layers[1].q_len = np.array([5, 5, 5], np.int32)  # ignored: layer 0's rows rule
    layers[0].q_req = np.array([0, 1, 7], np.int32)  # row 2: request out of range
    layers[1].q_req = np.array([0, 1, 2], np.int32)  # ignored too
    P = [O.Problem(w) for w in layers]
    keep, sc, pages, flags = o.recall(P, True, 2.0, 0, 0)
    assert flags & O.PAGE_OOB and flags & O.BAD_REQUEST
    _, sc0, _, _ = o.recall([P[0]], False, 2.0, 0, 0)
    assert np.all(sc[0, 128:192] == sc0[0, 128:192] / 2)
    assert np.all(sc[0, :128] > sc0[0, :128] / 2)   # both layers score there
    assert sc[1, 299] > 0.0                          # layer 1's q_len of 5 is not used
    assert not keep[2].any() and len(pages[2]) == 0 and np.all(sc[2] == 0.0)


# ---------------------------------------------------------------- FP4 (MXFP4) variant

E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # OCP FP4 E2M1 magnitudes, codes 0..7


def _grid_block(rng, s):
    """32 values on the e2m1 grid times 2^s, the largest magnitude present."""
    top = float(rng.choice(E2M1_VALUES[1:]))
    mags = rng.choice([g for g in E2M1_VALUES if g <= top], 32)
    x = mags * rng.choice([-1.0, 1.0], 32) * 2.0 ** s
    x[int(rng.integers(32))] = top * 2.0 ** s
    return x.astype(np.float32)


def pin_fp4_e2m1_table(o: O.Oracle):
    """The 16 e2m1 codes decode to the OCP FP4 E2M1 table (sign in bit 3); a UE8M0
    byte is 2^(e - 127), 255 is NaN."""
    for c in range(16):
        want = E2M1_VALUES[c & 7] * (-1.0 if c & 8 else 1.0)
        got = o.e2m1(c)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), (c, got)
    for e in (0, 1, 100, 126, 127, 128, 254):
        assert o.ue8m0(e) == 2.0 ** (e - 127)
    assert math.isnan(o.ue8m0(255))


def pin_fp4_encode_nearest_even(o: O.Oracle):
    """Encoding picks the nearest e2m1 magnitude (brute force over the table), a tie
    goes to the even code, magnitudes at or past 6 saturate; the seven midpoints."""
    grid = np.array(E2M1_VALUES)
    rng = np.random.default_rng(41)
    for v in list(rng.uniform(-7.0, 7.0, 3000)) + [6.0, 6.5, 1e9, -1e9, 0.0]:
        c = o.e2m1_encode(v)
        a = abs(v)
        if a >= 6.0:
            assert c & 7 == 7, (v, c)
        else:
            d = np.abs(grid - a)
            best = np.flatnonzero(d == d.min())
            want = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
            assert c & 7 == want, (v, c, want)
        assert (c >> 3) == (1 if v < 0 else 0), (v, c)
    for v, want in ((0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0), (3.5, 4.0), (5.0, 4.0)):
        assert o.e2m1(o.e2m1_encode(v)) == want and o.e2m1(o.e2m1_encode(-v)) == -want, v


def pin_fp4_block_scale(o: O.Oracle):
    """OCP MX scale X = 2^(floor(log2 amax) - 2): amax in [4, 8) x 2^s gives the scale
    byte 127 + s, values past 6 X saturate; scaling a block by 2^k adds k to the byte
    and keeps the codes; a block of zeros has scale byte 0 and zero codes."""
    rng = np.random.default_rng(42)
    for s in (-20, -3, 0, 5, 30):
        x = (rng.uniform(-1.0, 1.0, 32) * 2.0 ** s).astype(np.float32)
        for top, sat in ((6.0, False), (4.0, False), (7.5, True)):
            x[7] = np.float32(top * 2.0 ** s)
            codes, sc = o.mxfp4_block(x)
            assert sc == 127 + s, (s, top, sc)
            assert (codes[7] == 7) if sat else (o.e2m1(int(codes[7])) == top), (s, top, codes[7])
            c2, sc2 = o.mxfp4_block((x * np.float32(8.0)).astype(np.float32))
            assert sc2 == sc + 3 and np.array_equal(c2, codes)
        x[7] = np.float32(3.9 * 2.0 ** s)  # floor(log2 3.9) = 1: X = 2^(s - 1), 7.8 saturates
        codes, sc = o.mxfp4_block(x)
        assert sc == 126 + s and codes[7] == 7
    codes, sc = o.mxfp4_block(np.zeros(32, np.float32))
    assert sc == 0 and not codes.any()


def pin_fp4_grid_round_trip(o: O.Oracle):
    """Blocks whose values lie on the e2m1 grid times a power of two come back exactly,
    whatever their largest magnitude (the scale then maps every value onto the grid)."""
    rng = np.random.default_rng(43)
    for _ in range(60):
        x = _grid_block(rng, int(rng.integers(-12, 12)))
        assert np.array_equal(o.mxfp4_round(x), x.astype(np.float64)), x


def pin_fp4_record_layout(o: O.Oracle):
    """A record is 64 code bytes (element 2j in the low nibble of byte j) then the four
    block scale bytes; decoding gives the row back when it lies on the grid."""
    rng = np.random.default_rng(44)
    x = np.concatenate([_grid_block(rng, s) for s in (-3, 0, 2, 7)])
    rec = o.fp4_record(x)
    codes = np.concatenate([o.mxfp4_block(x[32 * b:32 * b + 32])[0] for b in range(4)])
    for b in range(4):
        assert rec[64 + b] == o.mxfp4_block(x[32 * b:32 * b + 32])[1]
    for j in range(64):
        assert rec[j] == (codes[2 * j] | (codes[2 * j + 1] << 4)), j
    assert np.array_equal(o.fp4_decode(rec), x.astype(np.float64))


def pin_fp4_logit_equals_fp8_indexer(o: O.Oracle):
    """Keys and queries on the e2m1 grid (times powers of two per block) are exact both
    as MXFP4 and as e4m3 records with a power-of-two scale / bf16 queries: there the
    FP4 logit equals the logit of the FP8 indexer (pinned on its own above)."""
    rng = np.random.default_rng(45)
    keys = np.stack([np.concatenate([_grid_block(rng, int(rng.integers(-2, 3))) for _ in range(4)])
                     for _ in range(20)])
    q = np.stack([np.concatenate([_grid_block(rng, int(rng.integers(-3, 2))) for _ in range(4)])
                  for _ in range(H)])
    w = (rng.standard_normal(H) / 8.0).astype(np.float32)
    scale = 2.0 ** -3
    recs = np.stack([record({d: e4m3_code(float(keys[i, d]) / scale) for d in range(D)}, scale)
                     for i in range(keys.shape[0])])
    P = O.Problem(hand_workload(recs, q, w))
    qb = bf16_bits(q).reshape(H, D)
    for i in range(keys.shape[0]):
        lg8 = o.logit(P, 0, i)
        lg4 = o.fp4_logit(o.fp4_record(keys[i]), qb, w)
        assert abs(lg4 - lg8) <= 1e-12 * (1.0 + abs(lg8)), (i, lg4, lg8)


def pin_fp4_logit_composes_rounding(o: O.Oracle):
    """Off the grid: the FP4 logit is the relu'd, head-weighted sum over the decoded key
    and the block-rounded bf16 query (both pinned above), recomputed here with numpy."""
    rng = np.random.default_rng(46)
    for t in range(8):
        key = (rng.standard_normal(D) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        q = (rng.standard_normal((3, D)) * 10.0 ** rng.uniform(-2, 2)).astype(np.float32)
        w = rng.standard_normal(3).astype(np.float32)
        qb = bf16_bits(q).reshape(3, D)
        qf = torch.from_numpy(qb.view(np.int16)).view(torch.bfloat16).float().numpy()
        k = o.fp4_decode(o.fp4_record(key))
        want = sum(max(0.0, float(k @ o.mxfp4_round(qf[h]))) * float(w[h]) for h in range(3))
        got = o.fp4_logit(o.fp4_record(key), qb, w)
        assert abs(got - want) <= 1e-12 * (1.0 + abs(want)), (t, got, want)


def pin_fp4_paged_logits_match_records(o: O.Oracle):
    """Over a paged MXFP4 cache (full history and resident pages) the oracle's logit at
    every visible position is the per-record FP4 logit (pinned above) of the record
    that the page table and the position name."""
    for resident in (None, 2):
        base = synth.make_workload("fp4p", num_q=3, history=[300, 130, 64], resident_pages=resident,
                                   seed=47, threads=1)
        w = synth.mxfp4_cache(base, seed=48)
        P = O.Problem(w)
        lg, valid, flags = o.logits(P)
        assert flags == 0
        checked = 0
        for b in range(w.num_q):
            req = b if w.q_req is None else int(w.q_req[b])
            pos, col, _ = o.visible(P, b)
            assert valid[b].sum() == len(col)
            for n, c in zip(pos.tolist(), col.tolist()):
                page = int(w.page_table[req, n // PAGE])
                rec = w.kv[page, (n % PAGE) * 68:(n % PAGE + 1) * 68]
                want = o.fp4_logit(rec, w.q[b], w.fused_w[b])
                assert abs(lg[b, c] - want) <= 1e-12 * (1.0 + abs(want)), (b, n)
                checked += 1
        assert checked > 100


def pin_fp4_writer(o: O.Oracle):
    """The FP4 writer puts each valid row's record (oracle's fp4_record, pinned above)
    at page_table[req][pos / 64], row pos % 64, touches nothing else, and skips and
    flags a bad request, position, page or a non-finite value, in that order; the
    paged oracle then reads the rows back as its keys."""
    rng = np.random.default_rng(49)
    num_req, pts, num_pages = 3, 2, 8
    pt = rng.permutation(num_pages)[: num_req * pts].reshape(num_req, pts).astype(np.int32)
    kv = np.full((num_pages, 64 * 68), 0xA5, dtype=np.uint8)
    x = (rng.standard_normal((10, D)) * 10.0 ** rng.uniform(-3, 3, (10, 1))).astype(np.float32)
    req = np.array([0, 1, 2, 0, 3, -1, 1, 2, 0, 1], np.int32)
    pos = np.array([0, 70, 127, 5, 1, 2, 128, 64, 9, 30], np.int32)
    x[8, 3] = np.nan
    pt_bad = pt.copy()
    pt_bad[2, 1] = num_pages + 1                       # row 7 (request 2, position 64) lands on a bad page
    want = kv.copy()
    for i in range(10):
        if req[i] in (0, 1, 2) and 0 <= pos[i] < 128 and not (req[i] == 2 and pos[i] >= 64) and i != 8:
            page = int(pt_bad[req[i], pos[i] // 64])
            want[page, (pos[i] % 64) * 68:(pos[i] % 64 + 1) * 68] = o.fp4_record(x[i])
    got = kv.copy()
    flags = o.fp4_write_keys(x, req, pos, got, pt_bad)
    assert flags == O.BAD_REQUEST | O.LEN_OOB | O.PAGE_OOB | O.RANGE, flags
    assert np.array_equal(got, want)
    # written rows read back through the paged oracle: record i is row pos % 64 of its page
    for i in (0, 1, 3, 9):
        page = int(pt[req[i], pos[i] // 64])
        assert np.array_equal(o.fp4_decode(got[page, (pos[i] % 64) * 68:(pos[i] % 64 + 1) * 68]),
                              o.fp4_decode(o.fp4_record(x[i])))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
