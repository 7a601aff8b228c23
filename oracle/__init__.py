"""fp64 CPU oracle of the CSA indexer (ctypes binding of csa_oracle.c).

TEST INFRASTRUCTURE ONLY: tests/, the smoke check and the CPU-baseline leg of
the benchmark use it. The product package never imports this module, and this
module imports nothing from the product package.

What it computes (FlashMemory-DeepSeek-V4, "Retriever architecture" and
"compressed_k format"; "Two-level recall algorithm", Level 2):
    k      = e4m3(record[:128]) * fp32(record[128:132])
    logit  = sum_h relu(k . q_h) * fused_w_h
    score  = sigmoid(logit)
and the top-k records of each query by (logit desc, position asc); and the
compressed-K writer that produces such records from key rows (scale = amax/448,
codes = nearest e4m3 of x / scale in binary32).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libcsa_oracle.so")
_lock = threading.Lock()
_lib = None

PAGE_OOB = 1
RESIDENT_OOB = 2
RANGE = 4
BAD_REQUEST = 16
LEN_OOB = 32


def build(force: bool = False) -> str:
    """Compiles csa_oracle.c into oracle/libcsa_oracle.so (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
           "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Problem(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p),
        ("w", ctypes.c_void_p),
        ("num_q", ctypes.c_int32),
        ("H", ctypes.c_int32),
        ("D", ctypes.c_int32),
        ("kv", ctypes.c_void_p),
        ("num_pages", ctypes.c_int64),
        ("page_stride", ctypes.c_int64),
        ("page_table", ctypes.c_void_p),
        ("num_req", ctypes.c_int32),
        ("pt_stride", ctypes.c_int32),
        ("q_req", ctypes.c_void_p),
        ("q_len", ctypes.c_void_p),
        ("resident", ctypes.c_void_p),
        ("n_resident", ctypes.c_void_p),
        ("res_stride", ctypes.c_int32),
        ("format", ctypes.c_int32),
    ]


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(_Problem)
    lib.oracle_e4m3.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3.restype = ctypes.c_double
    lib.oracle_bf16.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16.restype = ctypes.c_double
    lib.oracle_scale.argtypes = [ctypes.c_void_p]
    lib.oracle_scale.restype = ctypes.c_double
    lib.oracle_sigmoid.argtypes = [ctypes.c_double]
    lib.oracle_sigmoid.restype = ctypes.c_double
    lib.oracle_logit.argtypes = [P, ctypes.c_int32, ctypes.c_int64]
    lib.oracle_logit.restype = ctypes.c_double
    lib.oracle_visible.argtypes = [P, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p]
    lib.oracle_visible.restype = ctypes.c_int64
    lib.oracle_logits.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    lib.oracle_logits.restype = ctypes.c_int32
    lib.oracle_topk.argtypes = [P, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p]
    lib.oracle_topk.restype = ctypes.c_int32
    lib.oracle_topk_sample.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                       ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_topk_sample.restype = ctypes.c_int64
    lib.oracle_threads.argtypes = []
    lib.oracle_threads.restype = ctypes.c_int32
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e4m3_encode_many.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    lib.oracle_e4m3_encode_many.restype = None
    lib.oracle_quantise_row.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_quantise_row.restype = ctypes.c_int32
    lib.oracle_write_keys.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                      ctypes.c_int32, ctypes.c_int32]
    lib.oracle_write_keys.restype = ctypes.c_int32
    lib.oracle_recall.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_double, ctypes.c_int64,
                                  ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_int32, ctypes.c_void_p]
    lib.oracle_recall.restype = ctypes.c_int32
    lib.oracle_e2m1.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1.restype = ctypes.c_double
    lib.oracle_ue8m0.argtypes = [ctypes.c_uint8]
    lib.oracle_ue8m0.restype = ctypes.c_double
    lib.oracle_e2m1_encode.argtypes = [ctypes.c_double]
    lib.oracle_e2m1_encode.restype = ctypes.c_uint8
    lib.oracle_mxfp4_block.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_mxfp4_block.restype = None
    lib.oracle_mxfp4_round.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    lib.oracle_mxfp4_round.restype = None
    lib.oracle_fp4_record.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_fp4_record.restype = None
    lib.oracle_fp4_decode.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_fp4_decode.restype = None
    lib.oracle_fp4_logit.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
    lib.oracle_fp4_logit.restype = ctypes.c_double
    lib.oracle_fp4_write_keys.argtypes = lib.oracle_write_keys.argtypes
    lib.oracle_fp4_write_keys.restype = ctypes.c_int32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB_PATH)
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


class Problem:
    """Keeps the host arrays alive and exposes them to the C oracle.

    Takes any object with the attributes of a synthetic workload: q (uint16 bf16
    bits [num_q, H, D]), fused_w, kv ([num_pages, page_stride] uint8),
    page_table, q_len, q_req, resident, n_resident, and the record format
    ("e4m3" or "mxfp4"; taken from the workload's `record_format` when not given).
    """

    FORMATS = {"e4m3": 0, "mxfp4": 1}

    def __init__(self, w, record_format=None):
        record_format = record_format or getattr(w, "record_format", "e4m3")
        c = np.ascontiguousarray
        self.q = c(w.q, dtype=np.uint16)
        self.fused_w = c(w.fused_w, dtype=np.float32)
        self.kv = c(w.kv, dtype=np.uint8)
        self.page_table = c(w.page_table, dtype=np.int32)
        self.q_len = c(w.q_len, dtype=np.int32)
        self.q_req = None if w.q_req is None else c(w.q_req, dtype=np.int32)
        self.resident = None if w.resident is None else c(w.resident, dtype=np.int32)
        self.n_resident = None if w.n_resident is None else c(w.n_resident, dtype=np.int32)
        self.num_q, self.H, self.D = (int(x) for x in self.q.shape)
        self.num_req, self.pt_stride = (int(x) for x in self.page_table.shape)
        self.res_stride = 0 if self.resident is None else int(self.resident.shape[1])
        self._s = _Problem(
            _ptr(self.q), _ptr(self.fused_w), self.num_q, self.H, self.D,
            _ptr(self.kv), int(self.kv.shape[0]), int(self.kv.shape[1]),
            _ptr(self.page_table), self.num_req, self.pt_stride,
            _ptr(self.q_req), _ptr(self.q_len), _ptr(self.resident), _ptr(self.n_resident),
            self.res_stride, self.FORMATS[record_format])

    @property
    def ref(self):
        return ctypes.byref(self._s)

    def score_stride(self) -> int:
        return 64 * max(self.res_stride if self.resident is not None else self.pt_stride, 1)


class Oracle:
    """The oracle's entry points bound to one build of csa_oracle.c."""

    def __init__(self, lib=None):
        self._lib = lib

    @property
    def lib(self):
        return self._lib if self._lib is not None else _load()

    def e4m3(self, byte: int) -> float:
        return self.lib.oracle_e4m3(int(byte) & 0xFF)

    def bf16(self, bits: int) -> float:
        return self.lib.oracle_bf16(int(bits) & 0xFFFF)

    def scale(self, record: np.ndarray) -> float:
        rec = np.ascontiguousarray(record, dtype=np.uint8)
        return self.lib.oracle_scale(rec.ctypes.data)

    def sigmoid(self, x: float) -> float:
        return self.lib.oracle_sigmoid(float(x))

    def logit(self, problem: Problem, b: int, position: int) -> float:
        return self.lib.oracle_logit(problem.ref, int(b), int(position))

    def visible(self, problem: Problem, b: int):
        return _visible(self.lib, problem, b)

    def logits(self, problem: Problem, stride: int | None = None):
        return _logits(self.lib, problem, stride)

    def scores(self, problem: Problem, stride: int | None = None):
        return _scores(self.lib, problem, stride)

    def topk(self, problem: Problem, k: int):
        return _topk(self.lib, problem, k)

    def e4m3_encode(self, values) -> np.ndarray:
        return _e4m3_encode(self.lib, values)

    def quantise_row(self, x):
        return _quantise_row(self.lib, x)

    def write_keys(self, keys, req, pos, kv, page_table) -> int:
        return _write_keys(self.lib, keys, req, pos, kv, page_table)

    def recall(self, layers, mean: bool, threshold: float, sink: int, recent: int):
        return _recall(self.lib, layers, mean, threshold, sink, recent)

    def e2m1(self, code: int) -> float:
        return float(self.lib.oracle_e2m1(int(code)))

    def ue8m0(self, byte: int) -> float:
        return float(self.lib.oracle_ue8m0(int(byte)))

    def e2m1_encode(self, v: float) -> int:
        return int(self.lib.oracle_e2m1_encode(float(v)))

    def mxfp4_block(self, x):
        return _mxfp4_block(self.lib, x)

    def mxfp4_round(self, x):
        return _mxfp4_round(self.lib, x)

    def fp4_record(self, x):
        return _fp4_record(self.lib, x)

    def fp4_decode(self, rec):
        return _fp4_decode(self.lib, rec)

    def fp4_logit(self, rec, q_bits, w):
        return _fp4_logit(self.lib, rec, q_bits, w)

    def fp4_write_keys(self, keys, req, pos, kv, page_table) -> int:
        return _write_keys(self.lib, keys, req, pos, kv, page_table, fp4=True)


def load_build(path: str) -> Oracle:
    """An Oracle bound to another build of csa_oracle.c (used by mutation tests)."""
    return Oracle(_bind(path))


def e4m3(byte: int) -> float:
    return Oracle().e4m3(byte)


def bf16(bits: int) -> float:
    return Oracle().bf16(bits)


def scale(record: np.ndarray) -> float:
    return Oracle().scale(record)


def sigmoid(x: float) -> float:
    return Oracle().sigmoid(x)


def logit(problem: Problem, b: int, position: int) -> float:
    return Oracle().logit(problem, b, position)


def visible(problem: Problem, b: int):
    """(positions, columns, flags) of the visible records of row b."""
    return _visible(_load(), problem, b)


def _visible(lib, problem: Problem, b: int):
    flags = ctypes.c_int32(0)
    n = lib.oracle_visible(problem.ref, int(b), None, None, ctypes.byref(flags))
    pos = np.zeros(max(n, 1), dtype=np.int64)
    col = np.zeros(max(n, 1), dtype=np.int64)
    lib.oracle_visible(problem.ref, int(b), pos.ctypes.data, col.ctypes.data, None)
    return pos[:n], col[:n], int(flags.value)


def logits(problem: Problem, stride: int | None = None):
    """(logits [num_q, stride] fp64 (NaN where invisible), valid mask, flags)."""
    return _logits(_load(), problem, stride)


def _logits(lib, problem: Problem, stride: int | None = None):
    stride = stride or problem.score_stride()
    out = np.full((problem.num_q, stride), np.nan, dtype=np.float64)
    valid = np.zeros((problem.num_q, stride), dtype=np.uint8)
    flags = lib.oracle_logits(problem.ref, out.ctypes.data, valid.ctypes.data, int(stride))
    return out, valid.astype(bool), int(flags)


def scores(problem: Problem, stride: int | None = None):
    """(scores [num_q, stride] fp64 (NaN where invisible), valid mask, flags)."""
    return _scores(_load(), problem, stride)


def _scores(lib, problem: Problem, stride: int | None = None):
    lg, valid, flags = _logits(lib, problem, stride)
    with np.errstate(over="ignore"):
        sc = 1.0 / (1.0 + np.exp(-lg))
    return sc, valid, flags


def topk(problem: Problem, k: int):
    """(idx int32 [num_q, k], score fp64, logit fp64, flags) by (logit desc, position asc)."""
    return _topk(_load(), problem, k)


def _topk(lib, problem: Problem, k: int):
    idx = np.zeros((problem.num_q, k), dtype=np.int32)
    sc = np.zeros((problem.num_q, k), dtype=np.float64)
    lg = np.zeros((problem.num_q, k), dtype=np.float64)
    flags = lib.oracle_topk(problem.ref, int(k), idx.ctypes.data, sc.ctypes.data, lg.ctypes.data)
    return idx, sc, lg, int(flags)


def topk_sample(problem: Problem, b0: int, b1: int, max_records: int, k: int):
    """Top-k of rows [b0, b1) over at most max_records visible records each.

    Returns (idx, score, records scored). Used to time the oracle on a bounded
    sample of a large workload.
    """
    n = b1 - b0
    idx = np.zeros((n, k), dtype=np.int32)
    sc = np.zeros((n, k), dtype=np.float64)
    scored = _load().oracle_topk_sample(problem.ref, int(b0), int(b1), int(max_records), int(k),
                                        idx.ctypes.data, sc.ctypes.data)
    return idx, sc, int(scored)


def threads() -> int:
    return int(_load().oracle_threads())


def _e4m3_encode(lib, values) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib.oracle_e4m3_encode_many(v.ctypes.data, int(v.size), out.ctypes.data)
    return out


def _quantise_row(lib, x):
    v = np.ascontiguousarray(x, dtype=np.float32)
    assert v.shape == (128,)
    rec = np.zeros(132, dtype=np.uint8)
    flags = lib.oracle_quantise_row(v.ctypes.data, rec.ctypes.data)
    return rec, int(flags)


def _write_keys(lib, keys, req, pos, kv, page_table, fp4: bool = False) -> int:
    """Writes key rows into `kv` ([num_pages, page_stride] uint8, C-contiguous) in
    place as e4m3 (132-byte) or, with fp4, MXFP4 (68-byte) records; returns the OR
    of the flag bits."""
    k = np.ascontiguousarray(keys, dtype=np.float32)
    assert k.ndim == 2 and k.shape[1] == 128
    assert kv.dtype == np.uint8 and kv.flags["C_CONTIGUOUS"]
    p = np.ascontiguousarray(pos, dtype=np.int32)
    r = None if req is None else np.ascontiguousarray(req, dtype=np.int32)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    fn = lib.oracle_fp4_write_keys if fp4 else lib.oracle_write_keys
    return int(fn(k.ctypes.data, int(k.shape[0]), _ptr(r), p.ctypes.data, kv.ctypes.data,
                                     int(kv.shape[0]), int(kv.shape[1]), pt.ctypes.data, int(pt.shape[0]),
                                     int(pt.shape[1])))


def e4m3_encode(values) -> np.ndarray:
    """binary32 values -> e4m3 codes (nearest, ties to even, saturating at 448)."""
    return _e4m3_encode(_load(), values)


def quantise_row(x):
    """One key row of 128 binary32 values -> (132-byte record, flags)."""
    return _quantise_row(_load(), x)


def write_keys(keys, req, pos, kv, page_table) -> int:
    return _write_keys(_load(), keys, req, pos, kv, page_table)


def _recall(lib, layers, mean: bool, threshold: float, sink: int, recent: int):
    """Level-1 recall over `layers` (a list of Problem, one per target layer).
    Returns (keep uint8 [num_q, stride], scores float64, pages list of arrays, flags)
    with stride = 64 * pt_stride."""
    n = len(layers)
    arr = (_Problem * n)(*[p._s for p in layers])
    num_q = layers[0].num_q
    stride = 64 * layers[0].pt_stride
    keep = np.zeros((num_q, stride), dtype=np.uint8)
    sc = np.zeros((num_q, stride), dtype=np.float64)
    ps = max(1, layers[0].pt_stride)
    pages = np.zeros((num_q, ps), dtype=np.int32)
    npg = np.zeros(num_q, dtype=np.int32)
    flags = lib.oracle_recall(ctypes.addressof(arr), n, 1 if mean else 0, float(threshold), int(sink), int(recent),
                              keep.ctypes.data, stride, sc.ctypes.data, pages.ctypes.data, ps, npg.ctypes.data)
    return keep, sc, [pages[b, :npg[b]].copy() for b in range(num_q)], int(flags)


def recall(layers, mean: bool, threshold: float, sink: int, recent: int):
    return _recall(_load(), layers, mean, threshold, sink, recent)


# ------------------------------------------------------------------ FP4 (MXFP4) variant

def _mxfp4_block(lib, x):
    """32 values -> (32 e2m1 codes, one per byte; the UE8M0 scale byte)."""
    v = np.ascontiguousarray(x, dtype=np.float32)
    assert v.shape == (32,)
    codes = np.zeros(32, dtype=np.uint8)
    sc = ctypes.c_uint8(0)
    lib.oracle_mxfp4_block(v.ctypes.data, codes.ctypes.data, ctypes.byref(sc))
    return codes, int(sc.value)


def _mxfp4_round(lib, x):
    """Values (length a multiple of 32) MXFP4-rounded block by block, as fp64."""
    v = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    assert v.size % 32 == 0
    out = np.zeros(v.size, dtype=np.float64)
    lib.oracle_mxfp4_round(v.ctypes.data, int(v.size), out.ctypes.data)
    return out


def _fp4_record(lib, x):
    """A key row of 128 values -> its 68-byte FP4 record."""
    v = np.ascontiguousarray(x, dtype=np.float32)
    assert v.shape == (128,)
    rec = np.zeros(68, dtype=np.uint8)
    lib.oracle_fp4_record(v.ctypes.data, rec.ctypes.data)
    return rec


def _fp4_decode(lib, rec):
    r = np.ascontiguousarray(rec, dtype=np.uint8)
    assert r.shape == (68,)
    k = np.zeros(128, dtype=np.float64)
    lib.oracle_fp4_decode(r.ctypes.data, k.ctypes.data)
    return k


def _fp4_logit(lib, rec, q_bits, w):
    """Logit of a 68-byte FP4 key record against q (bf16 bit patterns [H, 128]) and
    head weights w [H]; both sides MXFP4-rounded."""
    r = np.ascontiguousarray(rec, dtype=np.uint8)
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    wv = np.ascontiguousarray(w, dtype=np.float32)
    assert r.shape == (68,) and q.ndim == 2 and q.shape[1] == 128 and wv.shape == (q.shape[0],)
    return float(lib.oracle_fp4_logit(r.ctypes.data, q.ctypes.data, wv.ctypes.data, int(q.shape[0])))


def e2m1(code: int) -> float:
    return Oracle().e2m1(code)


def e2m1_encode(v: float) -> int:
    return Oracle().e2m1_encode(v)


def mxfp4_block(x):
    return _mxfp4_block(_load(), x)


def mxfp4_round(x):
    return _mxfp4_round(_load(), x)


def fp4_record(x):
    return _fp4_record(_load(), x)


def fp4_decode(rec):
    return _fp4_decode(_load(), rec)


def fp4_logit(rec, q_bits, w):
    return _fp4_logit(_load(), rec, q_bits, w)


def fp4_write_keys(keys, req, pos, kv, page_table) -> int:
    return _write_keys(_load(), keys, req, pos, kv, page_table, fp4=True)
