"""Seeded synthetic workloads for the CSA indexer.

This module only makes inputs: the query, the head weights, the paged FP8
compressed-K cache, the page table, the lengths and the resident lists. It
holds none of the indexer's arithmetic. The fp8 and bf16 encodings are done by
torch's own casts (round to nearest even). Both the CUDA path and the oracle
read the arrays made here; neither side is imported by this module.

Workload shapes follow the indexer plane of DeepSeek-V4 serving as the pages
describe it (FlashMemory-DeepSeek-V4, "Retriever architecture" and
"compressed_k format"; "Quick start" for KMAX = 96/192/384 resident pages at
256K/512K/1M context):

  q        bf16  ~ N(0, 1)                               [num_q, 64, 128]
  fused_w  fp32  = N(0, 1) * 128^-0.5 * 64^-0.5          [num_q, 64]
  record   128 e4m3 bytes of x / s, x ~ N(0, 1), then the fp32 scale
           s = amax(|x|) / 448 in 4 little-endian bytes   (132 bytes)
  page     64 records; pages `page_stride` bytes apart

Draw order from `numpy.random.Generator(PCG64(seed))`: lengths (when random),
q, fused_w, outlier mask, page permutation, resident lists. The K values of
physical page chunk c come from their own stream
`PCG64(SeedSequence(seed, spawn_key=(1, c)))`, so they can be drawn by several
threads and still be identical run to run.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field
from typing import Callable, Optional

import numpy as np
import torch

HEADS = 64
HEAD_DIM = 128
PAGE_RECORDS = 64
RECORD_BYTES = HEAD_DIM + 4
PAGE_BYTES = PAGE_RECORDS * RECORD_BYTES
E4M3_MAX = 448.0
_CHUNK_PAGES = 1024
FP4_RECORD_BYTES = HEAD_DIM // 2 + HEAD_DIM // 32  # 64 code bytes + 4 block-scale bytes
FP4_PAGE_BYTES = PAGE_RECORDS * FP4_RECORD_BYTES


@dataclass
class Workload:
    """Host arrays of one indexer problem, in the layout the C ABI takes."""

    name: str
    q: np.ndarray                    # uint16 [num_q, H, D] bf16 bit patterns
    fused_w: np.ndarray              # float32 [num_q, H]
    kv: np.ndarray                   # uint8 [num_pages, page_stride]
    page_table: np.ndarray           # int32 [num_req, pt_stride]
    q_len: np.ndarray                # int32 [num_q]
    q_req: Optional[np.ndarray] = None       # int32 [num_q] or None (identity)
    resident: Optional[np.ndarray] = None    # int32 [num_req, res_stride] or None
    n_resident: Optional[np.ndarray] = None  # int32 [num_req] or None
    meta: dict = field(default_factory=dict)
    record_format: str = "e4m3"              # "e4m3" (132-byte records) or "mxfp4" (68-byte)

    @property
    def num_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_req(self) -> int:
        return int(self.page_table.shape[0])

    @property
    def pt_stride(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def res_stride(self) -> int:
        return 0 if self.resident is None else int(self.resident.shape[1])

    @property
    def num_pages(self) -> int:
        return int(self.kv.shape[0])

    @property
    def page_stride(self) -> int:
        return int(self.kv.shape[1])

    def score_stride(self) -> int:
        """Columns of a score matrix that holds every visible record."""
        if self.resident is not None:
            return PAGE_RECORDS * max(self.res_stride, 1)
        return PAGE_RECORDS * max(self.pt_stride, 1)

    def visible_counts(self) -> np.ndarray:
        """Visible records per query row (geometry assumed valid)."""
        req = self.q_req if self.q_req is not None else np.arange(self.num_q)
        L = np.clip(self.q_len.astype(np.int64), 0, PAGE_RECORDS * self.pt_stride)
        if self.resident is None:
            return L
        out = np.zeros(self.num_q, dtype=np.int64)
        for b in range(self.num_q):
            r = int(req[b])
            pages = self.resident[r, : int(self.n_resident[r])].astype(np.int64)
            rows = np.clip(L[b] - pages * PAGE_RECORDS, 0, PAGE_RECORDS)
            out[b] = int(rows.sum())
        return out

    def k_bytes(self) -> int:
        """Bytes of K rows that the visible records occupy (132 or 68 per record)."""
        rec = FP4_RECORD_BYTES if self.record_format == "mxfp4" else RECORD_BYTES
        return int(self.visible_counts().sum()) * rec


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _fill_pages(kv: np.ndarray, seed: int, threads: int) -> None:
    """K values of every physical page: x ~ N(0,1), s = amax/448, bytes = e4m3(x/s)."""
    num_pages = kv.shape[0]
    chunks = [(c, c * _CHUNK_PAGES, min(num_pages, (c + 1) * _CHUNK_PAGES))
              for c in range((num_pages + _CHUNK_PAGES - 1) // _CHUNK_PAGES)]

    def work(item):
        c, p0, p1 = item
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(1, c))))
        x = g.standard_normal((p1 - p0, PAGE_RECORDS, HEAD_DIM), dtype=np.float32)
        amax = np.abs(x).max(axis=-1)
        s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
        y = np.clip(x / s[..., None], -E4M3_MAX, E4M3_MAX)
        codes = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        recs = kv[p0:p1, :PAGE_BYTES].reshape(p1 - p0, PAGE_RECORDS, RECORD_BYTES)
        recs[..., :HEAD_DIM] = codes
        recs[..., HEAD_DIM:] = s.astype("<f4").view(np.uint8).reshape(p1 - p0, PAGE_RECORDS, 4)

    if threads <= 1 or len(chunks) == 1:
        for it in chunks:
            work(it)
    else:
        with _cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, chunks))


def make_workload(
    name: str,
    *,
    num_q: int,
    history: np.ndarray | list | Callable,
    q_len: Optional[Callable] = None,
    single_request: bool = False,
    shuffle: bool = True,
    outlier_frac: float = 0.0,
    outlier_scale: float = 8.0,
    resident_pages: Optional[int] = None,
    page_pad: int = 0,
    seed: int = 0,
    threads: Optional[int] = None,
) -> Workload:
    """Builds one workload.

    history        records allocated per request: a list, or a callable
                   (rng, num_req) -> array drawn from the seeded generator.
    q_len          optional callable (history_array, num_q) -> per-row length;
                   default: each decode row sees its request's whole history.
    single_request all query rows read request 0 (chunked prefill).
    shuffle        random permutation of physical pages; else contiguous.
    outlier_frac   fraction of records whose stored scale is multiplied by
                   `outlier_scale` after quantisation (fp8 bytes unchanged).
    resident_pages distinct logical pages per request to score (resident mode).
    page_pad       extra bytes between pages (multiple of 16), filled with 0xA5.
    """
    if page_pad % 16:
        raise ValueError("page_pad must be a multiple of 16")
    rng = np.random.Generator(np.random.PCG64(seed))
    num_req = 1 if single_request else num_q
    hist = history(rng, num_req) if callable(history) else history
    hist = np.asarray(hist, dtype=np.int64).reshape(num_req)
    q = rng.standard_normal((num_q, HEADS, HEAD_DIM), dtype=np.float32)
    w = (rng.standard_normal((num_q, HEADS)) * HEAD_DIM ** -0.5 * HEADS ** -0.5).astype(np.float32)

    pages_per_req = (hist + PAGE_RECORDS - 1) // PAGE_RECORDS
    num_pages = int(pages_per_req.sum())
    pt_stride = int(max(1, pages_per_req.max()))
    stride = PAGE_BYTES + page_pad
    kv = np.full((max(num_pages, 1), stride), 0xA5, dtype=np.uint8)
    threads = threads if threads is not None else min(16, os.cpu_count() or 1)
    _fill_pages(kv, seed, threads)

    if outlier_frac > 0.0:
        mask = rng.random(kv.shape[0] * PAGE_RECORDS) < outlier_frac
        sc = kv[:, :PAGE_BYTES].reshape(-1, RECORD_BYTES)[:, HEAD_DIM:].copy().view("<f4").reshape(-1)
        sc[mask] *= np.float32(outlier_scale)
        kv[:, :PAGE_BYTES].reshape(-1, RECORD_BYTES)[:, HEAD_DIM:] = sc.view(np.uint8).reshape(-1, 4)

    phys = rng.permutation(num_pages) if shuffle else np.arange(num_pages)
    page_table = np.zeros((num_req, pt_stride), dtype=np.int32)
    base = 0
    for r in range(num_req):
        n = int(pages_per_req[r])
        page_table[r, :n] = phys[base:base + n]
        base += n

    if q_len is None:
        lens = hist.copy() if not single_request else np.full(num_q, hist[0])
    else:
        lens = np.asarray(q_len(hist, num_q), dtype=np.int64)
    lens = lens.astype(np.int32)

    resident = n_res = None
    if resident_pages is not None:
        res_stride = resident_pages
        resident = np.zeros((num_req, res_stride), dtype=np.int32)
        n_res = np.zeros(num_req, dtype=np.int32)
        for r in range(num_req):
            n = min(resident_pages, int(pages_per_req[r]))
            resident[r, :n] = rng.choice(int(pages_per_req[r]), size=n, replace=False)
            n_res[r] = n

    return Workload(
        name=name,
        q=_bf16_bits(q),
        fused_w=w,
        kv=kv,
        page_table=page_table,
        q_len=lens,
        q_req=np.zeros(num_q, dtype=np.int32) if single_request else None,
        resident=resident,
        n_resident=n_res,
        meta=dict(seed=seed, shuffle=shuffle, outlier_frac=outlier_frac,
                  resident_pages=resident_pages, page_pad=page_pad),
    )


LEVEL1_HEADS = 128


def level1_layers(w: Workload, n_layers: int, seed: int) -> list:
    """Target layers of a Level-1 recall over the history of `w`: each layer draws
    its own 128-head query and weights, N(0,1) and N(0,1) * 128^-0.5 * 128^-0.5
    (the distributions of the 64-head indexer inputs above, at 128 heads); the
    cache bytes, page table and rows of `w` stand in for every layer's cache."""
    out = []
    for l in range(n_layers):
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(7, l))))
        q = rng.standard_normal((w.num_q, LEVEL1_HEADS, HEAD_DIM), dtype=np.float32)
        fw = (rng.standard_normal((w.num_q, LEVEL1_HEADS)) * HEAD_DIM ** -0.5 * LEVEL1_HEADS ** -0.5)
        out.append(Workload(name=f"{w.name}_l{l}", q=_bf16_bits(q), fused_w=fw.astype(np.float32), kv=w.kv,
                            page_table=w.page_table, q_len=w.q_len, q_req=w.q_req, meta=dict(w.meta, layer=l)))
    return out


def mxfp4_cache(w: Workload, seed: int) -> Workload:
    """The same rows, lengths and page table over an MXFP4 cache (68-byte records:
    64 bytes of e2m1 codes, element 2j in the low nibble of byte j, then 4 UE8M0
    block-scale bytes). The records are drawn directly, codes as uniform bytes and
    scale bytes in [124, 128] (block scales 2^-3 .. 2^1), so nothing is quantised
    here; from `PCG64(SeedSequence(seed, spawn_key=(9,)))`."""
    import dataclasses

    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(9,))))
    n = w.kv.shape[0]
    kv = np.zeros((n, FP4_PAGE_BYTES), dtype=np.uint8)
    recs = kv.reshape(n, PAGE_RECORDS, FP4_RECORD_BYTES)
    recs[..., :HEAD_DIM // 2] = rng.integers(0, 256, size=(n, PAGE_RECORDS, HEAD_DIM // 2), dtype=np.uint8)
    recs[..., HEAD_DIM // 2:] = rng.integers(124, 129, size=(n, PAGE_RECORDS, HEAD_DIM // 32), dtype=np.uint8)
    return dataclasses.replace(w, kv=kv, record_format="mxfp4", meta=dict(w.meta, record_format="mxfp4"))


def _uniform(lo: int, hi: int):
    return lambda rng, n: rng.integers(lo, hi + 1, size=n)


def _prefill_primary(hist, num_q):
    # row t sees positions below t//4 + 1024, capped by the history
    t = np.arange(num_q)
    return np.minimum(int(hist[0]), t // 4 + 1024)


def _prefill_tail(hist, num_q):
    # the chunk is the last num_q tokens of the history: row t sees N - 1024 + t//4 + 1
    t = np.arange(num_q)
    return np.minimum(int(hist[0]), int(hist[0]) - 1024 + t // 4 + 1)


# The five workloads the indexer is measured and checked on.
CONFIGS = {
    "tiny_decode": dict(num_q=1, history=[4096], shuffle=False),
    "decode_batch": dict(num_q=32, history=[32768] * 32),
    "long_ragged_decode": dict(num_q=64, history=_uniform(65536, 131072), outlier_frac=0.05),
    "resident_1m": dict(num_q=16, history=[262144] * 16, resident_pages=384),
    "prefill_chunk": dict(num_q=4096, history=[16384], single_request=True, q_len=_prefill_primary),
    "prefill_chunk_tail": dict(num_q=4096, history=[16384], single_request=True, q_len=_prefill_tail),
}


def config(name: str, seed: int = 0, **overrides) -> Workload:
    kw = dict(CONFIGS[name])
    kw.update(overrides)
    return make_workload(name, seed=seed, **kw)
