"""Thin Python binding of libcsa_index.so (include/csa_index.h).

Argument marshalling only: every step of the indexer runs in the library's CUDA
kernels. PyTorch supplies device memory and the current stream. The library
must have been built (`sparse_attention_kv_e4m3_gb300.build.build()`); there is
no fallback, and calling without it raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

from . import build as _build

CSA_OK = 0
STATUS_NAMES = {0: "CSA_OK", 1: "CSA_ERR_INVALID_ARG", 2: "CSA_ERR_UNSUPPORTED", 3: "CSA_ERR_ALIGNMENT",
                4: "CSA_ERR_WORKSPACE", 5: "CSA_ERR_CUDA"}
DEV_PAGE_OOB, DEV_RESIDENT_OOB, DEV_RANGE, DEV_TIMEOUT, DEV_BAD_REQUEST, DEV_LEN_OOB = 1, 2, 4, 8, 16, 32
HEAD_DIM, NUM_HEADS, RECORD_BYTES, PAGE_RECORDS, PAGE_BYTES, MAX_K, MAX_CTAS = 128, 64, 132, 64, 8448, 1024, 1024


class CsaError(RuntimeError):
    def __init__(self, what: str, status: int, text: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({text})")
        self.status = status


class Args(ctypes.Structure):
    """Mirror of `csa_index_args`."""

    _fields_ = [
        ("q", ctypes.c_void_p),
        ("fused_w", ctypes.c_void_p),
        ("num_q", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("kv", ctypes.c_void_p),
        ("num_pages", ctypes.c_int64),
        ("page_stride_bytes", ctypes.c_int64),
        ("page_table", ctypes.c_void_p),
        ("num_req", ctypes.c_int32),
        ("pt_stride", ctypes.c_int32),
        ("q_req", ctypes.c_void_p),
        ("q_len", ctypes.c_void_p),
        ("resident", ctypes.c_void_p),
        ("n_resident", ctypes.c_void_p),
        ("res_stride", ctypes.c_int32),
        ("record_format", ctypes.c_int32),
        ("dev_status", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def load(path: Optional[str] = None):
    """Loads the library (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is missing: build it with sparse_attention_kv_e4m3_gb300.build.build()")
            lib = ctypes.CDLL(p)
            A = ctypes.POINTER(Args)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            lib.csa_index_abi_version.argtypes = []
            lib.csa_index_abi_version.restype = i32
            lib.csa_status_str.argtypes = [ctypes.c_int]
            lib.csa_status_str.restype = ctypes.c_char_p
            lib.csa_index_workspace_bytes.argtypes = [A, i32]
            lib.csa_index_workspace_bytes.restype = sz
            lib.csa_index_score.argtypes = [A, vp, i64, vp]
            lib.csa_index_score.restype = ctypes.c_int
            lib.csa_index_topk.argtypes = [vp, i64, A, i32, vp, vp, vp, sz, vp]
            lib.csa_index_topk.restype = ctypes.c_int
            lib.csa_index_score_topk_fused.argtypes = [A, i32, vp, vp, vp, sz, vp]
            lib.csa_index_score_topk_fused.restype = ctypes.c_int
            lib.csa_index_score_topk_fused_marked.argtypes = [A, i32, vp, vp, vp, sz, vp, vp]
            lib.csa_index_score_topk_fused_marked.restype = ctypes.c_int
            lib.csa_index_write_keys.argtypes = [ctypes.POINTER(WriteArgs), vp]
            lib.csa_index_write_keys.restype = ctypes.c_int
            lib.csa_index_logits.argtypes = [A, vp, i64, vp]
            lib.csa_index_logits.restype = ctypes.c_int
            lib.csa_recall_workspace_bytes.argtypes = [ctypes.POINTER(RecallArgs)]
            lib.csa_recall_workspace_bytes.restype = sz
            lib.csa_recall_level1.argtypes = [ctypes.POINTER(RecallArgs), vp, sz, vp]
            lib.csa_recall_level1.restype = ctypes.c_int
            lib.csa_index_merge_topk.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp]
            lib.csa_index_merge_topk.restype = ctypes.c_int
            _lib = lib
    return _lib


KEYS_F32, KEYS_BF16 = 0, 1
RECORD_E4M3, RECORD_MXFP4 = 0, 1


class WriteArgs(ctypes.Structure):
    """Mirror of csa_write_args."""
    _fields_ = [
        ("keys", ctypes.c_void_p),
        ("key_dtype", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("n", ctypes.c_int64),
        ("row_req", ctypes.c_void_p),
        ("row_pos", ctypes.c_void_p),
        ("kv", ctypes.c_void_p),
        ("num_pages", ctypes.c_int64),
        ("page_stride_bytes", ctypes.c_int64),
        ("page_table", ctypes.c_void_p),
        ("num_req", ctypes.c_int32),
        ("pt_stride", ctypes.c_int32),
        ("dev_status", ctypes.c_void_p),
    ]


ENSEMBLE_MAX, ENSEMBLE_MEAN = 0, 1


class RecallArgs(ctypes.Structure):
    """Mirror of csa_recall_args."""
    _fields_ = [
        ("layers", ctypes.c_void_p),
        ("n_layers", ctypes.c_int32),
        ("ensemble", ctypes.c_int32),
        ("threshold", ctypes.c_float),
        ("sink", ctypes.c_int32),
        ("recent", ctypes.c_int32),
        ("pages_stride", ctypes.c_int32),
        ("keep", ctypes.c_void_p),
        ("keep_stride", ctypes.c_int64),
        ("pages", ctypes.c_void_p),
        ("n_pages", ctypes.c_void_p),
        ("scores", ctypes.c_void_p),
    ]


def status_str(status: int) -> str:
    return load().csa_status_str(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(st: int, what: str):
    if st != CSA_OK:
        raise CsaError(what, st, status_str(st))


@dataclass
class Problem:
    """Device tensors of one indexer call (the fields of `csa_index_args`).

    q [num_q, 64, 128] bf16; fused_w [num_q, 64] fp32; kv [num_pages, page_stride]
    uint8; page_table [num_req, pt_stride] int32; q_len [num_q] int32; optional
    q_req [num_q], resident [num_req, res_stride], n_resident [num_req] int32 and
    dev_status [1] int32.
    """

    q: Optional[torch.Tensor]
    fused_w: Optional[torch.Tensor]
    kv: Optional[torch.Tensor]
    page_table: Optional[torch.Tensor]
    q_len: torch.Tensor
    q_req: Optional[torch.Tensor] = None
    resident: Optional[torch.Tensor] = None
    n_resident: Optional[torch.Tensor] = None
    dev_status: Optional[torch.Tensor] = None
    num_req: Optional[int] = None
    record_format: int = 0  # RECORD_E4M3 or RECORD_MXFP4

    def args(self) -> Args:
        a = Args()
        nq = int(self.q_len.shape[0])
        a.q = _ptr(self.q)
        a.fused_w = _ptr(self.fused_w)
        a.num_q = nq
        a.num_heads = int(self.q.shape[1]) if self.q is not None else NUM_HEADS
        a.head_dim = int(self.q.shape[2]) if self.q is not None else HEAD_DIM
        a.kv = _ptr(self.kv)
        if self.kv is not None:
            a.num_pages = int(self.kv.shape[0])
            a.page_stride_bytes = int(self.kv.stride(0)) * self.kv.element_size()
        a.page_table = _ptr(self.page_table)
        if self.page_table is not None:
            a.num_req = int(self.page_table.shape[0])
            a.pt_stride = int(self.page_table.stride(0))
        if self.num_req is not None:
            a.num_req = int(self.num_req)
        a.q_req = _ptr(self.q_req)
        a.q_len = _ptr(self.q_len)
        a.resident = _ptr(self.resident)
        a.n_resident = _ptr(self.n_resident)
        if self.resident is not None:
            a.res_stride = int(self.resident.stride(0))
        a.dev_status = _ptr(self.dev_status)
        a.record_format = int(self.record_format)
        return a

    @property
    def num_q(self) -> int:
        return int(self.q_len.shape[0])

    def score_stride(self) -> int:
        a = self.args()
        return PAGE_RECORDS * max(a.res_stride if self.resident is not None else a.pt_stride, 1)

    @staticmethod
    def from_workload(w, device="cuda", dev_status: bool = True) -> "Problem":
        """Copies a host workload (synth.Workload) to the device."""
        def t(x, dtype=None):
            if x is None:
                return None
            return torch.from_numpy(x).to(device=device, dtype=dtype) if dtype else torch.from_numpy(x).to(device)

        q = torch.from_numpy(w.q.view("int16")).to(device).view(torch.bfloat16)
        return Problem(
            q=q, fused_w=t(w.fused_w), kv=t(w.kv), page_table=t(w.page_table), q_len=t(w.q_len),
            q_req=t(w.q_req), resident=t(w.resident), n_resident=t(w.n_resident),
            dev_status=torch.zeros(1, dtype=torch.int32, device=device) if dev_status else None,
            record_format=RECORD_MXFP4 if getattr(w, "record_format", "e4m3") == "mxfp4" else RECORD_E4M3)


def workspace_bytes(problem_or_args, k: int) -> int:
    a = problem_or_args.args() if isinstance(problem_or_args, Problem) else problem_or_args
    return int(load().csa_index_workspace_bytes(ctypes.byref(a), int(k)))


def alloc_workspace(problem: Problem, k: int, device="cuda") -> torch.Tensor:
    n = workspace_bytes(problem, k)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def csa_index_score(problem: Problem, scores: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Scores of every visible record; invisible columns keep their initial value (NaN)."""
    a = problem.args()
    if scores is None:
        scores = torch.full((problem.num_q, problem.score_stride()), float("nan"), dtype=torch.float32,
                            device=problem.q_len.device)
    st = load().csa_index_score(ctypes.byref(a), scores.data_ptr(), int(scores.stride(0)), _stream(stream))
    _check(st, "csa_index_score")
    return scores


def csa_index_score_topk_fused(problem: Problem, k: int = 512, ws: Optional[torch.Tensor] = None,
                               idx: Optional[torch.Tensor] = None, vals: Optional[torch.Tensor] = None,
                               stream=None, mark: Optional[torch.cuda.Event] = None):
    """Fused score + top-k. Returns (idx int32 [num_q, k], vals fp32 [num_q, k]).

    `mark`, when given, is recorded between the scoring and the merge kernel."""
    a = problem.args()
    dev = problem.q_len.device
    if ws is None:
        ws = alloc_workspace(problem, k, dev)
    if idx is None:
        idx = torch.empty((problem.num_q, k), dtype=torch.int32, device=dev)
    if vals is None:
        vals = torch.empty((problem.num_q, k), dtype=torch.float32, device=dev)
    if mark is None:
        st = load().csa_index_score_topk_fused(ctypes.byref(a), int(k), idx.data_ptr(), vals.data_ptr(),
                                               ws.data_ptr(), ws.numel(), _stream(stream))
    else:
        # torch only lets elapsed_time() read events it recorded itself: record once
        # here; the library records the same event again between its two kernels.
        mark.record(torch.cuda.current_stream() if stream is None else stream)
        st = load().csa_index_score_topk_fused_marked(ctypes.byref(a), int(k), idx.data_ptr(), vals.data_ptr(),
                                                      ws.data_ptr(), ws.numel(), _stream(stream),
                                                      ctypes.c_void_p(mark.cuda_event))
    _check(st, "csa_index_score_topk_fused")
    return idx, vals


class PreparedFused:
    """`csa_index_score_topk_fused` with its arguments marshalled once, for a
    serving loop that repeats the same call on the same buffers: calling the
    object issues the call again (about half the host time of the plain binding,
    which builds the argument struct on every call). The tensors are kept alive
    here; they must not be resized or reallocated while the object is used, and
    their contents may change between calls (new queries, lengths, pages).

    `mark`, when given, is recorded between the scoring and the merge kernel."""

    def __init__(self, problem: Problem, k: int, ws: torch.Tensor, idx: torch.Tensor, vals: torch.Tensor,
                 stream=None):
        nq = problem.num_q
        if tuple(idx.shape) != (nq, k) or tuple(vals.shape) != (nq, k):
            raise ValueError(f"idx and vals must be [{nq}, {k}]")
        if idx.dtype != torch.int32 or vals.dtype != torch.float32 or ws.dtype != torch.uint8:
            raise ValueError("idx int32, vals float32, ws uint8")
        lib = load()
        self._keep = (problem, ws, idx, vals)
        self._args = problem.args()
        self._stream = stream if stream is not None else torch.cuda.current_stream()
        self._fn = lib.csa_index_score_topk_fused
        self._fn_marked = lib.csa_index_score_topk_fused_marked
        self._call = (ctypes.byref(self._args), int(k), idx.data_ptr(), vals.data_ptr(), ws.data_ptr(),
                      ws.numel(), self._stream.cuda_stream)

    def __call__(self, mark: Optional[torch.cuda.Event] = None) -> None:
        if mark is None:
            st = self._fn(*self._call)
        else:
            mark.record(self._stream)  # see csa_index_score_topk_fused
            st = self._fn_marked(*self._call, ctypes.c_void_p(mark.cuda_event))
        if st != CSA_OK:
            _check(st, "csa_index_score_topk_fused")


def csa_index_topk(scores: torch.Tensor, problem: Problem, k: int = 512, ws: Optional[torch.Tensor] = None,
                   idx: Optional[torch.Tensor] = None, vals: Optional[torch.Tensor] = None, stream=None):
    """Top-k over a score matrix laid out as csa_index_score writes it."""
    a = problem.args()
    dev = problem.q_len.device
    if ws is None:
        ws = alloc_workspace(problem, k, dev)
    if idx is None:
        idx = torch.empty((problem.num_q, k), dtype=torch.int32, device=dev)
    if vals is None:
        vals = torch.empty((problem.num_q, k), dtype=torch.float32, device=dev)
    st = load().csa_index_topk(scores.data_ptr(), int(scores.stride(0)), ctypes.byref(a), int(k), idx.data_ptr(),
                               vals.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream))
    _check(st, "csa_index_topk")
    return idx, vals


def csa_index_write_keys(keys: torch.Tensor, row_pos: torch.Tensor, kv: torch.Tensor, page_table: torch.Tensor,
                         row_req: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None,
                         stream=None) -> None:
    """Compressed-K writer: quantises key rows `keys` [n, 128] (fp32 or bf16) into
    records of the paged cache `kv` [num_pages, page_stride] (uint8), row i at
    logical position row_pos[i] of request row_req[i] (identity when None), through
    `page_table` [num_req, pt_stride]. Every tensor is on the GPU."""
    if keys.dtype == torch.float32:
        dt = KEYS_F32
    elif keys.dtype == torch.bfloat16:
        dt = KEYS_BF16
    else:
        raise TypeError("keys must be float32 or bfloat16")
    assert keys.dim() == 2 and keys.shape[1] == HEAD_DIM and keys.is_contiguous()
    assert kv.dtype == torch.uint8 and kv.dim() == 2 and kv.is_contiguous()
    assert row_pos.dtype == torch.int32 and page_table.dtype == torch.int32
    pt = page_table.contiguous()
    a = WriteArgs(keys.data_ptr(), dt, 0, int(keys.shape[0]), _ptr(row_req), row_pos.data_ptr(), kv.data_ptr(),
                  int(kv.shape[0]), int(kv.shape[1]), pt.data_ptr(), int(pt.shape[0]), int(pt.shape[1]),
                  _ptr(dev_status))
    _check(load().csa_index_write_keys(ctypes.byref(a), _stream(stream)), "csa_index_write_keys")


def csa_index_merge_topk(idx: torch.Tensor, vals: torch.Tensor, k: int, out_idx: Optional[torch.Tensor] = None,
                         out_vals: Optional[torch.Tensor] = None, stream=None):
    """Exact top-k per row from G gathered top-k lists: idx int32 and vals fp32,
    both [G, num_q, k_in] on the device. Returns (out_idx [num_q, k], out_vals)."""
    if idx.dim() != 3 or vals.shape != idx.shape or idx.dtype != torch.int32 or vals.dtype != torch.float32:
        raise ValueError("idx int32 and vals fp32 of one shape [G, num_q, k_in]")
    idx, vals = idx.contiguous(), vals.contiguous()
    g, nq, k_in = idx.shape
    if out_idx is None:
        out_idx = torch.empty((nq, k), dtype=torch.int32, device=idx.device)
    if out_vals is None:
        out_vals = torch.empty((nq, k), dtype=torch.float32, device=idx.device)
    _check(load().csa_index_merge_topk(idx.data_ptr(), vals.data_ptr(), int(g), int(nq), int(k_in), int(k),
                                       out_idx.data_ptr(), out_vals.data_ptr(), _stream(stream)),
           "csa_index_merge_topk")
    return out_idx, out_vals


def csa_index_logits(problem: "Problem", logits: Optional[torch.Tensor] = None, stride=None, stream=None):
    """csa_index_score writing logits (before the sigmoid). Returns the [num_q, stride] tensor."""
    a = problem.args()
    stride = stride or problem.score_stride()
    if logits is None:
        logits = torch.full((problem.num_q, stride), float("nan"), dtype=torch.float32, device=problem.q_len.device)
    _check(load().csa_index_logits(ctypes.byref(a), logits.data_ptr(), int(stride), _stream(stream)),
           "csa_index_logits")
    return logits


def csa_recall_level1(layers, mean: bool = False, threshold: float = 0.5, sink: int = 0, recent: int = 0,
                      scores: bool = True, ws: Optional[torch.Tensor] = None, out=None, stream=None):
    """Level-1 recall over `layers` (one Problem per target layer, 128-head queries).
    Returns (keep uint8 [num_q, stride], pages int32 [num_q, pt_stride], n_pages int32 [num_q],
    scores fp32 [num_q, stride] or None), stride = 64 * pt_stride; `out` may hold these four
    tensors, preallocated (keep and scores with equal row strides)."""
    args = [p.args() for p in layers]
    arr = (Args * len(args))(*args)
    p0 = layers[0]
    num_q, pts = p0.num_q, int(p0.page_table.shape[1])
    stride = PAGE_RECORDS * pts
    dev = p0.q_len.device
    if out is None:
        keep = torch.zeros((num_q, stride), dtype=torch.uint8, device=dev)
        pages = torch.full((num_q, pts), -1, dtype=torch.int32, device=dev)
        npg = torch.zeros(num_q, dtype=torch.int32, device=dev)
        sc = torch.full((num_q, stride), float("nan"), dtype=torch.float32, device=dev) if scores else None
    else:
        keep, pages, npg, sc = out
        stride = int(keep.stride(0))
        assert sc is None or int(sc.stride(0)) == stride
    ra = RecallArgs(ctypes.addressof(arr), len(args), ENSEMBLE_MEAN if mean else ENSEMBLE_MAX, float(threshold),
                    int(sink), int(recent), int(pages.stride(0)), keep.data_ptr(), stride, pages.data_ptr(),
                    npg.data_ptr(), _ptr(sc))
    need = load().csa_recall_workspace_bytes(ctypes.byref(ra))
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check(load().csa_recall_level1(ctypes.byref(ra), ws.data_ptr(), ws.numel(), _stream(stream)),
           "csa_recall_level1")
    return keep, pages, npg, sc
