"""The fused score + top-k variant that allocates nothing.

Some callers cannot give the library device memory: a C host without a device
allocator, a plugin whose host application owns all device allocations, or a
decode loop that must not call cudaMalloc while it runs. For them
csa_index_score_topk_fused_static keeps its scratch in an array built into the
library. These tests call it through the C ABI and check that it returns what
the workspace-taking entry point returns, on two calls in a row (the second
with other shapes, so stale scratch from the first must not matter), and that
it turns away a request too large for the built-in array.
"""
import ctypes

import numpy as np
import pytest
import torch

import _parity
from sparse_attention_kv_e4m3_gb300 import native, synth

pytestmark = pytest.mark.gpu

CSA_ERR_WORKSPACE = 4


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_kv_e4m3_gb300 import build

    build.build()
    lib = native.load()
    f = lib.csa_index_score_topk_fused_static
    f.argtypes = [ctypes.POINTER(native.Args), ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return lib


def _static_call(lib, prob, k):
    idx = torch.full((prob.num_q, k), -7, dtype=torch.int32, device="cuda")
    vals = torch.full((prob.num_q, k), -7.0, dtype=torch.float32, device="cuda")
    a = prob.args()
    st = lib.csa_index_score_topk_fused_static(ctypes.byref(a), k, idx.data_ptr(), vals.data_ptr(),
                                               torch.cuda.current_stream().cuda_stream)
    assert st == 0, native.status_str(st)
    return idx, vals


def test_matches_workspace_entry_point_twice(lib):
    cases = [
        (synth.make_workload("na1", num_q=6, history=[20000, 7000, 300, 64, 12000, 1], seed=51), 512),
        (synth.make_workload("na2", num_q=3, history=[9000, 2600, 777], outlier_frac=0.05, seed=52), 100),
    ]
    for w, k in cases:
        prob = native.Problem.from_workload(w)
        ref_idx, ref_vals = native.csa_index_score_topk_fused(prob, k)
        idx, vals = _static_call(lib, prob, k)
        torch.cuda.synchronize()
        assert int(prob.dev_status.item()) == 0
        ri, rv = ref_idx.cpu().numpy(), ref_vals.cpu().numpy().astype(np.float64)
        gi, gv = idx.cpu().numpy(), vals.cpu().numpy().astype(np.float64)
        # same positions in the same order, same padding
        assert np.array_equal(gi, ri)
        assert np.max(np.abs(gv - rv)) <= _parity.STRICT_SCORE_TOL
        # and the oracle's set rule, as for every other top-k path
        _parity.check_topk(w, gi, gv.astype(np.float32), k)


def test_rejects_requests_beyond_the_builtin_scratch(lib):
    w = synth.make_workload("na3", num_q=2, history=[500, 300], seed=53)
    prob = native.Problem.from_workload(w)
    a = prob.args()
    # 3000 rows at k = 512 need about 13 MB of scratch, more than the 4 MiB built in;
    # the call must refuse before launching anything (the pointers are never read).
    a.num_q = 3000
    a.num_req = 3000
    idx = torch.empty((2, 512), dtype=torch.int32, device="cuda")
    st = lib.csa_index_score_topk_fused_static(ctypes.byref(a), 512, idx.data_ptr(), idx.data_ptr(),
                                               torch.cuda.current_stream().cuda_stream)
    assert st == CSA_ERR_WORKSPACE


def _static_need(num_q: int, k: int, sms: int) -> int:
    """The header's bound for csa_index_score_topk_fused_static, written out:
    256-byte-rounded 4 * (num_q + 2), plus (num_q + SMs) slots of
    16 + 8 * min(1024, k + k / 2) bytes rounded up to 16."""
    head = (4 * (num_q + 2) + 255) // 256 * 256
    slot = (16 + 8 * min(1024, k + k // 2) + 15) // 16 * 16
    return head + (num_q + sms) * slot


@pytest.mark.parametrize("k", [512, 1024])
def test_largest_request_that_fits_the_builtin_scratch(lib, k):
    """At the largest num_q the bound accepts on this GPU the call must run and
    match the workspace entry point exactly (the kernel writes slots up to
    num_q - 1 + grid - 1); one more row must be refused before anything runs."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    limit = (4 << 20)
    nq = 1
    while _static_need(nq + 1, k, sms) <= limit:
        nq += 1
    assert _static_need(nq, k, sms) <= limit < _static_need(nq + 1, k, sms)
    rng = np.random.default_rng(60 + k)
    hist = rng.integers(1, 3 * 64, size=nq).tolist()
    w = synth.make_workload("edge%d" % k, num_q=nq, history=hist, seed=61)
    prob = native.Problem.from_workload(w)
    ref_idx, ref_vals = native.csa_index_score_topk_fused(prob, k)
    idx, vals = _static_call(lib, prob, k)
    torch.cuda.synchronize()
    assert int(prob.dev_status.item()) == 0
    assert torch.equal(idx, ref_idx) and torch.equal(vals, ref_vals)
    # one row more: refused before launching (the pointers are never read)
    a = prob.args()
    a.num_q = nq + 1
    a.num_req = max(a.num_req, nq + 1)
    st = lib.csa_index_score_topk_fused_static(ctypes.byref(a), k, idx.data_ptr(), vals.data_ptr(),
                                               torch.cuda.current_stream().cuda_stream)
    assert st == CSA_ERR_WORKSPACE
