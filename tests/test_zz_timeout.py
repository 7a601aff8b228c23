"""The bounded waits: a wait that runs out ends the call with CSA_DEV_TIMEOUT
instead of hanging, and leaves the device clean.

A test build of the library (build.TEST_VARIANTS["timeout"], never the product
build) shortens the pipeline waits' limit to 20 us and makes the page walker
publish nothing for its first 200 us, so that the roles waiting on it run out.
No GPU fault, trap or endless loop is involved: every wait in the kernels has a
limit, after which it raises the CTA's abort flag; the other roles see the flag
at their next look, copies in flight are drained under the normal limit, TMEM
is freed, and the kernel ORs CSA_DEV_TIMEOUT into dev_status. A normal call
made afterwards in the same process (the product library) must still pass
parity, which it could not if a CTA had left TMEM allocated or a copy in flight.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import _parity
from sparse_attention_kv_e4m3_gb300 import native, synth

pytestmark = pytest.mark.gpu

CSA_DEV_TIMEOUT = 8


@pytest.fixture(scope="module")
def timeout_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_kv_e4m3_gb300 import build

    build.build()
    native.load()
    lib = ctypes.CDLL(build.build_test_variant("timeout"))
    vp = ctypes.c_void_p
    f = lib.csa_index_score_topk_fused
    f.argtypes = [ctypes.POINTER(native.Args), ctypes.c_int32, vp, vp, vp, ctypes.c_size_t, vp]
    f.restype = ctypes.c_int
    return lib


def test_a_wait_that_runs_out_reports_timeout_and_leaves_the_device_clean(timeout_lib):
    w = synth.make_workload("to", num_q=3, history=[5000, 2000, 700], seed=71)
    prob = native.Problem.from_workload(w)
    k = 64
    ws = native.alloc_workspace(prob, k)
    idx = torch.full((w.num_q, k), -7, dtype=torch.int32, device="cuda")
    vals = torch.zeros((w.num_q, k), dtype=torch.float32, device="cuda")
    a = prob.args()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = timeout_lib.csa_index_score_topk_fused(ctypes.byref(a), k, idx.data_ptr(), vals.data_ptr(), ws.data_ptr(),
                                                ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, native.status_str(st)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    status = int(prob.dev_status.item())
    assert status & CSA_DEV_TIMEOUT, status
    assert elapsed < 0.5, elapsed  # the short limit ended the call, not the 1 s drain bound

    # the device is clean: the product library's next call on the same problem is exact
    prob.dev_status.zero_()
    idx2, vals2 = native.csa_index_score_topk_fused(prob, k)
    torch.cuda.synchronize()
    assert int(prob.dev_status.item()) == 0
    _parity.check_topk(w, idx2.cpu().numpy(), vals2.cpu().numpy(), k)
    # and so is a second call of the test build, which times out the same way
    prob.dev_status.zero_()
    st = timeout_lib.csa_index_score_topk_fused(ctypes.byref(a), k, idx.data_ptr(), vals.data_ptr(), ws.data_ptr(),
                                                ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(prob.dev_status.item()) & CSA_DEV_TIMEOUT
    assert np.all(np.isfinite(vals2.cpu().numpy()))
