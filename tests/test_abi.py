"""The C ABI without a GPU: the library builds and loads, exports every symbol the
header declares, the ctypes mirror matches the C struct layout, the workspace
size is pure arithmetic and bad host arguments are rejected before any launch."""
import ctypes
import os
import re
import subprocess

import pytest

from sparse_attention_kv_e4m3_gb300 import build, native

HEADER = os.path.join(build.INCLUDE, "csa_index.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return native.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"csa_index_score", "csa_index_topk", "csa_index_score_topk_fused", "csa_index_workspace_bytes",
            "csa_status_str", "csa_index_abi_version"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_struct_layout_matches_header(tmp_path):
    fields = [f[0] for f in native.Args._fields_]
    src = tmp_path / "layout.c"
    body = "".join(f'printf("{f} %zu\\n", offsetof(csa_index_args, {f}));' for f in fields)
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "csa_index.h"\n'
                   'int main(void){' + body + 'printf("sizeof %zu\\n", sizeof(csa_index_args));return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", f"-I{build.INCLUDE}", "-o", str(exe), str(src)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                        check=True).stdout.splitlines())
    for f in fields:
        assert int(got[f]) == getattr(native.Args, f).offset, f
    assert int(got["sizeof"]) == ctypes.sizeof(native.Args)


def test_version_and_strings(lib):
    assert lib.csa_index_abi_version() == 4
    for s in range(6):
        assert native.status_str(s)
    assert native.status_str(99) == "unknown status"


def test_workspace_bytes_is_host_arithmetic(lib):
    a = native.Args()
    a.num_q = 64
    slots = 64 + native.MAX_CTAS
    # a slot holds up to min(1024, k + k/2) keys of 8 bytes after a 16-byte header
    assert native.workspace_bytes(a, 512) == 512 + slots * (16 + 8 * 768)
    assert native.workspace_bytes(a, 1000) == 512 + slots * (16 + 8 * 1024)
    # from 512 rows the fused path takes the short-row scorer: a slot holds a whole
    # uncut row of up to 2048 keys, whatever k
    a.num_q = 600
    assert native.workspace_bytes(a, 512) == 2560 + (600 + native.MAX_CTAS) * (16 + 8 * 2048)
    assert native.workspace_bytes(a, 8) == 2560 + (600 + native.MAX_CTAS) * (16 + 8 * 2048)
    a.num_q = 64
    assert native.workspace_bytes(a, 0) == 0
    assert native.workspace_bytes(a, native.MAX_K + 1) == 0
    a.num_q = -1
    assert native.workspace_bytes(a, 8) == 0


def _fake_args(**kw):
    """Host-side args with well-aligned fake device addresses: validation only."""
    a = native.Args()
    a.q, a.fused_w, a.kv, a.page_table, a.q_len = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000
    a.num_q, a.num_heads, a.head_dim = 4, 64, 128
    a.num_pages, a.page_stride_bytes = 16, native.PAGE_BYTES
    a.num_req, a.pt_stride = 4, 4
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("change,want", [
    (dict(head_dim=64), 2), (dict(num_heads=96), 2), (dict(num_heads=256), 2), (dict(q=0), 1), (dict(q=0x10008), 3),
    (dict(kv=0x30004), 3), (dict(page_stride_bytes=8440), 1), (dict(page_stride_bytes=8456), 3),
    (dict(num_q=-1), 1), (dict(reserved0=1), 1), (dict(record_format=2), 1), (dict(q_len=0), 1), (dict(num_req=2), 1),
    (dict(resident=0x60000), 1), (dict(num_pages=0), 1), (dict(page_table=0x40002), 3),
])
def test_score_rejects_bad_args(lib, change, want):
    a = _fake_args(**change)
    st = lib.csa_index_score(ctypes.byref(a), ctypes.c_void_p(0x70000), 256, None)
    assert st == want, (change, st)


def test_topk_rejects_bad_args(lib):
    a = _fake_args()
    ws = native.workspace_bytes(a, 512)
    f = lib.csa_index_score_topk_fused
    assert f(ctypes.byref(a), 0, 0x1000, 0x2000, 0x3000, ws, None) == 1            # k = 0
    assert f(ctypes.byref(a), 2048, 0x1000, 0x2000, 0x3000, ws, None) == 1         # k too large
    assert f(ctypes.byref(a), 512, 0x1000, 0x2000, 0x3000, ws - 1, None) == 4      # workspace too small
    assert f(ctypes.byref(a), 512, 0x1000, 0x2000, None, ws, None) == 4            # no workspace
    assert f(ctypes.byref(a), 512, 0x1000, 0x2000, 0x3008, ws, None) == 3          # misaligned workspace
    assert f(ctypes.byref(a), 512, 0x1002, 0x2000, 0x3000, ws, None) == 3          # misaligned idx
    t = lib.csa_index_topk
    assert t(0x5000, 128, ctypes.byref(a), 512, 0x1000, 0x2000, 0x3000, ws, None) == 1  # stride < 64*pt_stride
    assert t(None, 256, ctypes.byref(a), 512, 0x1000, 0x2000, 0x3000, ws, None) == 1
    assert lib.csa_index_score(None, 0x1000, 256, None) == 1


def test_merge_topk_validates_on_the_host(lib):
    f = lib.csa_index_merge_topk
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    ok = (0x1000, 0x2000)
    assert f(*ok, 0, 4, 512, 512, 0x3000, 0x4000, None) == 1      # no lists
    assert f(*ok, 2, -1, 512, 512, 0x3000, 0x4000, None) == 1     # negative rows
    assert f(*ok, 2, 4, 0, 512, 0x3000, 0x4000, None) == 1        # k_in = 0
    assert f(*ok, 2, 4, 1025, 512, 0x3000, 0x4000, None) == 1     # k_in > CSA_MAX_K
    assert f(*ok, 2, 4, 512, 1025, 0x3000, 0x4000, None) == 1     # k > CSA_MAX_K
    assert f(None, 0x2000, 2, 4, 512, 512, 0x3000, 0x4000, None) == 1
    assert f(*ok, 2, 4, 512, 512, 0x3002, 0x4000, None) == 3      # misaligned output
    assert f(*ok, 2, 0, 512, 512, None, None, None) == 0          # no rows: nothing to do


def test_static_scratch_variant_validates_on_the_host(lib):
    f = lib.csa_index_score_topk_fused_static
    f.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    a = _fake_args()
    assert f(None, 512, 0x1000, 0x2000, None) == 1
    assert f(ctypes.addressof(a), 0, 0x1000, 0x2000, None) == 1
    assert f(ctypes.addressof(a), 512, 0x1002, 0x2000, None) == 3
    assert f(ctypes.addressof(_fake_args(head_dim=64)), 512, 0x1000, 0x2000, None) == 2


def test_128_heads_only_in_score_and_logit_modes(lib):
    """The scorer takes 64 or 128 heads; the top-k entry points only 64."""
    a = _fake_args(num_heads=128, num_q=0)
    assert lib.csa_index_score(ctypes.byref(a), None, 0, None) == 0
    assert lib.csa_index_logits(ctypes.byref(a), None, 0, None) == 0
    a = _fake_args(num_heads=128)
    ws = native.workspace_bytes(a, 512)
    assert lib.csa_index_score_topk_fused(ctypes.byref(a), 512, 0x1000, 0x2000, 0x3000, ws, None) == 2
    assert lib.csa_index_logits(ctypes.byref(a), 0x70002, 256, None) == 3  # validated like 64 heads


def test_empty_batch_is_a_no_op(lib):
    a = _fake_args(num_q=0)
    assert lib.csa_index_score(ctypes.byref(a), None, 0, None) == 0
    assert lib.csa_index_score_topk_fused(ctypes.byref(a), 512, None, None, None, 0, None) == 0


def test_write_args_layout_matches_header(tmp_path):
    fields = [f[0] for f in native.WriteArgs._fields_]
    src = tmp_path / "wlayout.c"
    body = "".join(f'printf("{f} %zu\\n", offsetof(csa_write_args, {f}));' for f in fields)
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "csa_index.h"\n'
                   'int main(void){' + body + 'printf("sizeof %zu\\n", sizeof(csa_write_args));return 0;}\n')
    exe = tmp_path / "wlayout"
    subprocess.run(["gcc", "-std=c11", f"-I{build.INCLUDE}", "-o", str(exe), str(src)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                        check=True).stdout.splitlines())
    for f in fields:
        assert int(got[f]) == getattr(native.WriteArgs, f).offset, f
    assert int(got["sizeof"]) == ctypes.sizeof(native.WriteArgs)


def _fake_write_args(**kw):
    """Host-side writer args with aligned fake device addresses: validation only."""
    a = native.WriteArgs(0x10000, native.KEYS_F32, 0, 4, 0, 0x20000, 0x30000, 8, native.PAGE_BYTES, 0x40000, 2, 4, 0)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("change,want", [
    (dict(keys=0), 1), (dict(row_pos=0), 1), (dict(kv=0), 1), (dict(page_table=0), 1),
    (dict(n=-1), 1), (dict(key_dtype=7), 1), (dict(reserved0=1), 1), (dict(num_req=0), 1),
    (dict(pt_stride=0), 1), (dict(num_pages=0), 1), (dict(page_stride_bytes=native.PAGE_BYTES - 16), 1),
    (dict(page_stride_bytes=native.PAGE_BYTES + 4), 1),
    (dict(keys=0x10004), 3), (dict(kv=0x30008), 3), (dict(row_pos=0x20002), 3), (dict(row_req=0x50001), 3),
])
def test_write_keys_rejects_bad_args(lib, change, want):
    st = lib.csa_index_write_keys(ctypes.byref(_fake_write_args(**change)), None)
    assert st == want, native.status_str(st)


def test_write_keys_empty_is_a_no_op(lib):
    assert lib.csa_index_write_keys(ctypes.byref(_fake_write_args(n=0)), None) == 0
    assert lib.csa_index_write_keys(None, None) == 1


def test_recall_args_layout_matches_header(tmp_path):
    fields = [f[0] for f in native.RecallArgs._fields_]
    src = tmp_path / "rlayout.c"
    body = "".join(f'printf("{f} %zu\\n", offsetof(csa_recall_args, {f}));' for f in fields)
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "csa_index.h"\n'
                   'int main(void){' + body + 'printf("sizeof %zu\\n", sizeof(csa_recall_args));return 0;}\n')
    exe = tmp_path / "rlayout"
    subprocess.run(["gcc", "-std=c11", f"-I{build.INCLUDE}", "-o", str(exe), str(src)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                        check=True).stdout.splitlines())
    for f in fields:
        assert int(got[f]) == getattr(native.RecallArgs, f).offset, f
    assert int(got["sizeof"]) == ctypes.sizeof(native.RecallArgs)


def test_recall_rejects_bad_args(lib):
    layer = _fake_args(num_heads=128)
    arr = (native.Args * 2)(layer, layer)
    base = dict(layers=ctypes.addressof(arr), n_layers=2, ensemble=0, threshold=0.5, sink=0, recent=0,
                pages_stride=4, keep=0x60000, keep_stride=256, pages=0x70000, n_pages=0x80000, scores=0)

    def call(**kw):
        d = dict(base)
        d.update(kw)
        return lib.csa_recall_level1(ctypes.byref(native.RecallArgs(**d)), ctypes.c_void_p(0x90000), 1 << 30, None)

    assert call(n_layers=0) == 1 and call(n_layers=9) == 1 and call(ensemble=2) == 1
    assert call(threshold=float("nan")) == 1 and call(sink=-1) == 1 and call(recent=-2) == 1
    assert call(keep_stride=255) == 1 and call(pages_stride=3) == 1 and call(keep=0) == 1
    assert call(pages=0x70002) == 3
    arr[1].num_heads = 64  # layers must all have 128 heads
    assert call() == 1
    arr[1].num_heads = 128
    arr[1].pt_stride = 5   # and agree on the rows' geometry
    assert call() == 1
    arr[1].pt_stride = 4
    assert call(layers=0) == 1
    arr[0].pt_stride = arr[1].pt_stride = 65535 * 64 + 1  # more page windows than a grid dimension holds
    assert call(pages_stride=65535 * 64 + 1, keep_stride=64 * (65535 * 64 + 1)) == 2
    arr[0].pt_stride = arr[1].pt_stride = 4
    need = lib.csa_recall_workspace_bytes(ctypes.byref(native.RecallArgs(**base)))
    assert need > 0
    assert lib.csa_recall_level1(ctypes.byref(native.RecallArgs(**base)), ctypes.c_void_p(0x90000), need - 1,
                                 None) == 4


def test_recall_workspace_bytes_arithmetic(lib):
    """The combined-score plane (num_q x keep_stride fp32) and one flag per row and
    logical page, each rounded up to 256 bytes; 0 for nonsense sizes."""
    def ws(num_q, stride, pts):
        layer = _fake_args(num_q=num_q, pt_stride=pts, num_heads=128)
        arr = (native.Args * 1)(layer)
        ra = native.RecallArgs(layers=ctypes.addressof(arr), n_layers=1, keep_stride=stride, pages_stride=pts)
        return lib.csa_recall_workspace_bytes(ctypes.byref(ra))

    r256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for num_q, stride, pts in ((1, 64, 1), (3, 5056, 79), (64, 131072, 2048), (4096, 1 << 14, 256)):
        assert ws(num_q, stride, pts) == r256(num_q * stride * 4) + r256(num_q * pts)
    assert ws(-1, 64, 1) == 0 and ws(2, -5, 1) == 0
    assert lib.csa_recall_workspace_bytes(None) == 0
