"""The C-ABI library: loads, exports what include/tsk_mha.h declares, and
rejects bad arguments on the host before touching the GPU (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

import gqa_attention_prefill_gb300 as pkg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tsk_mha.h")


@pytest.fixture(scope="module")
def lib():
    from gqa_attention_prefill_gb300 import build
    build.build()
    return pkg.load_library()


def declared_functions():
    src = open(HEADER).read()
    return re.findall(r"^TSK_API\s+[\w\s\*]+?\b(tsk_\w+)\s*\(", src, flags=re.M)


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert "tsk_mha_prefill" in names and "tsk_get_device_status" in names
    assert len(names) == len(set(names)) >= 8


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", pkg.library_path()],
                         capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == set(declared_functions()), exported ^ set(declared_functions())


def test_no_oracle_in_product_library():
    out = subprocess.run(["nm", "-D", pkg.library_path()], capture_output=True, text=True).stdout
    assert "oracle" not in out
    src_dir = os.path.join(ROOT, "gqa_attention_prefill_gb300")
    for dirpath, _, files in os.walk(src_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "oracle/" not in text, f


def test_status_strings(lib):
    assert pkg.tsk_status_string(0) == "ok"
    for c in range(-8, 0):
        assert pkg.tsk_status_string(c) != "unknown status"
    assert pkg.tsk_version() >= 100
    assert pkg.tsk_kernels_per_call() == 2


FAKE = 0x10000  # 16-byte aligned fake device addresses: never dereferenced by these calls


def call(lib, **kw):
    a = dict(q=FAKE, k=FAKE * 3, v=FAKE * 5, sinks=None, cu=FAKE * 7, num_seqs=1,
             total_tokens=128, Hq=8, Hkv=2, D=64, window=0, scale=0.125, out=FAKE * 9, lse=None)
    a.update(kw)
    return lib.tsk_mha_prefill(a["q"], a["k"], a["v"], a["sinks"], a["cu"], a["num_seqs"],
                               a["total_tokens"], a["Hq"], a["Hkv"], a["D"], a["window"],
                               a["scale"], a["out"], a["lse"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(k=None), -1), (dict(v=None), -1), (dict(out=None), -1),
    (dict(cu=None), -1), (dict(num_seqs=-1), -1), (dict(total_tokens=-5), -1),
    (dict(Hq=0), -1), (dict(Hkv=0), -1), (dict(scale=0.0), -1), (dict(scale=-1.0), -1),
    (dict(scale=float("nan")), -1), (dict(scale=float("inf")), -1),
    (dict(D=96), -2), (dict(D=32), -2), (dict(Hq=6, Hkv=4), -2),
    (dict(total_tokens=1 << 26, Hq=64), -2), (dict(num_seqs=1 << 24), -2),
    (dict(q=FAKE + 8), -3), (dict(k=FAKE * 3 + 2), -3), (dict(v=FAKE * 5 + 4), -3),
    (dict(out=FAKE * 9 + 1), -3), (dict(cu=FAKE * 7 + 2), -3), (dict(sinks=FAKE + 1), -3),
    (dict(lse=FAKE * 11 + 2), -3),
    (dict(out=FAKE + 64), -1),            # out overlaps q
    (dict(out=FAKE * 3 + 16), -1),        # out overlaps k
])
def test_host_side_rejections(lib, kw, code):
    assert call(lib, **kw) == code


@pytest.mark.parametrize("kw", [dict(num_seqs=0), dict(total_tokens=0)])
def test_empty_problems_return_ok_without_launch(lib, kw):
    assert call(lib, **kw) == 0


def kv_call(lib, **kw):
    a = dict(q=FAKE, k=FAKE * 3, v=FAKE * 5, sinks=None, cu=FAKE * 7, cu_k=FAKE * 13, num_seqs=1,
             total_q=128, total_k=512, Hq=8, Hkv=2, D=64, window=0, scale=0.125, out=FAKE * 9,
             lse=None)
    a.update(kw)
    return lib.tsk_mha_prefill_kvcache(a["q"], a["k"], a["v"], a["sinks"], a["cu"], a["cu_k"],
                                       a["num_seqs"], a["total_q"], a["total_k"], a["Hq"],
                                       a["Hkv"], a["D"], a["window"], a["scale"], a["out"],
                                       a["lse"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(cu_k=None), -1), (dict(total_k=100), -1), (dict(total_k=-1), -1), (dict(D=256), -2),
    (dict(cu_k=FAKE * 13 + 2), -3), (dict(total_k=(1 << 30), Hkv=2), -2),
    (dict(out=FAKE * 3 + 16), -1),
])
def test_kvcache_host_side_rejections(lib, kw, code):
    assert kv_call(lib, **kw) == code


def test_kvcache_empty_returns_ok(lib):
    assert kv_call(lib, total_q=0, total_k=0) == 0


def dec_call(lib, **kw):
    a = dict(q=FAKE, k=FAKE * 3, v=FAKE * 5, sinks=None, cu_k=FAKE * 13, num_seqs=4, total_k=512,
             max_k=256, Hq=8, Hkv=2, D=64, window=0, scale=0.125, out=FAKE * 9, lse=None)
    a.update(kw)
    return lib.tsk_mha_decode_kvcache(a["q"], a["k"], a["v"], a["sinks"], a["cu_k"], a["num_seqs"],
                                      a["total_k"], a["max_k"], a["Hq"], a["Hkv"], a["D"],
                                      a["window"], a["scale"], a["out"], a["lse"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(cu_k=None), -1), (dict(q=None), -1), (dict(max_k=0), -1), (dict(max_k=1000), -1),
    (dict(total_k=2), -1), (dict(scale=0.0), -1), (dict(D=96), -2), (dict(Hq=6, Hkv=4), -2),
    (dict(num_seqs=70000, total_k=1 << 20, max_k=64), -2), (dict(q=FAKE + 8), -3),
    (dict(cu_k=FAKE * 13 + 2), -3), (dict(out=FAKE * 3 + 16), -1),
])
def test_decode_host_side_rejections(lib, kw, code):
    assert dec_call(lib, **kw) == code


def test_decode_empty_returns_ok(lib):
    assert dec_call(lib, num_seqs=0, total_k=0) == 0


def _host_call(lib, cu, num_seqs, total, D=64, Hq=8, Hkv=2, scale=0.125):
    """tsk_mha_prefill_host with host buffers (numpy) and stream 0."""
    import numpy as np
    T = max(int(total), 1)
    q = np.zeros((T, Hq, D), dtype=np.uint16)
    kv = np.zeros((T, Hkv, D), dtype=np.uint16)
    out = np.zeros((T, Hq, D), dtype=np.uint16)
    cu = np.asarray(cu, dtype=np.int32)
    return pkg.tsk_mha_prefill_host(q, kv, kv, None, cu, num_seqs, total, Hq, Hkv, D, 0, scale,
                                    out, None, 0)


@pytest.mark.parametrize("cu,n,total,code", [
    ([1, 5], 1, 5, -1),          # does not start at 0
    ([0, 5, 3], 2, 3, -1),       # decreasing
    ([0, 5], 1, 6, -1),          # last offset != total_tokens
    ([0, 5], -1, 5, -1),         # negative count
])
def test_host_buffer_entry_checks_offsets_on_the_host(lib, cu, n, total, code):
    assert _host_call(lib, cu, n, total) == code


def test_host_buffer_entry_rejects_unsupported_shapes(lib):
    assert _host_call(lib, [0, 5], 1, 5, D=96) == -2
    assert _host_call(lib, [0, 5], 1, 5, Hq=6, Hkv=4) == -2
    assert _host_call(lib, [0, 5], 1, 5, scale=float("nan")) == -1


def test_host_buffer_entry_empty_returns_ok(lib):
    assert _host_call(lib, [0], 0, 0) == 0
    assert _host_call(lib, [0, 0, 0], 2, 0) == 0


def test_host_buffer_entry_rejects_out_overlapping_inputs(lib):
    import numpy as np
    T, Hq, Hkv, D = 64, 8, 2, 64
    q = np.zeros((T, Hq, D), dtype=np.uint16)
    kv = np.zeros((T, Hkv, D), dtype=np.uint16)
    cu = np.asarray([0, T], dtype=np.int32)
    rc = pkg.tsk_mha_prefill_host(q, kv, kv, None, cu, 1, T, Hq, Hkv, D, 0, 0.125,
                                  q.ctypes.data + 128, None, 0)
    assert rc == -1


def test_bounds_checked_build_compiles_and_exports_the_same_symbols(tmp_path):
    from gqa_attention_prefill_gb300 import build
    path = build.build(out=str(tmp_path / "libtsk_mha_debug.so"), defines=["TSK_DEBUG"])
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True,
                         text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == set(declared_functions())
