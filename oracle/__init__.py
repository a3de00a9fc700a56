"""CPU oracle for mha_prefill -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path (``gqa_attention_prefill_gb300`` and its CUDA library) never imports it,
and the two share no code.

The arithmetic lives in ``mha_oracle.c`` (plain C, fp64 accumulation), whose
header states the formula and the readings of the pages it follows.  This
module only compiles and marshals.

Parity pins (all in ``tests/test_oracle_pins.py``): library softmax attention
(``torch.nn.functional.scaled_dot_product_attention`` in float64 on CPU, with
the sink as an extra zero-value key and the causal/window mask as an additive
mask), closed forms (first token, W=1, identical keys, sink -> +inf), the
hand-derived fixture under ``tests/golden/``, and invariants (packing order,
GQA == MHA with repeated K/V, W >= L == full causal).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mha_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build_lib(force: bool = False, extra_flags=(), out_path: str | None = None) -> str:
    """Compile mha_oracle.c with gcc (portable C99, -O2, no -ffast-math)."""
    out = out_path or _LIB
    if force or out_path or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", *extra_flags, "-o",
                               tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, out)
    return out


def _bind(lib):
    P = ctypes.c_void_p
    lib.oracle_mha_prefill.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_double, P, P,
                                       ctypes.c_int]
    lib.oracle_mha_prefill.restype = ctypes.c_int
    lib.oracle_mha_prefill_rows.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, P, P, ctypes.c_int64, P, P,
                                            ctypes.c_int]
    lib.oracle_mha_prefill_rows.restype = ctypes.c_int
    lib.oracle_mha_prefill_kvcache.argtypes = [P, P, P, P, P, P, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_double, P, P, ctypes.c_int]
    lib.oracle_mha_prefill_kvcache.restype = ctypes.c_int
    lib.oracle_mha_prefill_kvcache_rows.argtypes = [P, P, P, P, P, P, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_double, P, P,
                                                    ctypes.c_int64, P, P, ctypes.c_int]
    lib.oracle_mha_prefill_kvcache_rows.restype = ctypes.c_int
    return lib


def _load():
    """The oracle library: $ORACLE_LIB_PATH if set (another build of the same
    source, e.g. with sanitizers), else the in-tree build."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(os.environ.get("ORACLE_LIB_PATH") or build_lib()))
    return _lib


def load_variant(path: str):
    """Load another build of the same source (used by tests that plant a mistake)."""
    return _bind(ctypes.CDLL(path))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _prep(q, k, v, sinks, cu):
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    s = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float64)
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    return q, k, v, s, cu


def mha_prefill(q, k, v, sinks, cu_seqlens, Hq, Hkv, D, window, scale, nthreads=0, lib=None):
    """Every row.  q/k/v are bf16 bit patterns (uint16) shaped [T,H,D].
    Returns (out [T,Hq,D] float64, lse [T,Hq] float64, threads used)."""
    lib = lib or _load()
    q, k, v, s, cu = _prep(q, k, v, sinks, cu_seqlens)
    T = int(cu[-1])
    out = np.zeros((T, Hq, D), dtype=np.float64)
    lse = np.zeros((T, Hq), dtype=np.float64)
    n = lib.oracle_mha_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(s), _ptr(cu), len(cu) - 1, Hq,
                               Hkv, D, window, float(scale), _ptr(out), _ptr(lse), nthreads)
    if n < 0:
        raise ValueError(f"oracle rejected the problem (rc={n})")
    return out, lse, n


def mha_prefill_rows(q, k, v, sinks, cu_seqlens, Hq, Hkv, D, window, scale, row_t, row_h,
                     nthreads=0, lib=None):
    """Selected rows (token row_t[i], head row_h[i]).  Returns (out [n,D], lse [n], threads)."""
    lib = lib or _load()
    q, k, v, s, cu = _prep(q, k, v, sinks, cu_seqlens)
    row_t = np.ascontiguousarray(row_t, dtype=np.int64)
    row_h = np.ascontiguousarray(row_h, dtype=np.int32)
    out = np.zeros((len(row_t), D), dtype=np.float64)
    lse = np.zeros(len(row_t), dtype=np.float64)
    n = lib.oracle_mha_prefill_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(s), _ptr(cu), len(cu) - 1,
                                    Hq, Hkv, D, window, float(scale), _ptr(row_t), _ptr(row_h),
                                    len(row_t), _ptr(out), _ptr(lse), nthreads)
    if n < 0:
        raise ValueError(f"oracle rejected the problem (rc={n})")
    return out, lse, n


def mha_prefill_kvcache(q, k, v, sinks, cu_q, cu_k, Hq, Hkv, D, window, scale, rows=None,
                        nthreads=0, lib=None):
    """Prefill over a key/value cache (query i of a sequence at key position
    Lk - Lq + i).  Returns (out, lse, threads) for every row, or for the rows
    (t, h) given."""
    lib = lib or _load()
    q, k, v, s, cu_q = _prep(q, k, v, sinks, cu_q)
    cu_k = np.ascontiguousarray(cu_k, dtype=np.int32)
    if rows is None:
        Tq = int(cu_q[-1])
        out = np.zeros((Tq, Hq, D), dtype=np.float64)
        lse = np.zeros((Tq, Hq), dtype=np.float64)
        n = lib.oracle_mha_prefill_kvcache(_ptr(q), _ptr(k), _ptr(v), _ptr(s), _ptr(cu_q),
                                           _ptr(cu_k), len(cu_q) - 1, Hq, Hkv, D, window,
                                           float(scale), _ptr(out), _ptr(lse), nthreads)
    else:
        row_t = np.ascontiguousarray(rows[0], dtype=np.int64)
        row_h = np.ascontiguousarray(rows[1], dtype=np.int32)
        out = np.zeros((len(row_t), D), dtype=np.float64)
        lse = np.zeros(len(row_t), dtype=np.float64)
        n = lib.oracle_mha_prefill_kvcache_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(s), _ptr(cu_q),
                                                _ptr(cu_k), len(cu_q) - 1, Hq, Hkv, D, window,
                                                float(scale), _ptr(row_t), _ptr(row_h),
                                                len(row_t), _ptr(out), _ptr(lse), nthreads)
    if n < 0:
        raise ValueError(f"oracle rejected the problem (rc={n})")
    return out, lse, n


def run_workload(w, rows=None, nthreads=0):
    """Convenience over an inputgen.Workload (full, or sampled rows (t, h))."""
    sinks = None if w.sinks is None else w.sinks.astype(np.float64)
    if getattr(w, "cu_seqlens_k", None) is not None:
        return mha_prefill_kvcache(w.q, w.k, w.v, sinks, w.cu_seqlens, w.cu_seqlens_k, w.Hq,
                                   w.Hkv, w.D, w.window, w.scale, rows=rows, nthreads=nthreads)
    if rows is None:
        return mha_prefill(w.q, w.k, w.v, sinks, w.cu_seqlens, w.Hq, w.Hkv, w.D, w.window,
                           w.scale, nthreads)
    return mha_prefill_rows(w.q, w.k, w.v, sinks, w.cu_seqlens, w.Hq, w.Hkv, w.D, w.window,
                            w.scale, rows[0], rows[1], nthreads)
