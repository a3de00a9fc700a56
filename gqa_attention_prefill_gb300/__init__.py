"""GB300 (sm_103a) mha_prefill: causal grouped-query attention with attention
sinks and an optional sliding window over packed variable-length sequences.

This package is a thin ctypes binding over the C ABI in ``include/tsk_mha.h``
(library ``libtsk_mha.so``, built in-tree by ``build.py``).  It only marshals
arguments: every step of the computation runs in the library's CUDA kernels.
There is no fallback: if the library is missing or fails to load, every call
raises.

The operation is the ``mha_prefill`` call of the TokenSpeed-kernel public API
(README, section "Public API"), for the GPT-OSS attention layers described on
page "TokenSpeed-kernel: multi-silicon ...", section "Числа: Gluon на AMD
MI355X" (BF16, head_dim 64, 64 query / 8 KV heads, causal, sinks, sliding
window).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["tsk_mha_prefill", "tsk_mha_prefill_noalloc", "tsk_mha_prefill_kvcache",
           "tsk_mha_decode_kvcache", "tsk_mha_prefill_paged", "tsk_mha_decode_paged", "tsk_mha_prefill_fp8", "tsk_mha_prefill_fp8_kvcache", "mha_prefill", "mha_prefill_kvcache", "mha_decode_kvcache",
           "tsk_get_device_status", "tsk_noalloc_status", "tsk_status_string",
           "tsk_last_error", "tsk_debug_set_wait",
           "tsk_profile_enable", "tsk_profile_read", "tsk_release", "tsk_kernels_per_call",
           "tsk_bench_ex2_rate",
           "tsk_version", "TskError", "library_path", "load_library"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libtsk_mha.so")
_lock = threading.Lock()
_lib = None

STATUS = {0: "TSK_OK", -1: "TSK_ERR_INVALID_ARG", -2: "TSK_ERR_UNSUPPORTED",
          -3: "TSK_ERR_ALIGNMENT", -4: "TSK_ERR_DEVICE", -5: "TSK_ERR_OOM", -6: "TSK_ERR_LAUNCH",
          -7: "TSK_ERR_DEVICE_TIMEOUT", -8: "TSK_ERR_BAD_SEQLENS", -9: "TSK_ERR_BOUNDS"}


class TskError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        detail = tsk_last_error() if code in (-4, -5, -6) else ""
        super().__init__(f"{where}: {STATUS.get(code, code)} ({tsk_status_string(code)})"
                         + (f" [{detail}]" if detail else ""))


def tsk_last_error() -> str:
    try:
        return load_library().tsk_last_error().decode()
    except Exception:
        return ""


def library_path() -> str:
    """The library file to load: $TSK_LIB_PATH if set (another build of the
    same sources, e.g. with different compile-time options), else the in-tree
    libtsk_mha.so."""
    return os.environ.get("TSK_LIB_PATH") or _LIB_PATH


def load_library():
    """Loads libtsk_mha.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run __graft_entry__.build() "
                               "(or python -m gqa_attention_prefill_gb300.build)")
        lib = ctypes.CDLL(path)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.tsk_mha_prefill.argtypes = [P, P, P, P, P, i32, i64, i32, i32, i32, i32,
                                        ctypes.c_float, P, P, P]
        lib.tsk_mha_prefill.restype = ctypes.c_int
        lib.tsk_mha_prefill_noalloc.argtypes = lib.tsk_mha_prefill.argtypes
        lib.tsk_mha_prefill_noalloc.restype = ctypes.c_int
        lib.tsk_mha_prefill_host.argtypes = lib.tsk_mha_prefill.argtypes
        lib.tsk_mha_prefill_host.restype = ctypes.c_int
        lib.tsk_mha_prefill_kvcache.argtypes = [P, P, P, P, P, P, i32, i64, i64, i32, i32, i32,
                                                i32, ctypes.c_float, P, P, P]
        lib.tsk_mha_prefill_kvcache.restype = ctypes.c_int
        lib.tsk_mha_decode_kvcache.argtypes = [P, P, P, P, P, i32, i64, i32, i32, i32, i32, i32,
                                               ctypes.c_float, P, P, P]
        lib.tsk_mha_decode_kvcache.restype = ctypes.c_int
        lib.tsk_mha_prefill_paged.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i64, i64,
                                              i32, i32, i32, i32, ctypes.c_float, P, P, P]
        lib.tsk_mha_prefill_paged.restype = ctypes.c_int
        lib.tsk_mha_decode_paged.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i64, i32, i32,
                                             i32, i32, i32, ctypes.c_float, P, P, P]
        lib.tsk_mha_decode_paged.restype = ctypes.c_int
        f32 = ctypes.c_float
        lib.tsk_mha_prefill_fp8.argtypes = [P, P, P, f32, f32, f32, P, P, i32, i64, i32, i32, i32,
                                            i32, f32, P, P, P]
        lib.tsk_mha_prefill_fp8.restype = ctypes.c_int
        lib.tsk_mha_prefill_fp8_kvcache.argtypes = [P, P, P, f32, f32, f32, P, P, P, i32, i64,
                                                    i64, i32, i32, i32, i32, f32, P, P, P]
        lib.tsk_mha_prefill_fp8_kvcache.restype = ctypes.c_int
        lib.tsk_status_string.argtypes = [ctypes.c_int]
        lib.tsk_status_string.restype = ctypes.c_char_p
        lib.tsk_last_error.argtypes = []
        lib.tsk_last_error.restype = ctypes.c_char_p
        lib.tsk_get_device_status.argtypes = [P]
        lib.tsk_get_device_status.restype = ctypes.c_int
        lib.tsk_noalloc_status.argtypes = [P]
        lib.tsk_noalloc_status.restype = ctypes.c_int
        lib.tsk_profile_enable.argtypes = [ctypes.c_int]
        lib.tsk_profile_enable.restype = ctypes.c_int
        lib.tsk_profile_read.argtypes = [ctypes.POINTER(ctypes.c_float),
                                         ctypes.POINTER(ctypes.c_float)]
        lib.tsk_profile_read.restype = ctypes.c_int
        lib.tsk_bench_ex2_rate.argtypes = [ctypes.POINTER(ctypes.c_double), P]
        lib.tsk_bench_ex2_rate.restype = ctypes.c_int
        lib.tsk_kernels_per_call.argtypes = []
        lib.tsk_kernels_per_call.restype = i32
        lib.tsk_release.argtypes = []
        lib.tsk_release.restype = ctypes.c_int
        lib.tsk_debug_shrink_extent.argtypes = [i32]
        lib.tsk_debug_shrink_extent.restype = ctypes.c_int
        lib.tsk_debug_set_wait.argtypes = [ctypes.c_ulonglong, ctypes.c_int]
        lib.tsk_debug_set_wait.restype = ctypes.c_int
        lib.tsk_version.argtypes = []
        lib.tsk_version.restype = i32
        _lib = lib
        return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return x.ctypes.data  # numpy array (host memory)


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def tsk_status_string(code: int) -> str:
    try:
        return load_library().tsk_status_string(code).decode()
    except Exception:
        return STATUS.get(code, str(code))


def tsk_mha_prefill(q, k, v, sinks, cu_seqlens, num_seqs, total_tokens, Hq, Hkv, D, window,
                    scale, out, lse, stream=None) -> int:
    """Same arguments as the C function; tensors (or raw device addresses) for
    the buffers, ``stream`` a torch.cuda.Stream / handle / None (current
    stream).  Returns the status code (0 = TSK_OK)."""
    lib = load_library()
    return lib.tsk_mha_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(sinks), _ptr(cu_seqlens),
                               int(num_seqs), int(total_tokens), int(Hq), int(Hkv), int(D),
                               int(window), float(scale), _ptr(out), _ptr(lse),
                               _stream_handle(stream))


def tsk_mha_prefill_host(q, k, v, sinks, cu_seqlens, num_seqs, total_tokens, Hq, Hkv, D, window,
                         scale, out, lse, stream=None) -> int:
    """``tsk_mha_prefill`` with every buffer in host memory (CPU tensors,
    numpy arrays or raw host addresses; page-locked for overlapped copies).
    The library pipelines chunked copies in, attention and copies out; the
    call is asynchronous: read ``out``/``lse`` after ``stream`` (default: the
    current stream) has been synchronised.  Returns the status code."""
    lib = load_library()
    return lib.tsk_mha_prefill_host(_ptr(q), _ptr(k), _ptr(v), _ptr(sinks), _ptr(cu_seqlens),
                                    int(num_seqs), int(total_tokens), int(Hq), int(Hkv), int(D),
                                    int(window), float(scale), _ptr(out), _ptr(lse),
                                    _stream_handle(stream))


def tsk_mha_prefill_noalloc(q, k, v, sinks, cu_seqlens, num_seqs, total_tokens, Hq, Hkv, D,
                            window, scale, out, lse, stream=None) -> int:
    """Allocation-free variant (same arguments as ``tsk_mha_prefill``): its
    scratch is a fixed array inside the library, for callers that may not
    allocate device memory while running.  Calls that overlap on the GPU
    race on that shared array; problems beyond its limits return
    TSK_ERR_UNSUPPORTED."""
    lib = load_library()
    return lib.tsk_mha_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(sinks), _ptr(cu_seqlens),
                                       int(num_seqs), int(total_tokens), int(Hq), int(Hkv),
                                       int(D), int(window), float(scale), _ptr(out), _ptr(lse),
                                       _stream_handle(stream))


def tsk_mha_prefill_kvcache(q, k, v, sinks, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q,
                            total_k, Hq, Hkv, D, window, scale, out, lse, stream=None) -> int:
    """Prefill over a key/value cache (same arguments as the C function): new
    token i of a sequence with Lq new tokens and Lk keys sits at key position
    Lk - Lq + i.  Returns the status code."""
    lib = load_library()
    return lib.tsk_mha_prefill_kvcache(_ptr(q), _ptr(k), _ptr(v), _ptr(sinks),
                                       _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(num_seqs),
                                       int(total_q), int(total_k), int(Hq), int(Hkv), int(D),
                                       int(window), float(scale), _ptr(out), _ptr(lse),
                                       _stream_handle(stream))


def tsk_mha_decode_kvcache(q, k, v, sinks, cu_seqlens_k, num_seqs, total_k, max_seqlen_k, Hq,
                           Hkv, D, window, scale, out, lse, stream=None) -> int:
    """One decoding step over a key/value cache (same arguments as the C
    function): the query of sequence s sits at key position Lk - 1.  Returns
    the status code."""
    lib = load_library()
    return lib.tsk_mha_decode_kvcache(_ptr(q), _ptr(k), _ptr(v), _ptr(sinks), _ptr(cu_seqlens_k),
                                      int(num_seqs), int(total_k), int(max_seqlen_k), int(Hq),
                                      int(Hkv), int(D), int(window), float(scale), _ptr(out),
                                      _ptr(lse), _stream_handle(stream))


def tsk_mha_prefill_paged(q, k_pages, v_pages, sinks, cu_seqlens_q, cu_seqlens_k, block_table,
                          max_blocks_per_seq, page_size, num_pages, num_seqs, total_q, total_k,
                          Hq, Hkv, D, window, scale, out, lse, stream=None) -> int:
    """Prefill over a paged key/value cache (same arguments as the C
    function).  Returns the status code."""
    lib = load_library()
    return lib.tsk_mha_prefill_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(sinks),
                                     _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(block_table),
                                     int(max_blocks_per_seq), int(page_size), int(num_pages),
                                     int(num_seqs), int(total_q), int(total_k), int(Hq), int(Hkv),
                                     int(D), int(window), float(scale), _ptr(out), _ptr(lse),
                                     _stream_handle(stream))


def tsk_mha_decode_paged(q, k_pages, v_pages, sinks, cu_seqlens_k, block_table, max_blocks_per_seq,
                         page_size, num_pages, num_seqs, total_k, max_seqlen_k, Hq, Hkv, D, window,
                         scale, out, lse, stream=None) -> int:
    """One decoding step over a paged key/value cache (same arguments as the C
    function).  Returns the status code."""
    lib = load_library()
    return lib.tsk_mha_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(sinks),
                                    _ptr(cu_seqlens_k), _ptr(block_table), int(max_blocks_per_seq),
                                    int(page_size), int(num_pages), int(num_seqs), int(total_k),
                                    int(max_seqlen_k), int(Hq), int(Hkv), int(D), int(window),
                                    float(scale), _ptr(out), _ptr(lse), _stream_handle(stream))


def tsk_mha_prefill_fp8(q8, k8, v8, q_scale, k_scale, v_scale, sinks, cu_seqlens, num_seqs,
                        total_tokens, Hq, Hkv, D, window, scale, out, lse, stream=None) -> int:
    """Prefill with E4M3 inputs and per-tensor scales (same arguments as the C
    function; q8/k8/v8 are uint8 tensors or addresses).  Returns the status."""
    lib = load_library()
    return lib.tsk_mha_prefill_fp8(_ptr(q8), _ptr(k8), _ptr(v8), float(q_scale), float(k_scale),
                                   float(v_scale), _ptr(sinks), _ptr(cu_seqlens), int(num_seqs),
                                   int(total_tokens), int(Hq), int(Hkv), int(D), int(window),
                                   float(scale), _ptr(out), _ptr(lse), _stream_handle(stream))


def tsk_mha_prefill_fp8_kvcache(q8, k8, v8, q_scale, k_scale, v_scale, sinks, cu_seqlens_q,
                                cu_seqlens_k, num_seqs, total_q, total_k, Hq, Hkv, D, window,
                                scale, out, lse, stream=None) -> int:
    """E4M3 prefill over a contiguous key/value cache (same arguments as the C
    function).  Returns the status."""
    lib = load_library()
    return lib.tsk_mha_prefill_fp8_kvcache(
        _ptr(q8), _ptr(k8), _ptr(v8), float(q_scale), float(k_scale), float(v_scale),
        _ptr(sinks), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(num_seqs), int(total_q),
        int(total_k), int(Hq), int(Hkv), int(D), int(window), float(scale), _ptr(out), _ptr(lse),
        _stream_handle(stream))


def mha_decode_kvcache(q, k, v, cu_seqlens_k, max_seqlen_k: int, sinks=None, window: int = 0,
                       scale: float | None = None, out=None, lse=None, return_lse=True,
                       stream=None):
    """Tensor-level convenience over ``tsk_mha_decode_kvcache``: q [B, Hq, D],
    k/v [Tk, Hkv, D] bf16 CUDA (D = 64 or 128), cu_seqlens_k int32 CUDA [B+1].
    Returns (out, lse)."""
    import torch
    B, Hq, D = q.shape
    Tk, Hkv = k.shape[0], k.shape[1]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if v.shape != k.shape or k.shape[2] != D:
        raise ValueError("k and v must both be [Tk, Hkv, D]")
    if cu_seqlens_k.dtype != torch.int32 or not cu_seqlens_k.is_cuda or cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_k must be an int32 CUDA tensor of B + 1 offsets")
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    rc = tsk_mha_decode_kvcache(q, k, v, sinks, cu_seqlens_k, B, Tk, max_seqlen_k, Hq, Hkv, D,
                                window, scale, out, lse if return_lse else None, stream)
    if rc != 0:
        raise TskError(rc, "tsk_mha_decode_kvcache")
    return out, (lse if return_lse else None)


def mha_prefill_kvcache(q, k, v, cu_seqlens_q, cu_seqlens_k, sinks=None, window: int = 0,
                        scale: float | None = None, out=None, lse=None, return_lse=True,
                        stream=None):
    """Tensor-level convenience over ``tsk_mha_prefill_kvcache``: q [Tq, Hq, D],
    k/v [Tk, Hkv, D] bf16 CUDA (D = 64 or 128), int32 CUDA offsets.  Returns (out, lse)."""
    import torch
    Tq, Hq, D = q.shape
    Tk, Hkv = k.shape[0], k.shape[1]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if v.shape != k.shape or k.shape[2] != D:
        raise ValueError("k and v must both be [Tk, Hkv, D]")
    for name, c in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if c.dtype != torch.int32 or not c.is_cuda:
            raise ValueError(f"{name} must be an int32 CUDA tensor")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel():
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((Tq, Hq), dtype=torch.float32, device=q.device)
    rc = tsk_mha_prefill_kvcache(q, k, v, sinks, cu_seqlens_q, cu_seqlens_k,
                                 cu_seqlens_q.numel() - 1, Tq, Tk, Hq, Hkv, D, window, scale, out,
                                 lse if return_lse else None, stream)
    if rc != 0:
        raise TskError(rc, "tsk_mha_prefill_kvcache")
    return out, (lse if return_lse else None)


def mha_prefill(q, k, v, cu_seqlens, sinks=None, window: int = 0, scale: float | None = None,
                out=None, lse=None, return_lse: bool = True, stream=None):
    """Tensor-level convenience over ``tsk_mha_prefill``.

    q: [T, Hq, D] bf16 CUDA; k, v: [T, Hkv, D] bf16 CUDA (D = 64 or 128); cu_seqlens: int32
    CUDA [num_seqs+1]; sinks: fp32 CUDA [Hq] or None.  Returns (out, lse) with
    out [T, Hq, D] bf16 and lse [T, Hq] fp32 (None if return_lse is False).
    """
    import torch
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if k.shape != (T, Hkv, D) or v.shape != (T, Hkv, D):
        raise ValueError("k and v must be [T, Hkv, D] with q's T and D")
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
        raise ValueError("cu_seqlens must be an int32 CUDA tensor")
    if sinks is not None and (sinks.dtype != torch.float32 or not sinks.is_cuda
                              or sinks.numel() != Hq):
        raise ValueError("sinks must be a float32 CUDA tensor of Hq elements")
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    rc = tsk_mha_prefill(q, k, v, sinks, cu_seqlens, cu_seqlens.numel() - 1, T, Hq, Hkv, D,
                         window, scale, out, lse if return_lse else None, stream)
    if rc != 0:
        raise TskError(rc, "tsk_mha_prefill")
    return out, (lse if return_lse else None)


def tsk_get_device_status(stream=None) -> int:
    return load_library().tsk_get_device_status(_stream_handle(stream))


def tsk_noalloc_status(stream=None) -> int:
    """Device-side status of the most recent tsk_mha_prefill_noalloc call."""
    return load_library().tsk_noalloc_status(_stream_handle(stream))


def tsk_profile_enable(enable: bool = True) -> int:
    return load_library().tsk_profile_enable(1 if enable else 0)


def tsk_profile_read():
    """(prepass_ms, attention_ms) of the last call made while profiling was on."""
    a, b = ctypes.c_float(), ctypes.c_float()
    rc = load_library().tsk_profile_read(ctypes.byref(a), ctypes.byref(b))
    if rc != 0:
        raise TskError(rc, "tsk_profile_read")
    return a.value, b.value


def tsk_debug_set_wait(timeout_ns: int = 0, stall: bool = False) -> int:
    """Test hook: device wait limit for later calls (0 = 2 s) and stall injection."""
    return load_library().tsk_debug_set_wait(int(timeout_ns), 1 if stall else 0)


def tsk_bench_ex2_rate(stream=None) -> float:
    """Measured exponential (ex2.approx.f32) throughput of the device, per second."""
    r = ctypes.c_double()
    rc = load_library().tsk_bench_ex2_rate(ctypes.byref(r), _stream_handle(stream))
    if rc != 0:
        raise TskError(rc, "tsk_bench_ex2_rate")
    return r.value


def tsk_debug_shrink_extent(rows: int) -> int:
    """Test hook of -DTSK_DEBUG builds (TSK_ERR_UNSUPPORTED otherwise)."""
    return load_library().tsk_debug_shrink_extent(int(rows))


def tsk_kernels_per_call() -> int:
    return load_library().tsk_kernels_per_call()


def tsk_release() -> int:
    return load_library().tsk_release()


def tsk_version() -> int:
    return load_library().tsk_version()
