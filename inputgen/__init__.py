"""Seeded synthetic inputs for the attention-prefill workloads.

This module is shared by the CUDA path's tests/benchmark and by the CPU
oracle's tests.  It contains no attention arithmetic: only random number
generation (``gen.c``), the workload shapes, conversions between bf16 bit
patterns and wider floats, and the choice of sampled rows.

Workload shapes follow the GPT-OSS attention layer the TokenSpeed-kernel
pages benchmark (page "TokenSpeed-kernel: multi-silicon ...", section
"Числа: Gluon на AMD MI355X": BF16 Q/K/V, head_dim 64, 64 query heads, 8 KV
heads, full causal, sequence lengths 1K-8K, batch 1-16; sliding-window and
attention-sink layers are named in the same section and in the ai-radar.it
article, section "AMD MI355X: la prova sul campo").
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libinputgen.so")
_lock = threading.Lock()
_lib = None

# Stream ids: every tensor of a workload draws from its own counter stream.
STREAM_Q, STREAM_K, STREAM_V, STREAM_SINKS, STREAM_LENS, STREAM_ROWS = 1, 2, 3, 4, 5, 6


def build_lib(force: bool = False, extra_flags=(), out_path: str | None = None) -> str:
    """Compile gen.c into libinputgen.so next to it (plain gcc, portable C), or
    into `out_path` with extra compiler flags."""
    out = out_path or _LIB
    if force or out_path or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", *extra_flags, "-o",
                               tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, out)
    return out


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(os.environ.get("INPUTGEN_LIB_PATH") or build_lib())
            lib.ig_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float,
                                           ctypes.c_void_p, ctypes.c_int64, ctypes.c_int]
            lib.ig_normal_bf16.restype = None
            lib.ig_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float,
                                          ctypes.c_void_p, ctypes.c_int64, ctypes.c_int]
            lib.ig_normal_f32.restype = None
            lib.ig_uniform_int.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64]
            lib.ig_uniform_int.restype = ctypes.c_int
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16(seed: int, stream: int, shape, mult: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of fp32(N(0,1)) * mult, rounded to nearest even."""
    out = np.empty(shape, dtype=np.uint16)
    _load().ig_normal_bf16(seed, stream, mult, out.ctypes.data, out.size, _threads())
    return out


def normal_f32(seed: int, stream: int, shape, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load().ig_normal_f32(seed, stream, sigma, out.ctypes.data, out.size, _threads())
    return out


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    rc = _load().ig_uniform_int(seed, stream, lo, hi, out.ctypes.data, n)
    if rc != 0:
        raise ValueError("hi < lo")
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest even) and return the bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(x)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


@dataclasses.dataclass
class Workload:
    name: str
    seqlens: list            # per-sequence lengths
    Hq: int
    Hkv: int
    D: int
    window: int              # <= 0: full causal
    scale: float
    q: np.ndarray            # uint16 bf16 bits [T, Hq, D]
    k: np.ndarray            # uint16 bf16 bits [T, Hkv, D]
    v: np.ndarray            # uint16 bf16 bits [T, Hkv, D]
    sinks: np.ndarray | None  # float32 [Hq] or None
    cu_seqlens: np.ndarray   # int32 [S+1]
    seed: int
    # prefill over a key/value cache: keys/values per sequence (Lk >= Lq), the
    # new tokens' keys last; None for plain prefill (keys == queries)
    cu_seqlens_k: np.ndarray | None = None
    seqlens_k: list | None = None
    # FP8 inputs (E4M3 codes, per-tensor power-of-two scales): q/k/v above are
    # then the exact bf16 values code * scale; None for bf16 inputs
    fp8: dict | None = None

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def num_seqs(self) -> int:
        return len(self.seqlens)

    @property
    def total_keys(self) -> int:
        return int(self.cu_seqlens_k[-1]) if self.cu_seqlens_k is not None else self.total_tokens

    def allowed_keys(self) -> int:
        """Sum over query rows of the number of allowed keys, for one head."""
        tot = 0
        lks = self.seqlens_k if self.seqlens_k is not None else self.seqlens
        for L, Lk in zip(self.seqlens, lks):
            pos = np.arange(L, dtype=np.int64) + (Lk - L)   # key position of each query
            if self.window > 0:
                tot += int(np.minimum(pos + 1, self.window).sum())
            else:
                tot += int((pos + 1).sum())
        return tot

    def unmasked_flops(self) -> float:
        """4*D*Hq*sum|J|: the QK^T and PV multiply-adds of allowed pairs only."""
        return 4.0 * self.D * self.Hq * self.allowed_keys()

    def algorithmic_bytes(self) -> int:
        """Read Q, K, V once (2 bytes per element, 1 for FP8 inputs); write out
        (bf16) and lse (fp32) once."""
        T, Tk = self.total_tokens, self.total_keys
        b = 1 if self.fp8 is not None else 2
        return (T * (self.Hq * self.D * (b + 2) + 4 * self.Hq) +
                Tk * 2 * self.Hkv * self.D * b)


# --------------------------------------------------------------------- FP8
# OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; largest
# finite 448, no infinities, all-ones = NaN; subnormals down to 2^-9.
E4M3_MAX = 448.0


def f32_to_e4m3(x: np.ndarray) -> np.ndarray:
    """uint8 E4M3 codes of float32 `x`, round to nearest even, saturating to
    +-448 (NaN -> 0x7F)."""
    x = np.asarray(x, dtype=np.float64)
    sign = (np.signbit(x)).astype(np.uint8) << 7
    a = np.minimum(np.abs(np.nan_to_num(x, nan=0.0)), E4M3_MAX)
    # exponent of the binade, clamped to the normal range [-6, 8]; below 2^-6
    # the spacing stays 2^-9 (subnormals)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)
    quantum = np.exp2(e - 3)
    m = np.round(a / quantum)            # numpy rounds halves to even
    q = m * quantum                      # the representable value
    q = np.minimum(q, E4M3_MAX)
    # re-derive the fields from q (a carry may have moved it to the next binade)
    eq = np.floor(np.log2(np.where(q > 0, q, 1.0)))
    normal = q >= 2.0 ** -6
    exp_field = np.where(normal, eq + 7, 0).astype(np.int64)
    man_field = np.where(normal, q / np.exp2(eq) * 8 - 8, q / 2.0 ** -9).astype(np.int64)
    code = (exp_field << 3 | man_field).astype(np.uint8) | sign
    code[np.isnan(x)] = 0x7F
    return code


def e4m3_to_f32(code: np.ndarray) -> np.ndarray:
    """float32 values of uint8 E4M3 codes."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 7
    v = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    v = np.where((c & 0x7F) == 0x7F, np.nan, v)
    return (s * v).astype(np.float32)


def quantize_e4m3(x: np.ndarray):
    """(codes, scale): a power-of-two scale with max|x| / scale <= 448 and the
    E4M3 codes of x / scale."""
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    scale = 2.0 ** np.ceil(np.log2(amax / E4M3_MAX)) if amax > 0 else 1.0
    return f32_to_e4m3(x.astype(np.float64) / scale), float(scale)


def make_fp8(seqlens, Hq, Hkv, D=64, window=0, scale=0.125, seed=0, sink_sigma=1.0,
             k_mult=1.0, with_sinks=True, name="fp8") -> Workload:
    """As `make`, with Q, K, V drawn in fp32 and quantized to E4M3 with
    per-tensor power-of-two scales; w.q/k/v hold the exact dequantized values
    (as bf16, which represents every E4M3 value times a power of two)."""
    seqlens = [int(x) for x in seqlens]
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    if seqlens:
        cu[1:] = np.cumsum(np.asarray(seqlens, dtype=np.int64)).astype(np.int32)
    T = int(cu[-1])
    qf = normal_f32(seed, STREAM_Q, (T, Hq, D))
    kf = normal_f32(seed, STREAM_K, (T, Hkv, D), k_mult)
    vf = normal_f32(seed, STREAM_V, (T, Hkv, D))
    (q8, sq), (k8, sk), (v8, sv) = quantize_e4m3(qf), quantize_e4m3(kf), quantize_e4m3(vf)
    deq = lambda c, sc: f32_to_bf16_bits(e4m3_to_f32(c) * np.float32(sc))
    sinks = normal_f32(seed, STREAM_SINKS, (Hq,), sink_sigma) if with_sinks else None
    return Workload(name, seqlens, Hq, Hkv, D, window, scale, deq(q8, sq), deq(k8, sk),
                    deq(v8, sv), sinks, cu, seed,
                    fp8=dict(q=q8, k=k8, v=v8, q_scale=sq, k_scale=sk, v_scale=sv))


def make(seqlens, Hq, Hkv, D=64, window=0, scale=0.125, seed=0, sink_sigma=1.0,
         k_mult=1.0, with_sinks=True, name="custom") -> Workload:
    seqlens = [int(x) for x in seqlens]
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    if seqlens:
        cu[1:] = np.cumsum(np.asarray(seqlens, dtype=np.int64)).astype(np.int32)
    T = int(cu[-1])
    q = normal_bf16(seed, STREAM_Q, (T, Hq, D))
    k = normal_bf16(seed, STREAM_K, (T, Hkv, D), k_mult)
    v = normal_bf16(seed, STREAM_V, (T, Hkv, D))
    sinks = normal_f32(seed, STREAM_SINKS, (Hq,), sink_sigma) if with_sinks else None
    return Workload(name, seqlens, Hq, Hkv, D, window, scale, q, k, v, sinks, cu, seed)


def make_kvcache(q_lens, k_lens, Hq, Hkv, D=64, window=0, scale=0.125, seed=0, sink_sigma=1.0,
                 with_sinks=True, name="kvcache") -> Workload:
    """Prefill over a cache: sequence s has q_lens[s] new tokens and k_lens[s]
    >= q_lens[s] keys/values (cached prefix, then the new tokens' own)."""
    q_lens = [int(x) for x in q_lens]
    k_lens = [int(x) for x in k_lens]
    assert len(q_lens) == len(k_lens) and all(k >= q for q, k in zip(q_lens, k_lens))
    cu = np.zeros(len(q_lens) + 1, dtype=np.int32)
    cu_k = np.zeros(len(k_lens) + 1, dtype=np.int32)
    if q_lens:
        cu[1:] = np.cumsum(np.asarray(q_lens, dtype=np.int64)).astype(np.int32)
        cu_k[1:] = np.cumsum(np.asarray(k_lens, dtype=np.int64)).astype(np.int32)
    T, Tk = int(cu[-1]), int(cu_k[-1])
    q = normal_bf16(seed, STREAM_Q, (T, Hq, D))
    k = normal_bf16(seed, STREAM_K, (Tk, Hkv, D))
    v = normal_bf16(seed, STREAM_V, (Tk, Hkv, D))
    sinks = normal_f32(seed, STREAM_SINKS, (Hq,), sink_sigma) if with_sinks else None
    return Workload(name, q_lens, Hq, Hkv, D, window, scale, q, k, v, sinks, cu, seed,
                    cu_seqlens_k=cu_k, seqlens_k=k_lens)


def make_kvcache_fp8(q_lens, k_lens, Hq, Hkv, D=64, window=0, scale=0.125, seed=0,
                     sink_sigma=1.0, with_sinks=True, name="kvcache_fp8") -> Workload:
    """`make_kvcache` with Q, K, V drawn in fp32 and quantized to E4M3 with
    per-tensor power-of-two scales (as `make_fp8`); w.q/k/v hold the exact
    dequantized values."""
    q_lens = [int(x) for x in q_lens]
    k_lens = [int(x) for x in k_lens]
    assert len(q_lens) == len(k_lens) and all(k >= q for q, k in zip(q_lens, k_lens))
    cu = np.zeros(len(q_lens) + 1, dtype=np.int32)
    cu_k = np.zeros(len(k_lens) + 1, dtype=np.int32)
    if q_lens:
        cu[1:] = np.cumsum(np.asarray(q_lens, dtype=np.int64)).astype(np.int32)
        cu_k[1:] = np.cumsum(np.asarray(k_lens, dtype=np.int64)).astype(np.int32)
    T, Tk = int(cu[-1]), int(cu_k[-1])
    qf = normal_f32(seed, STREAM_Q, (T, Hq, D))
    kf = normal_f32(seed, STREAM_K, (Tk, Hkv, D))
    vf = normal_f32(seed, STREAM_V, (Tk, Hkv, D))
    (q8, sq), (k8, sk), (v8, sv) = quantize_e4m3(qf), quantize_e4m3(kf), quantize_e4m3(vf)
    deq = lambda c, sc: f32_to_bf16_bits(e4m3_to_f32(c) * np.float32(sc))
    sinks = normal_f32(seed, STREAM_SINKS, (Hq,), sink_sigma) if with_sinks else None
    return Workload(name, q_lens, Hq, Hkv, D, window, scale, deq(q8, sq), deq(k8, sk),
                    deq(v8, sv), sinks, cu, seed, cu_seqlens_k=cu_k, seqlens_k=k_lens,
                    fp8=dict(q=q8, k=k8, v=v8, q_scale=sq, k_scale=sk, v_scale=sv))


# The five configurations, smallest first.
CONFIGS = {
    "tiny_1x256_h4kv1": dict(desc="1 seq x 256 tokens, Hq=4, Hkv=1, D=64, sinks N(0,1), "
                                  "scale 1/8, full causal"),
    "causal_4x4096_h64kv8": dict(desc="4 seqs x 4096 tokens, Hq=64, Hkv=8, D=64, sinks N(0,1), "
                                      "scale 1/8, full causal"),
    "window128_4x4096_h64kv8": dict(desc="as causal_4x4096 with sliding window W=128"),
    "ragged32_h64kv8": dict(desc="32 seqs, lengths U{512..8192} from the seed, Hq=64, Hkv=8, "
                                 "sinks N(0,2), full causal"),
    "ragged32_w128_h64kv8": dict(desc="ragged32 rerun with W=128"),
    "long_1x32768_h64kv8": dict(desc="1 seq x 32768 tokens, K = bf16(3*N(0,1)), sinks N(0,1), "
                                     "full causal"),
    # prefill over a key/value cache (not one of the five above)
    "kvcache_4x2048_on_4096_h64kv8": dict(desc="4 seqs x 2048 new tokens over a 4096-token cache "
                                               "(Lk = 6144), Hq=64, Hkv=8, D=64, causal"),
    # one decoding step per sequence over its cache (query at key position Lk - 1)
    "decode_64x8192_h64kv8": dict(desc="64 seqs, one query token each over 8192 keys, Hq=64, "
                                       "Hkv=8, D=64, sinks N(0,1), causal"),
    "decode_ragged32_h64kv8": dict(desc="32 seqs, one query token each over U{512..32768} keys, "
                                        "Hq=64, Hkv=8, D=64, sinks N(0,2), causal"),
    # FP8 (E4M3) Q/K/V with per-tensor scales, otherwise the bench workload
    "fp8_causal_4x4096_h64kv8": dict(desc="as causal_4x4096 with E4M3 Q/K/V (per-tensor "
                                          "power-of-two scales)"),
    "fp8_causal_4x4096_h32kv8_d128": dict(desc="as causal_4x4096_h32kv8_d128 with E4M3 Q/K/V "
                                               "(per-tensor power-of-two scales)"),
    # head dimension 128 (the same unmasked FLOPs as causal_4x4096_h64kv8)
    "causal_4x4096_h32kv8_d128": dict(desc="4 seqs x 4096 tokens, Hq=32, Hkv=8, D=128, "
                                           "sinks N(0,1), scale 1/sqrt(128), full causal"),
    "long_1x32768_h32kv8_d128": dict(desc="1 seq x 32768 tokens, Hq=32, Hkv=8, D=128, "
                                          "K = bf16(3*N(0,1)), scale 1/sqrt(128), full causal"),
    # other query-head group sizes G = Hq / Hkv (1: plain multi-head attention)
    "causal_4x4096_h32kv32_d128": dict(desc="as causal_4x4096_h32kv8_d128 with Hkv=32 (G=1)"),
    "causal_4x4096_h64kv8_d128": dict(desc="as causal_4x4096_h32kv8_d128 with Hq=64 (G=8)"),
    "causal_4x4096_h64kv64": dict(desc="as causal_4x4096_h64kv8 with Hkv=64 (G=1)"),
}


def ragged_lengths(seed: int, n: int = 32, lo: int = 512, hi: int = 8192):
    return [int(x) for x in uniform_int(seed, STREAM_LENS, n, lo, hi)]


def config(name: str, seed: int = 0) -> Workload:
    if name == "tiny_1x256_h4kv1":
        return make([256], 4, 1, seed=seed, name=name)
    if name == "causal_4x4096_h64kv8":
        return make([4096] * 4, 64, 8, seed=seed, name=name)
    if name == "window128_4x4096_h64kv8":
        return make([4096] * 4, 64, 8, window=128, seed=seed, name=name)
    if name == "ragged32_h64kv8":
        return make(ragged_lengths(seed), 64, 8, sink_sigma=2.0, seed=seed, name=name)
    if name == "ragged32_w128_h64kv8":
        return make(ragged_lengths(seed), 64, 8, window=128, sink_sigma=2.0, seed=seed, name=name)
    if name == "long_1x32768_h64kv8":
        return make([32768], 64, 8, k_mult=3.0, seed=seed, name=name)
    if name == "kvcache_4x2048_on_4096_h64kv8":
        return make_kvcache([2048] * 4, [6144] * 4, 64, 8, seed=seed, name=name)
    if name == "decode_64x8192_h64kv8":
        return make_kvcache([1] * 64, [8192] * 64, 64, 8, seed=seed, name=name)
    if name == "decode_ragged32_h64kv8":
        return make_kvcache([1] * 32, ragged_lengths(seed, 32, 512, 32768), 64, 8, sink_sigma=2.0,
                            seed=seed, name=name)
    if name == "fp8_causal_4x4096_h64kv8":
        return make_fp8([4096] * 4, 64, 8, seed=seed, name=name)
    if name == "fp8_causal_4x4096_h32kv8_d128":
        return make_fp8([4096] * 4, 32, 8, D=128, scale=128 ** -0.5, seed=seed, name=name)
    if name == "causal_4x4096_h32kv8_d128":
        return make([4096] * 4, 32, 8, D=128, scale=128 ** -0.5, seed=seed, name=name)
    if name == "long_1x32768_h32kv8_d128":
        return make([32768], 32, 8, D=128, scale=128 ** -0.5, k_mult=3.0, seed=seed, name=name)
    if name == "causal_4x4096_h32kv32_d128":
        return make([4096] * 4, 32, 32, D=128, scale=128 ** -0.5, seed=seed, name=name)
    if name == "causal_4x4096_h64kv8_d128":
        return make([4096] * 4, 64, 8, D=128, scale=128 ** -0.5, seed=seed, name=name)
    if name == "causal_4x4096_h64kv64":
        return make([4096] * 4, 64, 64, seed=seed, name=name)
    raise KeyError(name)


def sample_rows(w: Workload, n_target: int = 4096, seed_stream: int = STREAM_ROWS,
                tile: int = 128):
    """(token, head) rows covering every sequence and head, sequence ends,
    q-tile boundaries, window edges; the rest uniform.  Returns (t int64, h int32)."""
    rows = set()
    cu = w.cu_seqlens
    H = w.Hq
    for s, L in enumerate(w.seqlens):
        if L == 0:
            continue
        st = int(cu[s])
        special = {0, L - 1}
        for b in range(0, L, tile):
            for off in (0, tile - 1):
                if b + off < L:
                    special.add(b + off)
        if w.window > 0:
            for off in (w.window - 1, w.window):
                if off < L:
                    special.add(off)
        sp = sorted(special)
        for i, off in enumerate(sp):
            rows.add((st + off, (i * 7 + s) % H))
        for h in range(H):
            rows.add((st + sp[(h * 5 + s) % len(sp)], h))
    T = w.total_tokens
    need = max(0, n_target - len(rows))
    if T > 0 and need > 0:
        r = uniform_int(w.seed, seed_stream, 2 * need + 16, 0, T * H - 1)
        for x in r:
            rows.add((int(x) // H, int(x) % H))
            if len(rows) >= n_target:
                break
    rows = sorted(rows)
    t = np.array([r[0] for r in rows], dtype=np.int64)
    h = np.array([r[1] for r in rows], dtype=np.int32)
    return t, h
