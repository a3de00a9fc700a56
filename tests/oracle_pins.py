"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin takes an oracle library handle (``lib``) so that the same pins can be
run against builds of the oracle with a planted mistake (see
``test_oracle_pins.py::test_planted_mistakes_are_caught``).  Every pin returns
``(ok, detail)`` instead of asserting.

Pins:
  * golden  -- the hand-derived fixture ``tests/golden/hand_sink_gqa.txt``;
  * sdpa    -- ``torch.nn.functional.scaled_dot_product_attention`` (float64,
               CPU) with the sink as an extra zero-value key whose logit is the
               sink, and the causal/window rule as an additive mask;
               ``torch.logsumexp`` of the same masked logits for the LSE;
  * first   -- the first token of a sequence sees one key: a two-term softmax;
  * w1      -- W = 1: every token sees only itself (two-term softmax);
  * same_k  -- all keys identical: out = mean(V_J) * (1 - sigma_sink);
  * big_sink-- sink -> +40: out -> 0, lse -> sink;
  * wide    -- W >= L gives exactly the full-causal result;
  * perm    -- permuting the packed sequences permutes the rows exactly;
  * gqa     -- GQA equals MHA with K/V repeated per group, exactly;
  * rows    -- the sampled-row entry point equals the full one at those rows.

Prefill over a key/value cache:
  * kv_equal   -- Lk == Lq is exactly plain prefill;
  * kv_chunked -- the last Lq tokens of a full prefill equal a prefill of
                  those tokens over the whole sequence's keys, exactly;
  * kv_sdpa    -- library softmax attention with the causal rule aligned to
                  the end of the keys (query i at key position Lk - Lq + i).
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import torch

import inputgen
import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "hand_sink_gqa.txt")


def _f64(bits):
    return inputgen.bf16_bits_to_f32(bits).astype(np.float64)


def _run(lib, w, window=None, sinks="w", rows=None, q=None, k=None, v=None, cu=None,
         Hkv=None, nthreads=2):
    window = w.window if window is None else window
    s = w.sinks if isinstance(sinks, str) else sinks
    s = None if s is None else np.asarray(s, dtype=np.float64)
    q = w.q if q is None else q
    k = w.k if k is None else k
    v = w.v if v is None else v
    cu = w.cu_seqlens if cu is None else cu
    Hkv = w.Hkv if Hkv is None else Hkv
    if rows is None:
        out, lse, _ = oracle.mha_prefill(q, k, v, s, cu, w.Hq, Hkv, w.D, window, w.scale,
                                         nthreads=nthreads, lib=lib)
    else:
        out, lse, _ = oracle.mha_prefill_rows(q, k, v, s, cu, w.Hq, Hkv, w.D, window, w.scale,
                                              rows[0], rows[1], nthreads=nthreads, lib=lib)
    return out, lse


def small_workload(seed=3, seqlens=(1, 5, 17, 40), Hq=4, Hkv=2, D=16, window=0, sinks=True,
                   scale=0.25):
    return inputgen.make(list(seqlens), Hq, Hkv, D=D, window=window, scale=scale, seed=seed,
                         with_sinks=sinks)


# --------------------------------------------------------------------------- golden
def load_golden():
    cfgs = {}
    cur = None
    hdr = {}
    with open(GOLDEN) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] in ("scale", "sinks", "cu_seqlens", "q", "k", "v"):
                hdr[tok[0]] = [x for x in tok[1:] if x != "|"]
            elif tok[0] == "config":
                cur = (tok[1], int(tok[3]))
                cfgs[cur] = []
            elif tok[0] == "row":
                t, h = int(tok[1]), int(tok[2])
                o = [Fraction(x) for x in tok[3:5]]
                z = Fraction(tok[5])
                cfgs[cur].append((t, h, o, z))
    return hdr, cfgs


def _num(s):
    if s.startswith("ln"):
        return math.log(float(s[2:]))
    return float(Fraction(s))


def pin_golden(lib):
    hdr, cfgs = load_golden()
    scale = _num(hdr["scale"][0])
    sinks = np.array([_num(x) for x in hdr["sinks"]], dtype=np.float64)
    cu = np.array([int(x) for x in hdr["cu_seqlens"]], dtype=np.int32)
    T = int(cu[-1])
    Hq, Hkv, D = len(sinks), 1, 2
    q = inputgen.f32_to_bf16_bits(np.array([float(x) for x in hdr["q"]], np.float32)).reshape(T, Hq, D)
    k = inputgen.f32_to_bf16_bits(np.array([float(x) for x in hdr["k"]], np.float32)).reshape(T, Hkv, D)
    v = inputgen.f32_to_bf16_bits(np.array([float(x) for x in hdr["v"]], np.float32)).reshape(T, Hkv, D)
    worst = 0.0
    for (name, W), rows in cfgs.items():
        out, lse, _ = oracle.mha_prefill(q, k, v, sinks, cu, Hq, Hkv, D, W, scale, nthreads=1,
                                         lib=lib)
        for t, h, o, z in rows:
            worst = max(worst, abs(out[t, h, 0] - float(o[0])), abs(out[t, h, 1] - float(o[1])),
                        abs(lse[t, h] - math.log(float(z))))
    return worst < 1e-12, f"max err {worst:.3g}"


# --------------------------------------------------------------------------- sdpa
def sdpa_reference(w, window=None, sinks="w"):
    """Library softmax attention in float64; returns (out [T,Hq,D], lse [T,Hq])."""
    window = w.window if window is None else window
    s = w.sinks if isinstance(sinks, str) else sinks
    G = w.Hq // w.Hkv
    T = w.total_tokens
    out = np.zeros((T, w.Hq, w.D))
    lse = np.zeros((T, w.Hq))
    qf, kf, vf = (torch.from_numpy(_f64(x)) for x in (w.q, w.k, w.v))
    for si, L in enumerate(w.seqlens):
        if L == 0:
            continue
        st = int(w.cu_seqlens[si])
        q = qf[st:st + L].permute(1, 0, 2)                                   # [Hq, L, D]
        k = kf[st:st + L].repeat_interleave(G, dim=1).permute(1, 0, 2)       # [Hq, L, D]
        v = vf[st:st + L].repeat_interleave(G, dim=1).permute(1, 0, 2)
        zero = torch.zeros(w.Hq, 1, w.D, dtype=torch.float64)
        kk = torch.cat([k, zero], dim=1)
        vv = torch.cat([v, zero], dim=1)
        ti = torch.arange(L)[:, None]
        ji = torch.arange(L)[None, :]
        allowed = ji <= ti
        if window > 0:
            allowed &= ji >= ti - window + 1
        m = torch.zeros(L, L, dtype=torch.float64).masked_fill(~allowed, float("-inf"))
        m = m.expand(w.Hq, L, L)
        if s is None:
            sink_col = torch.full((w.Hq, L, 1), float("-inf"), dtype=torch.float64)
        else:
            sink_col = torch.from_numpy(np.asarray(s, np.float64)).view(w.Hq, 1, 1).expand(w.Hq, L, 1)
        mask = torch.cat([m, sink_col], dim=2)
        o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=mask,
                                                             scale=w.scale)
        logits = w.scale * (q @ kk.transpose(1, 2)) + mask
        l = torch.logsumexp(logits, dim=-1)
        out[st:st + L] = o.permute(1, 0, 2).numpy()
        lse[st:st + L] = l.permute(1, 0).numpy()
    return out, lse


def pin_sdpa(lib):
    worst = 0.0
    for seed, window, sinks, Hq, Hkv in [(1, 0, True, 4, 2), (2, 0, False, 4, 4), (3, 3, True, 6, 2),
                                         (4, 1, True, 4, 1), (5, 7, False, 8, 2),
                                         (6, 100, True, 4, 2)]:
        w = small_workload(seed=seed, window=window, sinks=sinks, Hq=Hq, Hkv=Hkv)
        o, l = _run(lib, w)
        ro, rl = sdpa_reference(w)
        worst = max(worst, np.abs(o - ro).max(), np.abs(l - rl).max())
    return worst < 1e-10, f"max err {worst:.3g}"


# --------------------------------------------------------------------------- closed forms
def _score(w, t, h, j):
    G = w.Hq // w.Hkv
    return w.scale * float(np.dot(_f64(w.q[t, h]), _f64(w.k[j, h // G])))


def pin_first_token(lib):
    w = small_workload(seed=11, seqlens=(3, 1, 9), scale=0.3)
    o, l = _run(lib, w)
    G = w.Hq // w.Hkv
    worst = 0.0
    for si in range(w.num_seqs):
        t = int(w.cu_seqlens[si])
        for h in range(w.Hq):
            s = _score(w, t, h, t)
            sk = float(w.sinks[h])
            a = math.exp(s) / (math.exp(s) + math.exp(sk))
            worst = max(worst, np.abs(o[t, h] - a * _f64(w.v[t, h // G])).max(),
                        abs(l[t, h] - math.log(math.exp(s) + math.exp(sk))))
    return worst < 1e-12, f"max err {worst:.3g}"


def pin_window1(lib):
    w = small_workload(seed=12, window=1, scale=0.4)
    o, l = _run(lib, w)
    G = w.Hq // w.Hkv
    worst = 0.0
    for t in range(w.total_tokens):
        for h in range(w.Hq):
            s = _score(w, t, h, t)
            sk = float(w.sinks[h])
            a = 1.0 / (1.0 + math.exp(sk - s))
            worst = max(worst, np.abs(o[t, h] - a * _f64(w.v[t, h // G])).max(),
                        abs(l[t, h] - (max(s, sk) + math.log1p(math.exp(-abs(s - sk))))))
    return worst < 1e-12, f"max err {worst:.3g}"


def pin_identical_keys(lib):
    worst = 0.0
    for window in (0, 4):
        w = small_workload(seed=13, window=window, scale=0.2)
        # every key of a sequence equal to the sequence's first key (per KV head)
        k = w.k.copy()
        for si, L in enumerate(w.seqlens):
            st = int(w.cu_seqlens[si])
            k[st:st + L] = k[st]
        o, l = _run(lib, w, k=k)
        G = w.Hq // w.Hkv
        for si, L in enumerate(w.seqlens):
            st = int(w.cu_seqlens[si])
            for t in range(st, st + L):
                lo = st if window <= 0 else max(st, t - window + 1)
                n = t - lo + 1
                for h in range(w.Hq):
                    s = w.scale * float(np.dot(_f64(w.q[t, h]), _f64(k[st, h // G])))
                    sk = float(w.sinks[h])
                    Z = n * math.exp(s) + math.exp(sk)
                    mean_v = _f64(w.v[lo:t + 1, h // G]).mean(axis=0)
                    expect = mean_v * (1.0 - math.exp(sk) / Z)
                    worst = max(worst, np.abs(o[t, h] - expect).max(), abs(l[t, h] - math.log(Z)))
    return worst < 1e-12, f"max err {worst:.3g}"


def pin_big_sink(lib):
    w = small_workload(seed=14)
    big = np.full(w.Hq, 40.0)
    o, l = _run(lib, w, sinks=big)
    # |s_j| < 6 here, so the keys' share is below L*e^(6-40) ~ 1e-13.
    ok = np.abs(o).max() < 1e-11 and np.abs(l - 40.0).max() < 1e-11
    return ok, f"max|out| {np.abs(o).max():.3g}, max|lse-40| {np.abs(l - 40).max():.3g}"


# --------------------------------------------------------------------------- invariants
def pin_wide_window(lib):
    w = small_workload(seed=15)
    o0, l0 = _run(lib, w, window=0)
    o1, l1 = _run(lib, w, window=max(w.seqlens))
    o2, l2 = _run(lib, w, window=10 ** 6)
    ok = np.array_equal(o0, o1) and np.array_equal(l0, l1) and np.array_equal(o0, o2)
    return ok, "W>=L vs full"


def pin_permutation(lib):
    w = small_workload(seed=16, window=5)
    perm = [2, 0, 3, 1]
    lens = [w.seqlens[p] for p in perm]
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    idx = np.concatenate([np.arange(w.cu_seqlens[p], w.cu_seqlens[p + 1]) for p in perm])
    o, l = _run(lib, w)
    op, lp = _run(lib, w, q=w.q[idx], k=w.k[idx], v=w.v[idx], cu=cu)
    ok = np.array_equal(o[idx], op) and np.array_equal(l[idx], lp)
    return ok, "permuted pack"


def pin_gqa_repeat(lib):
    w = small_workload(seed=17, Hq=6, Hkv=2, window=3)
    G = w.Hq // w.Hkv
    o, l = _run(lib, w)
    kr = np.repeat(w.k, G, axis=1)
    vr = np.repeat(w.v, G, axis=1)
    o2, l2 = _run(lib, w, k=kr, v=vr, Hkv=w.Hq)
    ok = np.array_equal(o, o2) and np.array_equal(l, l2)
    return ok, "GQA vs repeated-KV MHA"


def pin_rows(lib):
    w = small_workload(seed=18, window=6)
    rows = inputgen.sample_rows(w, n_target=60, tile=8)
    o, l = _run(lib, w)
    orow, lrow = _run(lib, w, rows=rows)
    ok = np.array_equal(o[rows[0], rows[1]], orow) and np.array_equal(l[rows[0], rows[1]], lrow)
    return ok, "rows vs full"


def pin_no_sink_is_minus_inf(lib):
    w = small_workload(seed=19, window=2)
    o0, l0 = _run(lib, w, sinks=None)
    o1, l1 = _run(lib, w, sinks=np.full(w.Hq, -np.inf))
    ok = np.array_equal(o0, o1) and np.array_equal(l0, l1)
    return ok, "sinks NULL vs -inf"


ALL_PINS = {
    "golden": pin_golden,
    "sdpa": pin_sdpa,
    "first": pin_first_token,
    "w1": pin_window1,
    "same_k": pin_identical_keys,
    "big_sink": pin_big_sink,
    "wide": pin_wide_window,
    "perm": pin_permutation,
    "gqa": pin_gqa_repeat,
    "rows": pin_rows,
    "no_sink": pin_no_sink_is_minus_inf,
}


def run_all(lib):
    res = {}
    for name, fn in ALL_PINS.items():
        try:
            res[name] = fn(lib)
        except Exception as e:  # a mutant may also crash a pin
            res[name] = (False, f"raised {type(e).__name__}: {e}")
    return res


# --------------------------------------------------------------------------- prefill over a cache
def _kv_case(seed, q_lens, k_lens, window=0, Hq=4, Hkv=2, D=16, sinks=True, scale=0.25):
    return inputgen.make_kvcache(q_lens, k_lens, Hq, Hkv, D=D, window=window, scale=scale,
                                 seed=seed, with_sinks=sinks)


def _kv_run(lib, w, rows=None):
    s = None if w.sinks is None else w.sinks.astype(np.float64)
    out, lse, _ = oracle.mha_prefill_kvcache(w.q, w.k, w.v, s, w.cu_seqlens, w.cu_seqlens_k,
                                             w.Hq, w.Hkv, w.D, w.window, w.scale, rows=rows,
                                             nthreads=2, lib=lib)
    return out, lse


def pin_kv_equal_lengths(lib):
    """Lk == Lq is plain prefill, exactly."""
    w = _kv_case(31, [5, 17, 40], [5, 17, 40], window=6)
    o1, l1 = _kv_run(lib, w)
    o2, l2 = _run(lib, w)
    return np.array_equal(o1, o2) and np.array_equal(l1, l2), "kvcache(Lk=Lq) vs prefill"


def pin_kv_chunked_prefill(lib):
    """The last Lq tokens of a full prefill equal a prefill of those tokens
    over a cache holding the whole sequence's keys/values."""
    ok = True
    for window in (0, 5):
        full = small_workload(seed=32, seqlens=(9, 30, 41), window=window)
        o_full, l_full = _run(lib, full)
        q_lens = [3, 30, 7]
        idx = np.concatenate([np.arange(full.cu_seqlens[s + 1] - q, full.cu_seqlens[s + 1])
                              for s, q in enumerate(q_lens)])
        cu_q = np.zeros(4, np.int32)
        cu_q[1:] = np.cumsum(q_lens)
        s = full.sinks.astype(np.float64)
        o, l, _ = oracle.mha_prefill_kvcache(full.q[idx], full.k, full.v, s, cu_q,
                                             full.cu_seqlens, full.Hq, full.Hkv, full.D, window,
                                             full.scale, nthreads=2, lib=lib)
        ok &= np.array_equal(o, o_full[idx]) and np.array_equal(l, l_full[idx])
    return ok, "chunked prefill vs full prefill"


def sdpa_kvcache_reference(w):
    G = w.Hq // w.Hkv
    out = np.zeros((w.total_tokens, w.Hq, w.D))
    lse = np.zeros((w.total_tokens, w.Hq))
    qf, kf, vf = (torch.from_numpy(_f64(x)) for x in (w.q, w.k, w.v))
    for si, (Lq, Lk) in enumerate(zip(w.seqlens, w.seqlens_k)):
        if Lq == 0:
            continue
        sq, sk = int(w.cu_seqlens[si]), int(w.cu_seqlens_k[si])
        q = qf[sq:sq + Lq].permute(1, 0, 2)
        k = kf[sk:sk + Lk].repeat_interleave(G, dim=1).permute(1, 0, 2)
        v = vf[sk:sk + Lk].repeat_interleave(G, dim=1).permute(1, 0, 2)
        zero = torch.zeros(w.Hq, 1, w.D, dtype=torch.float64)
        kk, vv = torch.cat([k, zero], 1), torch.cat([v, zero], 1)
        pos = torch.arange(Lq)[:, None] + (Lk - Lq)
        ji = torch.arange(Lk)[None, :]
        allowed = ji <= pos
        if w.window > 0:
            allowed &= ji >= pos - w.window + 1
        m = torch.zeros(Lq, Lk, dtype=torch.float64).masked_fill(~allowed, float("-inf"))
        sink_col = torch.from_numpy(np.asarray(w.sinks, np.float64)).view(w.Hq, 1, 1).expand(w.Hq, Lq, 1)
        mask = torch.cat([m.expand(w.Hq, Lq, Lk), sink_col], 2)
        o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=mask, scale=w.scale)
        lg = torch.logsumexp(w.scale * (q @ kk.transpose(1, 2)) + mask, dim=-1)
        out[sq:sq + Lq] = o.permute(1, 0, 2).numpy()
        lse[sq:sq + Lq] = lg.permute(1, 0).numpy()
    return out, lse


def pin_kv_sdpa(lib):
    worst = 0.0
    for seed, ql, kl, window in [(33, [1, 4, 20], [9, 4, 50], 0), (34, [3, 16], [40, 17], 6),
                                 (35, [7], [7], 0), (36, [2, 1, 33], [2, 30, 33], 1)]:
        w = _kv_case(seed, ql, kl, window=window)
        o, l = _kv_run(lib, w)
        ro, rl = sdpa_kvcache_reference(w)
        worst = max(worst, np.abs(o - ro).max(), np.abs(l - rl).max())
    return worst < 1e-10, f"max err {worst:.3g}"


ALL_PINS.update({"kv_equal": pin_kv_equal_lengths, "kv_chunked": pin_kv_chunked_prefill,
                 "kv_sdpa": pin_kv_sdpa})
