"""Shared helpers for GPU parity tests: run the CUDA path through the C ABI on
a seeded workload and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np

import inputgen
import oracle

# Tolerances for bf16 I/O: outputs max |d| <= 2e-2 and mean |d| <= 2e-3;
# LSE |d| <= 1e-3 absolute.
OUT_MAX = 2e-2
OUT_MEAN = 2e-3
LSE_MAX = 1e-3


def to_device(w: inputgen.Workload, device="cuda"):
    import torch
    d = {
        "q": torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16).to(device),
        "k": torch.from_numpy(w.k.view(np.int16)).view(torch.bfloat16).to(device),
        "v": torch.from_numpy(w.v.view(np.int16)).view(torch.bfloat16).to(device),
        "cu": torch.from_numpy(w.cu_seqlens).to(device),
        "sinks": None if w.sinks is None else torch.from_numpy(w.sinks).to(device),
    }
    if w.cu_seqlens_k is not None:
        d["cu_k"] = torch.from_numpy(w.cu_seqlens_k).to(device)
    return d


def run_gpu(w: inputgen.Workload, d=None, with_lse=True, check_status=True):
    """Returns (out bf16 torch [T,Hq,D], lse fp32 torch [T,Hq] or None)."""
    import torch
    import gqa_attention_prefill_gb300 as pkg
    d = d or to_device(w)
    T = w.total_tokens
    out = torch.full((T, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device=d["q"].device)
    lse = torch.full((T, w.Hq), float("nan"), dtype=torch.float32, device=d["q"].device) \
        if with_lse else None
    if w.cu_seqlens_k is not None:
        rc = pkg.tsk_mha_prefill_kvcache(d["q"], d["k"], d["v"], d["sinks"], d["cu"], d["cu_k"],
                                         w.num_seqs, T, w.total_keys, w.Hq, w.Hkv, w.D, w.window,
                                         w.scale, out, lse)
    else:
        rc = pkg.tsk_mha_prefill(d["q"], d["k"], d["v"], d["sinks"], d["cu"], w.num_seqs, T,
                                 w.Hq, w.Hkv, w.D, w.window, w.scale, out, lse)
    assert rc == 0, f"{pkg.STATUS.get(rc, rc)} {pkg.tsk_last_error()}"
    torch.cuda.synchronize()
    if check_status:
        st = pkg.tsk_get_device_status()
        assert st == 0, f"{pkg.STATUS.get(st, st)}: {pkg.tsk_last_error()}"
    return out, lse


def compare(gpu_out, gpu_lse, ref_out, ref_lse, label=""):
    """gpu_*: numpy float64 (any shape matching ref_*)."""
    assert np.isfinite(gpu_out).all(), f"{label}: non-finite outputs"
    d = np.abs(gpu_out - ref_out)
    msg = f"{label}: out max {d.max():.3g} mean {d.mean():.3g}"
    assert d.max() <= OUT_MAX and d.mean() <= OUT_MEAN, msg
    if gpu_lse is not None:
        assert np.isfinite(gpu_lse).all(), f"{label}: non-finite lse"
        dl = np.abs(gpu_lse - ref_lse)
        msg += f", lse max {dl.max():.3g}"
        assert dl.max() <= LSE_MAX, msg
    return msg


def check_full(w: inputgen.Workload, with_lse=True, label=None):
    out, lse = run_gpu(w, with_lse=with_lse)
    ro, rl, _ = oracle.run_workload(w)
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64) if with_lse else None
    return compare(o, l, ro, rl, label or w.name)


def check_sampled(w: inputgen.Workload, n_rows=4096, label=None, d=None):
    out, lse = run_gpu(w, d=d)
    t, h = inputgen.sample_rows(w, n_target=n_rows)
    assert len(t) >= min(n_rows, w.total_tokens * w.Hq)
    ro, rl, _ = oracle.run_workload(w, rows=(t, h))
    import torch
    ti = torch.from_numpy(t).to(out.device)
    hi = torch.from_numpy(h.astype(np.int64)).to(out.device)
    o = out[ti, hi].float().cpu().numpy().astype(np.float64)
    l = lse[ti, hi].cpu().numpy().astype(np.float64)
    # every output must be finite, not only the sampled rows
    assert bool(torch.isfinite(out).all()) and bool(torch.isfinite(lse).all()), "non-finite rows"
    return compare(o, l, ro, rl, (label or w.name) + f" [{len(t)} rows]")


def few_key_rounding_bound(w):
    """sum_j (p_j / 256)|v_j| / l per output element for a window of a few
    keys (the bf16 rounding of P, relative to the maximum in use), with the
    query rows of a KV-cache sequence at key positions Lk - Lq + i."""
    q = inputgen.bf16_bits_to_f32(w.q).astype(np.float64)
    k = inputgen.bf16_bits_to_f32(w.k).astype(np.float64)
    v = inputgen.bf16_bits_to_f32(w.v).astype(np.float64)
    G, W = w.Hq // w.Hkv, w.window
    bound = np.zeros((w.total_tokens, w.Hq, w.D))
    for s_, Lq in enumerate(w.seqlens):
        a = int(w.cu_seqlens[s_])
        if w.cu_seqlens_k is not None:
            ak, Lk = int(w.cu_seqlens_k[s_]), int(w.seqlens_k[s_])
        else:
            ak, Lk = a, Lq
        pos = (Lk - Lq) + np.arange(Lq)
        for h in range(w.Hq):
            qh, kg, vg = q[a:a + Lq, h], k[ak:ak + Lk, h // G], np.abs(v[ak:ak + Lk, h // G])
            # scores of the keys d = 0 .. W-1 back from each query (-inf before the start)
            sc = np.full((W, Lq), -np.inf)
            for d in range(W):
                ok = pos - d >= 0
                sc[d, ok] = w.scale * np.einsum("id,id->i", qh[ok], kg[pos[ok] - d])
            m = np.maximum(sc.max(axis=0), w.sinks[h])
            pr = np.exp(sc - m)
            l = pr.sum(axis=0) + np.exp(w.sinks[h] - m)
            acc = np.zeros((Lq, w.D))
            for d in range(W):
                ok = pos - d >= 0
                acc[ok] += (pr[d, ok] / 256)[:, None] * vg[pos[ok] - d]
            bound[a:a + Lq, h] = acc / l[:, None]
    return bound
