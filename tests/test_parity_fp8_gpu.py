"""FP8 (E4M3) prefill against the CPU oracle on the exact dequantised inputs,
through the C ABI.

P is rounded to E4M3 before the PV product: three mantissa bits, round to
nearest, so the error of a probability p is at most p / 16, or half the
subnormal spacing 2^-10 below 2^-6 (the kernel's p is relative to a running
maximum no larger than the row's, so 2^-10 also bounds it relative to the
row maximum).  Hence for every output element
|out - exact| <= sum_j max(p_j / 16, 2^-10) |v_j| / l + bf16 rounding; the
small-case tests check exactly that bound per element (the bound is computed
here in float64 from the same dequantised inputs), the larger ones a
statistical tolerance: max|err| <= max|v| / 16 (one probability off by
p / 16 moving the output by at most that much, the dominant term), mean|err|
<= 5e-3 (about 10x the bf16 path's).  LSE comes from fp32 sums and keeps the
1e-3 bar."""
import numpy as np
import pytest

import inputgen
import oracle
import parity

pytestmark = pytest.mark.gpu
LSE_MAX = 1e-3
MEAN_MAX = 5e-3


def max_tol(w):
    return float(np.abs(inputgen.bf16_bits_to_f32(w.v)).max()) / 16 + 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import gqa_attention_prefill_gb300 as pkg
    from gqa_attention_prefill_gb300 import build
    build.build()
    pkg.load_library()


def run_fp8(w, with_lse=True):
    import torch
    import gqa_attention_prefill_gb300 as pkg
    f = w.fp8
    dev = "cuda"
    q8, k8, v8 = (torch.from_numpy(f[n]).to(dev) for n in ("q", "k", "v"))
    cu = torch.from_numpy(w.cu_seqlens).to(dev)
    sinks = None if w.sinks is None else torch.from_numpy(w.sinks).to(dev)
    T = w.total_tokens
    out = torch.full((T, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((T, w.Hq), float("nan"), dtype=torch.float32, device=dev) if with_lse else None
    rc = pkg.tsk_mha_prefill_fp8(q8, k8, v8, f["q_scale"], f["k_scale"], f["v_scale"], sinks, cu,
                                 w.num_seqs, T, w.Hq, w.Hkv, w.D, w.window, w.scale, out, lse)
    assert rc == 0, f"{pkg.STATUS.get(rc, rc)} {pkg.tsk_last_error()}"
    torch.cuda.synchronize()
    st = pkg.tsk_get_device_status()
    assert st == 0, pkg.STATUS.get(st, st)
    return (out.float().cpu().numpy().astype(np.float64),
            lse.cpu().numpy().astype(np.float64) if with_lse else None)


def p_rounding_bound(w):
    """sum_j max(p_j / 16, 2^-10) |v_j| / l per output element, float64 (small cases)."""
    q = inputgen.bf16_bits_to_f32(w.q).astype(np.float64)
    k = inputgen.bf16_bits_to_f32(w.k).astype(np.float64)
    v = inputgen.bf16_bits_to_f32(w.v).astype(np.float64)
    G = w.Hq // w.Hkv
    bound = np.zeros(q.shape)
    for s, L in enumerate(w.seqlens):
        a = int(w.cu_seqlens[s])
        for h in range(w.Hq):
            g = h // G
            sc = w.scale * q[a:a + L, h] @ k[a:a + L, g].T          # [L, L]
            i, j = np.meshgrid(np.arange(L), np.arange(L), indexing="ij")
            ok = (j <= i) & ((j > i - w.window) if w.window > 0 else True)
            sc = np.where(ok, sc, -np.inf)
            sink = w.sinks[h] if w.sinks is not None else -np.inf
            m = np.maximum(sc.max(axis=1), sink)
            pr = np.exp(sc - m[:, None])
            l = pr.sum(axis=1) + np.exp(sink - m)
            err_p = np.where(ok, np.maximum(pr / 16, 2.0 ** -10), 0.0)
            bound[a:a + L, h] = (err_p @ np.abs(v[a:a + L, g])) / l[:, None]
    return bound


@pytest.mark.parametrize("seqlens,window", [([1], 0), ([128], 0), ([129, 3, 300], 0),
                                             ([700], 0), ([400, 257], 100), ([500], 1)])
def test_small_cases_within_the_rounding_bound(seqlens, window):
    w = inputgen.make_fp8(seqlens, 8, 2, window=window, seed=sum(seqlens) + window)
    out, lse = run_fp8(w)
    ro, rl, _ = oracle.run_workload(w)
    b = p_rounding_bound(w)
    err = np.abs(out - ro)
    slack = np.abs(ro) * 2.0 ** -8 + 1e-4   # bf16 rounding of out, fp32 accumulation
    worst = (err - b - slack).max()
    print(f"L={seqlens} W={window}: out max {err.max():.3g} mean {err.mean():.3g} "
          f"(bound max {b.max():.3g}), lse max {np.abs(lse - rl).max():.3g}")
    assert worst <= 0, f"bound exceeded by {worst}"
    assert np.abs(lse - rl).max() <= LSE_MAX


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 1), (6, 2), (64, 8)])
def test_head_groupings(Hq, Hkv):
    w = inputgen.make_fp8([333, 129], Hq, Hkv, seed=Hq + Hkv)
    out, lse = run_fp8(w)
    ro, rl, _ = oracle.run_workload(w)
    err = np.abs(out - ro)
    print(f"Hq={Hq},Hkv={Hkv}: out max {err.max():.3g} mean {err.mean():.3g}, "
          f"lse max {np.abs(lse - rl).max():.3g}")
    assert err.max() <= max_tol(w) and err.mean() <= MEAN_MAX
    assert np.abs(lse - rl).max() <= LSE_MAX


def test_no_sinks_no_lse():
    w = inputgen.make_fp8([200, 77], 8, 2, seed=2, with_sinks=False)
    out, _ = run_fp8(w, with_lse=False)
    ro, _, _ = oracle.run_workload(w)
    err = np.abs(out - ro)
    assert err.max() <= max_tol(w) and err.mean() <= MEAN_MAX


def test_bench_config_sampled():
    w = inputgen.config("fp8_causal_4x4096_h64kv8")
    out, lse = run_fp8(w)
    t, h = inputgen.sample_rows(w, n_target=4096)
    ro, rl, _ = oracle.mha_prefill_rows(w.q, w.k, w.v, w.sinks, w.cu_seqlens, w.Hq, w.Hkv, w.D,
                                        w.window, w.scale, t, h)
    o = out[t, h]
    err = np.abs(o - ro)
    print(f"fp8 bench config [{len(t)} rows]: out max {err.max():.3g} mean {err.mean():.3g}, "
          f"lse max {np.abs(lse[t, h] - rl).max():.3g}")
    assert np.isfinite(out).all()
    assert err.max() <= max_tol(w) and err.mean() <= MEAN_MAX
    assert np.abs(lse[t, h] - rl).max() <= LSE_MAX
