"""The per-element bound that the few-key window tests hold the GPU output to
(tests/parity.py, few_key_rounding_bound) checked on the CPU: an output
whose probabilities are rounded to bf16 before P·V, as the kernels round P,
stays inside it, and one whose probabilities are off by 2^-6 (four times the
bf16 half-ulp) leaves it.  Rows take the window's one or two keys and the
sink; the KV-cache form puts them at the end of a longer key sequence."""
import numpy as np
import pytest

import inputgen
import oracle
import parity


def _bf16(x):
    """Round fp64 values to bf16 (round to nearest even) through fp32."""
    f = np.asarray(x, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16 << 16
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def _output_with(w, perturb):
    """out[t, h] = sum_j perturb(p_j) v_j / l with l from the exact p_j."""
    q = inputgen.bf16_bits_to_f32(w.q).astype(np.float64)
    k = inputgen.bf16_bits_to_f32(w.k).astype(np.float64)
    v = inputgen.bf16_bits_to_f32(w.v).astype(np.float64)
    G, W = w.Hq // w.Hkv, w.window
    out = np.zeros((w.total_tokens, w.Hq, w.D))
    for s_, Lq in enumerate(w.seqlens):
        a = int(w.cu_seqlens[s_])
        if w.cu_seqlens_k is not None:
            ak, Lk = int(w.cu_seqlens_k[s_]), int(w.seqlens_k[s_])
        else:
            ak, Lk = a, Lq
        for i in range(Lq):
            pos = Lk - Lq + i
            keys = [ak + pos - d for d in range(W) if pos - d >= 0]
            for h in range(w.Hq):
                sc = np.array([w.scale * q[a + i, h] @ k[j, h // G] for j in keys])
                m = max(sc.max(), w.sinks[h])
                p = np.exp(sc - m)
                l = p.sum() + np.exp(w.sinks[h] - m)
                out[a + i, h] = (perturb(p)[:, None] * v[keys, h // G]).sum(axis=0) / l
    return out


@pytest.mark.parametrize("kvcache", [False, True])
@pytest.mark.parametrize("window", [1, 2])
def test_bound_admits_bf16_probabilities_and_rejects_larger_errors(window, kvcache):
    if kvcache:
        w = inputgen.make_kvcache([130, 40], [300, 40], 4, 2, window=window, seed=60 + window)
    else:
        w = inputgen.make([130, 40], 4, 2, window=window, seed=70 + window)
    ro, _, _ = oracle.run_workload(w)
    bound = parity.few_key_rounding_bound(w)
    # the oracle's own output is the exact one: the bound is not needed for it
    np.testing.assert_allclose(_output_with(w, lambda p: p), ro, rtol=0, atol=1e-12)
    rounded = _output_with(w, _bf16)
    assert (np.abs(rounded - ro) - bound).max() <= 1e-12
    off = _output_with(w, lambda p: p * (1 + 2.0 ** -6))
    assert (np.abs(off - ro) - bound).max() > 0
