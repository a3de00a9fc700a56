"""tsk_mha_prefill_host: host buffers in and out, chunked copies overlapped
with the attention.  Each chunk of consecutive tokens is computed as a
prefill over the keys already on the device.  Chunks end at sequence ends or
at multiples of 128 rows from the start of the sequence they cut, so every
query tile (and every warp of 32 rows, which shares the softmax's rescaling
decisions) is the one the device entry point forms: the results must be bit
for bit the same.  These tests check that, and the host path against the
oracle, on problems whose sequences straddle chunk boundaries."""
import numpy as np
import pytest

import inputgen
import oracle
import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    import gqa_attention_prefill_gb300 as pkg
    from gqa_attention_prefill_gb300 import build
    build.build()
    pkg.load_library()
    return pkg


def run_host(pkg, w, pinned=True, with_lse=True, stream=None):
    import torch
    T = w.total_tokens

    def host(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if dtype is not None:
            t = t.view(dtype)
        return t.pin_memory() if pinned else t

    q = host(w.q.view(np.int16), torch.bfloat16)
    k = host(w.k.view(np.int16), torch.bfloat16)
    v = host(w.v.view(np.int16), torch.bfloat16)
    s = None if w.sinks is None else host(w.sinks)
    cu = host(w.cu_seqlens)
    out = torch.full((T, w.Hq, w.D), float("nan"), dtype=torch.bfloat16)
    lse = torch.full((T, w.Hq), float("nan"), dtype=torch.float32) if with_lse else None
    if pinned:
        out = out.pin_memory()
        lse = lse.pin_memory() if lse is not None else None
    stream = stream or torch.cuda.current_stream()
    rc = pkg.tsk_mha_prefill_host(q, k, v, s, cu, w.num_seqs, T, w.Hq, w.Hkv, w.D, w.window,
                                  w.scale, out, lse, stream)
    assert rc == 0, f"{pkg.STATUS.get(rc, rc)} {pkg.tsk_last_error()}"
    stream.synchronize()
    assert pkg.tsk_get_device_status(stream) == 0
    return out, lse


def same_as_device(pkg, w, **kw):
    """Host path against the oracle (4096 sampled rows, the usual
    tolerances), and bit for bit against the device path."""
    import torch
    with_lse = kw.get("with_lse", True)
    out, lse = run_host(pkg, w, **kw)
    t, h = inputgen.sample_rows(w, n_target=4096)
    ro, rl, _ = oracle.run_workload(w, rows=(t, h))
    o = out.float().numpy().astype(np.float64)
    l = lse.numpy().astype(np.float64) if with_lse else None
    print(parity.compare(o[t, h], l[t, h] if with_lse else None, ro, rl if with_lse else None,
                         f"host path {w.seqlens} W={w.window} [{len(t)} rows]"))
    ref_out, ref_lse = parity.run_gpu(w, with_lse=with_lse)
    assert torch.equal(out.view(torch.int16), ref_out.cpu().view(torch.int16))
    if with_lse:
        assert torch.equal(lse, ref_lse.cpu())
    return out, lse


@pytest.mark.parametrize("seqlens,window", [
    ([3000, 0, 5000, 1, 129, 7000], 0),      # 8 chunks of 2048 tokens, splits inside sequences
    ([3000, 0, 5000, 1, 129, 7000], 128),
    ([3000, 0, 5000, 1, 129, 7000], 1000),
    ([20000], 0),                            # one sequence cut into 8 chunks
    ([20000], 300),
    ([100, 2047, 2049, 1, 4096, 4095], 0),   # boundaries next to chunk edges
    ([200, 1, 129], 0),                      # a single chunk
])
def test_matches_device_entry_point(pkg, seqlens, window):
    w = inputgen.make(seqlens, 16, 2, window=window, seed=sum(seqlens) + window)
    same_as_device(pkg, w)


def test_one_query_head_per_kv_head(pkg):
    """Hq == Hkv: units of two row blocks of one head, chunks ending on odd
    128-row boundaries."""
    w = inputgen.make([3000, 0, 5000, 129, 7000], 4, 4, seed=68)
    same_as_device(pkg, w)
    w = inputgen.make([9000, 3000], 4, 4, D=128, window=300, scale=128 ** -0.5, seed=69)
    same_as_device(pkg, w)


def test_head_dim_128_and_no_sinks_no_lse(pkg):
    w = inputgen.make([5000, 9000, 3], 8, 2, D=128, window=0, seed=61)
    same_as_device(pkg, w)
    w = inputgen.make([6000, 6000], 8, 8, window=64, seed=62, with_sinks=False)
    same_as_device(pkg, w, with_lse=False)


def test_pageable_host_memory(pkg):
    w = inputgen.make([3000, 4000], 8, 2, seed=63)
    same_as_device(pkg, w, pinned=False)


def test_against_the_oracle_sampled(pkg):
    """Full-size bench problem through host buffers, sampled rows against the
    oracle."""
    w = inputgen.config("causal_4x4096_h64kv8")
    out, lse = run_host(pkg, w)
    t, h = inputgen.sample_rows(w, n_target=4096)
    ro, rl, _ = oracle.run_workload(w, rows=(t, h))
    o = out.float().numpy().astype(np.float64)[t, h]
    l = lse.numpy().astype(np.float64)[t, h]
    print(parity.compare(o, l, ro, rl, f"host path {w.name} [{len(t)} rows]"))


def test_buffer_grows_and_calls_stay_ordered(pkg):
    """Small, then large, then small again on one stream, without
    synchronising in between (the second call must wait for the first's
    copies back before it reuses the device buffer)."""
    import torch
    s = torch.cuda.Stream()
    ws = [inputgen.make([500, 700], 8, 2, seed=64), inputgen.make([9000, 7000], 8, 2, seed=65),
          inputgen.make([1300], 8, 2, seed=66)]
    for w in ws:
        same_as_device(pkg, w, stream=s)


def test_release_then_call_again(pkg):
    """tsk_release frees the pipeline's streams and buffer; the next call
    creates them again."""
    w = inputgen.make([2500, 300], 8, 2, seed=67)
    same_as_device(pkg, w)
    assert pkg.load_library().tsk_release() == 0
    same_as_device(pkg, w)
