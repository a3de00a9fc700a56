"""Prefill over a key/value cache (tsk_mha_prefill_kvcache) against the CPU
oracle, through the C ABI."""
import numpy as np
import pytest

import inputgen
import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import gqa_attention_prefill_gb300 as pkg
    from gqa_attention_prefill_gb300 import build
    build.build()
    pkg.load_library()


@pytest.mark.parametrize("q_lens,k_lens", [
    ([1], [1]), ([1], [9]), ([1], [129]), ([5], [300]), ([128], [128]), ([129], [1000]),
    ([300], [557]), ([64, 1, 200, 0, 3], [64, 700, 455, 10, 3]), ([2, 257], [4000, 257]),
])
def test_lengths(q_lens, k_lens):
    w = inputgen.make_kvcache(q_lens, k_lens, 8, 2, seed=sum(q_lens) + sum(k_lens))
    print(parity.check_full(w, label=f"Lq={q_lens} Lk={k_lens}"))


@pytest.mark.parametrize("window", [1, 5, 128, 129, 200, 600, 3000])
def test_windows(window):
    w = inputgen.make_kvcache([1, 100, 300, 129], [50, 1000, 300, 2048], 8, 2, window=window,
                              seed=window + 7)
    print(parity.check_full(w, label=f"W={window}"))


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (3, 1), (64, 8)])
def test_head_groupings(Hq, Hkv):
    w = inputgen.make_kvcache([77, 256], [500, 300], Hq, Hkv, seed=Hq + Hkv)
    print(parity.check_full(w, label=f"Hq={Hq},Hkv={Hkv}"))


def test_no_sinks_no_lse():
    w = inputgen.make_kvcache([100, 40], [900, 41], 8, 2, seed=3, with_sinks=False)
    print(parity.check_full(w, with_lse=False, label="no sinks, no lse"))


def test_chunked_prefill_matches_full_prefill():
    """Prefilling a sequence in chunks over the growing cache gives the rows of
    one full prefill (within rounding: tiles align differently)."""
    import torch
    full = inputgen.make([1000, 700], 16, 2, seed=41, window=0)
    d = parity.to_device(full)
    ref_out, ref_lse = parity.run_gpu(full, d)
    for chunk in (256, 300):
        for s, L in enumerate(full.seqlens):
            st = int(full.cu_seqlens[s])
            for c0 in range(0, L, chunk):
                c1 = min(L, c0 + chunk)
                w = inputgen.Workload("chunk", [c1 - c0], full.Hq, full.Hkv, full.D, 0, full.scale,
                                      full.q[st + c0:st + c1], full.k[st:st + c1],
                                      full.v[st:st + c1], full.sinks,
                                      np.array([0, c1 - c0], np.int32), 0,
                                      cu_seqlens_k=np.array([0, c1], np.int32), seqlens_k=[c1])
                out, lse = parity.run_gpu(w)
                a = out.float().cpu().numpy().astype(np.float64)
                b = ref_out[st + c0:st + c1].float().cpu().numpy().astype(np.float64)
                la = lse.cpu().numpy().astype(np.float64)
                lb = ref_lse[st + c0:st + c1].cpu().numpy().astype(np.float64)
                assert np.abs(a - b).max() <= parity.OUT_MAX and np.abs(la - lb).max() <= 1e-4


def test_bench_config_sampled():
    print(parity.check_sampled(inputgen.config("kvcache_4x2048_on_4096_h64kv8")))


def test_bad_offsets_reported():
    import torch
    import gqa_attention_prefill_gb300 as pkg
    w = inputgen.make_kvcache([100], [100], 4, 1, seed=5)
    d = parity.to_device(w)
    out = torch.zeros((100, 4, 64), dtype=torch.bfloat16, device="cuda")
    bad_k = torch.tensor([0, 99], dtype=torch.int32, device="cuda")   # Lk < Lq
    rc = pkg.tsk_mha_prefill_kvcache(d["q"], d["k"], d["v"], d["sinks"], d["cu"], bad_k, 1, 100,
                                     99, 4, 1, 64, 0, 0.125, out, None)
    assert rc == -1   # total_k < total_q is caught on the host
    bad_k = torch.tensor([0, 99], dtype=torch.int32, device="cuda")
    rc = pkg.tsk_mha_prefill_kvcache(d["q"], d["k"], d["v"], d["sinks"], d["cu"], bad_k, 1, 100,
                                     100, 4, 1, 64, 0, 0.125, out, None)
    assert rc == 0 and pkg.tsk_get_device_status() == -8
    assert bool((out == 0).all())
