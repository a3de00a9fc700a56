"""One decoding step over a key/value cache (tsk_mha_decode_kvcache) against
the CPU oracle's prefill-over-a-cache with one query per sequence, through
the C ABI."""
import numpy as np
import pytest

import inputgen
import oracle
import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import gqa_attention_prefill_gb300 as pkg
    from gqa_attention_prefill_gb300 import build
    build.build()
    pkg.load_library()


def run_decode(w, with_lse=True, max_k=None, check_status=True):
    import torch
    import gqa_attention_prefill_gb300 as pkg
    d = parity.to_device(w)
    B = w.num_seqs
    out = torch.full((B, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, w.Hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    mk = max(w.seqlens_k) if max_k is None else max_k
    rc = pkg.tsk_mha_decode_kvcache(d["q"], d["k"], d["v"], d["sinks"], d["cu_k"], B, w.total_keys,
                                    mk, w.Hq, w.Hkv, w.D, w.window, w.scale, out, lse)
    assert rc == 0, f"{pkg.STATUS.get(rc, rc)} {pkg.tsk_last_error()}"
    torch.cuda.synchronize()
    if check_status:
        st = pkg.tsk_get_device_status()
        assert st == 0, pkg.STATUS.get(st, st)
    return out, lse


def check(w, with_lse=True, label=""):
    out, lse = run_decode(w, with_lse=with_lse)
    ro, rl, _ = oracle.run_workload(w)
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64) if with_lse else None
    return parity.compare(o, l, ro, rl, label)


def decode_case(k_lens, Hq=8, Hkv=2, D=64, window=0, seed=0, **kw):
    scale = kw.pop("scale", D ** -0.5)
    return inputgen.make_kvcache([1] * len(k_lens), k_lens, Hq, Hkv, D=D, window=window,
                                 scale=scale, seed=seed, **kw)


@pytest.mark.parametrize("k_lens", [[1], [2], [127], [128], [129], [1000], [5000],
                                    [1, 300, 129, 4096, 2, 777]])
def test_lengths(k_lens):
    print(check(decode_case(k_lens, seed=sum(k_lens)), label=f"Lk={k_lens}"))


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 1), (6, 2), (3, 1), (32, 2), (64, 2), (64, 8)])
def test_head_groupings(Hq, Hkv):
    print(check(decode_case([700, 33, 2100], Hq, Hkv, seed=Hq * 3 + Hkv), label=f"Hq={Hq},Hkv={Hkv}"))


@pytest.mark.parametrize("window", [1, 5, 128, 129, 1000])
def test_windows(window):
    print(check(decode_case([1, 100, 2000, 129], window=window, seed=window), label=f"W={window}"))


@pytest.mark.parametrize("D", [64, 128])
def test_long_sequence_many_splits(D):
    """One or two sequences with long caches: the keys are split over many CTAs."""
    print(check(decode_case([20000, 3], Hq=16, Hkv=2, D=D, seed=D), label=f"D={D} split"))


@pytest.mark.parametrize("k_lens,window", [([1, 129, 1000, 4000], 0), ([300, 5000], 200)])
def test_head_dim_128(k_lens, window):
    print(check(decode_case(k_lens, Hq=32, Hkv=8, D=128, window=window, seed=5),
                label=f"D=128 Lk={k_lens} W={window}"))


def test_no_sinks_no_lse():
    print(check(decode_case([50, 3000], seed=2, with_sinks=False), with_lse=False,
                label="no sinks, no lse"))


def test_extreme_logits():
    print(check(decode_case([600, 4097], seed=13, scale=0.3, sink_sigma=6.0), label="large logits"))


@pytest.mark.parametrize("name", ["decode_64x8192_h64kv8", "decode_ragged32_h64kv8"])
def test_bench_configs_full(name):
    print(check(inputgen.config(name), label=name))


def test_matches_prefill_over_cache():
    """The decode path and the prefill-over-a-cache path compute the same rows."""
    w = decode_case([1, 700, 3000, 129], Hq=16, Hkv=4, seed=8)
    od, ld = run_decode(w)
    op, lp = parity.run_gpu(w)
    assert np.abs(od.float().cpu().numpy() - op.float().cpu().numpy()).max() < 2e-2
    assert np.abs(ld.cpu().numpy() - lp.cpu().numpy()).max() < 1e-3


def test_bad_offsets_reported_and_nothing_written():
    import torch
    import gqa_attention_prefill_gb300 as pkg
    w = decode_case([10, 20, 30], seed=1)
    d = parity.to_device(w)
    d["cu_k"] = torch.tensor([0, 10, 10, 60], dtype=torch.int32, device="cuda")  # empty sequence
    out = torch.full((3, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = pkg.tsk_mha_decode_kvcache(d["q"], d["k"], d["v"], d["sinks"], d["cu_k"], 3, 60, 50,
                                    w.Hq, w.Hkv, w.D, 0, w.scale, out, None)
    assert rc == 0
    torch.cuda.synchronize()
    assert pkg.tsk_get_device_status() == -8
    assert torch.isnan(out.float()).all()
    # a valid call afterwards works
    print(check(w, label="after a rejected call"))


def test_deterministic():
    w = decode_case([5000, 17, 900], Hq=16, Hkv=2, seed=3)
    o1, l1 = run_decode(w)
    o2, l2 = run_decode(w)
    assert np.array_equal(o1.float().cpu().numpy(), o2.float().cpu().numpy())
    assert np.array_equal(l1.cpu().numpy(), l2.cpu().numpy())
