"""Head dimension 128 (its own kernel) against the CPU oracle, through the C
ABI: every row on small cases, sampled rows on the full-size configs."""
import numpy as np
import pytest

import inputgen
import parity

pytestmark = pytest.mark.gpu
SCALE = 128 ** -0.5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import gqa_attention_prefill_gb300 as pkg
    from gqa_attention_prefill_gb300 import build
    build.build()
    pkg.load_library()


@pytest.mark.parametrize("seqlens", [[1], [2], [127], [128], [129], [255], [257],
                                     [1, 128, 0, 129, 3, 700]])
def test_lengths(seqlens):
    w = inputgen.make(seqlens, 8, 2, D=128, scale=SCALE, seed=sum(seqlens) + 11)
    print(parity.check_full(w, label=f"D=128 L={seqlens}"))


@pytest.mark.parametrize("window", [1, 2, 127, 128, 129, 200, 1000])
def test_windows(window):
    w = inputgen.make([300, 1, 1000, 129], 8, 2, D=128, scale=SCALE, window=window,
                      seed=window + 5)
    print(parity.check_full(w, label=f"D=128 W={window}"))


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 1), (6, 2), (3, 1), (32, 8)])
def test_head_groupings(Hq, Hkv):
    w = inputgen.make([200, 333], Hq, Hkv, D=128, scale=SCALE, seed=Hq * 7 + Hkv)
    print(parity.check_full(w, label=f"D=128 Hq={Hq},Hkv={Hkv}"))


def test_no_sinks_no_lse():
    w = inputgen.make([130, 64, 500], 8, 2, D=128, scale=SCALE, seed=9, with_sinks=False)
    print(parity.check_full(w, with_lse=False, label="D=128 no sinks, no lse"))


def test_extreme_logits():
    w = inputgen.make([600, 257], 8, 2, D=128, scale=0.3, k_mult=4.0, sink_sigma=6.0, seed=12)
    print(parity.check_full(w, label="D=128 large logits"))


@pytest.mark.parametrize("q_lens,k_lens", [([1, 100, 129], [1, 900, 300]), ([300], [2049])])
def test_kvcache(q_lens, k_lens):
    w = inputgen.make_kvcache(q_lens, k_lens, 8, 2, D=128, scale=SCALE, seed=sum(k_lens))
    print(parity.check_full(w, label=f"D=128 kvcache Lq={q_lens} Lk={k_lens}"))


@pytest.mark.parametrize("name", ["causal_4x4096_h32kv8_d128", "long_1x32768_h32kv8_d128"])
def test_bench_configs_sampled(name):
    w = inputgen.config(name)
    print(parity.check_sampled(w, n_rows=4096, label=name))


def test_deterministic():
    w = inputgen.make([1000, 517], 16, 4, D=128, scale=SCALE, seed=4)
    d = parity.to_device(w)
    o1, l1 = parity.run_gpu(w, d)
    o2, l2 = parity.run_gpu(w, d)
    assert np.array_equal(o1.view(dtype=o1.dtype).cpu().float().numpy(),
                          o2.cpu().float().numpy())
    assert np.array_equal(l1.cpu().numpy(), l2.cpu().numpy())
