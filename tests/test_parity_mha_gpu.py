"""One query head per KV head (Hq == Hkv, plain multi-head attention).

There a work unit takes two consecutive 128-row query tiles of one head
(schedule entries of 256 rows, key range the union of the two tiles'),
instead of two query heads of a group over the same rows.  These cases
cover an odd number of query tiles (a unit with one tile), sequence ends
inside either tile, windows (the second tile's first key tile can be fully
masked for it), the KV-cache path, D = 128 and the allocation-free entry
point, every row against the oracle."""
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


@pytest.mark.parametrize("seqlens", [[1], [128], [129], [256], [257], [383], [384], [385],
                                     [1, 255, 256, 257, 640, 0, 700]])
@pytest.mark.parametrize("D", [64, 128])
def test_lengths(seqlens, D):
    w = inputgen.make(seqlens, 4, 4, D=D, scale=D ** -0.5, seed=sum(seqlens) + D)
    print(parity.check_full(w, label=f"MHA D={D} L={seqlens}"))


@pytest.mark.parametrize("window", [1, 100, 128, 129, 200, 300, 1000])
@pytest.mark.parametrize("D", [64, 128])
def test_windows(window, D):
    w = inputgen.make([300, 1000, 129], 4, 4, D=D, window=window, scale=D ** -0.5,
                      seed=window + D)
    print(parity.check_full(w, label=f"MHA D={D} W={window}"))


def test_no_sinks_no_lse():
    w = inputgen.make([600, 257], 8, 8, seed=5, with_sinks=False)
    print(parity.check_full(w, with_lse=False, label="MHA no sinks, no lse"))


@pytest.mark.parametrize("q_lens,k_lens,window", [
    ([300, 1, 257], [1000, 9, 257], 0), ([129, 500], [700, 500], 200), ([256], [4096], 0)])
def test_kvcache(q_lens, k_lens, window):
    w = inputgen.make_kvcache(q_lens, k_lens, 4, 4, window=window, seed=sum(k_lens) + window)
    print(parity.check_full(w, label=f"MHA kvcache Lq={q_lens} Lk={k_lens} W={window}"))


def test_full_size_sampled():
    for name in ("causal_4x4096_h64kv64", "causal_4x4096_h32kv32_d128"):
        print(parity.check_sampled(inputgen.config(name)))


def test_noalloc_matches_allocating_entry_point():
    import torch
    import gqa_attention_prefill_gb300 as pkg
    w = inputgen.make([700, 129, 1024], 8, 8, window=0, seed=9)
    d = parity.to_device(w)
    ref_out, ref_lse = parity.run_gpu(w, d)
    out = torch.empty_like(ref_out)
    lse = torch.empty_like(ref_lse)
    rc = pkg.tsk_mha_prefill_noalloc(d["q"], d["k"], d["v"], d["sinks"], d["cu"], w.num_seqs,
                                     w.total_tokens, w.Hq, w.Hkv, w.D, w.window, w.scale, out, lse)
    assert rc == 0
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse, ref_lse)
