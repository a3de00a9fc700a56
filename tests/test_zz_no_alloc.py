"""The allocation-free entry point, tsk_mha_prefill_noalloc.

It exists for callers that must not allocate device memory while they run
(for instance code inside a serving engine that has reserved the whole
device, or latency-critical paths where an allocation's implicit
synchronisation is not acceptable).  Its scratch is a fixed array inside the
library.  This file is collected last so that a failure here does not stop
the other GPU tests; it passes both on its own in a fresh process and after
them.

The call runs the same scheduler and attention kernels as tsk_mha_prefill on
the same query tiles, so its outputs must be bit for bit those of the
allocating call; both are also compared with the CPU oracle.
"""
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


def _outputs(w, like):
    import torch
    out = torch.full((w.total_tokens, w.Hq, w.D), float("nan"), dtype=torch.bfloat16,
                     device=like.device)
    lse = torch.full((w.total_tokens, w.Hq), float("nan"), dtype=torch.float32,
                     device=like.device)
    return out, lse


def _noalloc(pkg, w, d, out, lse, stream=None, cu=None):
    return pkg.tsk_mha_prefill_noalloc(d["q"], d["k"], d["v"], d["sinks"],
                                       d["cu"] if cu is None else cu, w.num_seqs,
                                       w.total_tokens, w.Hq, w.Hkv, w.D, w.window, w.scale,
                                       out, lse, stream)


@pytest.mark.parametrize("seed,lens,Hq,Hkv,window", [
    (31, [300, 1, 4096, 129], 16, 2, 0),
    (32, [2048, 77, 515], 16, 2, 128),
    (33, [129, 700, 1], 4, 4, 0),          # one query head per KV head
])
def test_noalloc_is_bitwise_the_allocating_call_and_matches_the_oracle(pkg, seed, lens, Hq,
                                                                       Hkv, window):
    import torch
    w = inputgen.make(lens, Hq, Hkv, window=window, seed=seed)
    d = parity.to_device(w)
    ref_out, ref_lse = parity.run_gpu(w, d)
    ro, rl, _ = oracle.run_workload(w)
    print(parity.compare(ref_out.float().cpu().numpy().astype(np.float64),
                         ref_lse.cpu().numpy().astype(np.float64), ro, rl,
                         f"tsk_mha_prefill seed {seed}"))
    # two calls in a row: the second must not depend on what the first left
    # in the shared array
    for call in range(2):
        out, lse = _outputs(w, d["q"])
        rc = _noalloc(pkg, w, d, out, lse)
        assert rc == 0, f"{pkg.STATUS.get(rc, rc)} {pkg.tsk_last_error()}"
        assert pkg.tsk_noalloc_status() == 0
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), \
            f"seed {seed} call {call}: outputs differ from tsk_mha_prefill"
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32)), \
            f"seed {seed} call {call}: lse differs from tsk_mha_prefill"
        print(parity.compare(out.float().cpu().numpy().astype(np.float64),
                             lse.cpu().numpy().astype(np.float64), ro, rl,
                             f"noalloc seed {seed} call {call}"))


def test_noalloc_allocates_no_device_memory(pkg):
    import torch
    w = inputgen.make([1000, 3000, 17], 16, 2, window=0, seed=34)
    d = parity.to_device(w)
    out, lse = _outputs(w, d["q"])
    s = torch.cuda.Stream()   # a stream no entry point has used: nothing is cached for it
    assert _noalloc(pkg, w, d, out, lse, stream=s) == 0   # warm: module and symbol look-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    assert _noalloc(pkg, w, d, out, lse, stream=s) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert pkg.tsk_noalloc_status(s) == 0


def test_noalloc_reports_inconsistent_seqlens(pkg):
    import torch
    w = inputgen.make([300, 200, 500], 8, 2, window=0, seed=35)
    d = parity.to_device(w)
    bad = torch.tensor([0, 300, 200, 1000], dtype=torch.int32, device="cuda")  # decreasing
    out, lse = _outputs(w, d["q"])
    assert _noalloc(pkg, w, d, out, lse, cu=bad) == 0   # only the device can see it
    assert pkg.tsk_noalloc_status() == -8
    assert bool(torch.isnan(out.float()).all()), "outputs were written despite bad cu_seqlens"
    assert pkg.tsk_noalloc_status() == 0                 # read once, then cleared
    # the next call with valid offsets computes normally
    out, lse = _outputs(w, d["q"])
    assert _noalloc(pkg, w, d, out, lse) == 0
    assert pkg.tsk_noalloc_status() == 0
    ro, rl, _ = oracle.run_workload(w)
    print(parity.compare(out.float().cpu().numpy().astype(np.float64),
                         lse.cpu().numpy().astype(np.float64), ro, rl, "after bad seqlens"))


def test_noalloc_rejects_problems_beyond_its_scratch(pkg):
    import torch
    q = torch.zeros((16, 4, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((16, 1, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    cu = torch.zeros(20000, dtype=torch.int32, device="cuda")
    # too many sequences
    rc = pkg.tsk_mha_prefill_noalloc(q, k, k, None, cu, 19999, 16, 4, 1, 64, 0, 0.125, o, None)
    assert rc == -2 and "scratch" in pkg.tsk_last_error()
    # too many query tiles: 49152 * 128 tokens (host-side check, nothing is read)
    rc = pkg.tsk_mha_prefill_noalloc(q, k, k, None, cu, 1, 49152 * 128, 4, 1, 64, 0, 0.125, o,
                                     None)
    assert rc == -2 and "scratch" in pkg.tsk_last_error()
