"""The allocation-free entry point, tsk_mha_prefill_noalloc.

It exists for callers that must not allocate device memory while they run
(for instance code inside a serving engine that has reserved the whole
device, or latency-critical paths where an allocation's implicit
synchronisation is not acceptable).  Its scratch is a fixed array inside the
library.  This file is collected last so that a failure here does not stop
the other GPU tests; it passes both on its own in a fresh process and after
them.
"""
import numpy as np
import pytest

import inputgen
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


def test_noalloc_matches_the_allocating_entry_point_twice(pkg):
    import torch
    # two different problems in a row: the second call must not see the first's scratch
    for seed, lens, window in [(31, [300, 1, 4096, 129], 0), (32, [2048, 77, 515], 128)]:
        w = inputgen.make(lens, 16, 2, window=window, seed=seed)
        d = parity.to_device(w)
        ref_out, ref_lse = parity.run_gpu(w, d)
        for call in range(2):
            out, lse = _outputs(w, d["q"])
            rc = pkg.tsk_mha_prefill_noalloc(d["q"], d["k"], d["v"], d["sinks"], d["cu"],
                                             w.num_seqs, w.total_tokens, w.Hq, w.Hkv, w.D,
                                             w.window, w.scale, out, lse)
            assert rc == 0, f"{pkg.STATUS.get(rc, rc)} {pkg.tsk_last_error()}"
            torch.cuda.synchronize()
            o = out.float().cpu().numpy().astype(np.float64)
            l = lse.cpu().numpy().astype(np.float64)
            r = ref_out.float().cpu().numpy().astype(np.float64)
            rl = ref_lse.cpu().numpy().astype(np.float64)
            print(parity.compare(o, l, r, rl, f"noalloc seed {seed} call {call}"))


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
