"""The entry points under CUDA graph capture.

Once a stream's workspace is warm (one eager call on that stream with a
problem at least as large), a call enqueues only kernel launches, so it can
be captured into a CUDA graph and replayed; a replay reads whatever the
input buffers hold at that time.  Each test compares replays bit for bit
with eager calls on the same inputs (the kernels are deterministic), before
and after the inputs are overwritten in place.
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


def _same(a, b):
    import torch
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a, b)


def _capture(fn, stream):
    """Warms `fn` up on `stream`, then captures one call of it."""
    import torch
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def _check_replays(pkg, fn, outs, refill, stream):
    """Eager results, graph replay, refilled inputs, replay again."""
    import torch
    g = _capture(fn, stream)
    for round_ in range(2):
        if round_ == 1:
            refill()
            torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        want = [o.clone() for o in outs]
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for o, r in zip(outs, want):
            assert _same(o, r), f"replay differs from the eager call (round {round_})"
    assert pkg.tsk_get_device_status(stream) == 0


def _refill_from(dst, w_new, key):
    d = parity.to_device(w_new)
    dst.copy_(d[key])


def test_prefill_graph_replay(pkg):
    import torch
    w = inputgen.make([300, 1, 2048, 129], 16, 2, window=0, seed=41)
    d = parity.to_device(w)
    out = torch.empty((w.total_tokens, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.total_tokens, w.Hq), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def call():
        rc = pkg.tsk_mha_prefill(d["q"], d["k"], d["v"], d["sinks"], d["cu"], w.num_seqs,
                                 w.total_tokens, w.Hq, w.Hkv, w.D, w.window, w.scale, out, lse)
        assert rc == 0, f"{pkg.STATUS.get(rc, rc)} {pkg.tsk_last_error()}"

    w2 = inputgen.make([300, 1, 2048, 129], 16, 2, window=0, seed=42)

    def refill():
        for key in ("q", "k", "v"):
            _refill_from(d[key], w2, key)

    _check_replays(pkg, call, [out, lse], refill, s)


def test_two_calls_in_one_graph(pkg):
    """Two problems (full causal, then a window of 128 with head dimension
    128) captured back to back in one graph."""
    import torch
    wa = inputgen.make([1000, 77], 8, 2, seed=43)
    wb = inputgen.make([640, 300], 8, 4, D=128, window=128, seed=44)
    da, db = parity.to_device(wa), parity.to_device(wb)
    oa = torch.empty((wa.total_tokens, wa.Hq, wa.D), dtype=torch.bfloat16, device="cuda")
    ob = torch.empty((wb.total_tokens, wb.Hq, wb.D), dtype=torch.bfloat16, device="cuda")
    la = torch.empty((wa.total_tokens, wa.Hq), dtype=torch.float32, device="cuda")
    lb = torch.empty((wb.total_tokens, wb.Hq), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def call():
        for w, d, o, l in ((wa, da, oa, la), (wb, db, ob, lb)):
            rc = pkg.tsk_mha_prefill(d["q"], d["k"], d["v"], d["sinks"], d["cu"], w.num_seqs,
                                     w.total_tokens, w.Hq, w.Hkv, w.D, w.window, w.scale, o, l)
            assert rc == 0, f"{pkg.STATUS.get(rc, rc)} {pkg.tsk_last_error()}"

    wb2 = inputgen.make([640, 300], 8, 4, D=128, window=128, seed=45)

    def refill():
        _refill_from(db["q"], wb2, "q")

    _check_replays(pkg, call, [oa, la, ob, lb], refill, s)


def test_noalloc_graph_replay(pkg):
    import torch
    w = inputgen.make([129, 4096], 16, 2, window=128, seed=46)
    d = parity.to_device(w)
    out = torch.empty((w.total_tokens, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.total_tokens, w.Hq), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def call():
        rc = pkg.tsk_mha_prefill_noalloc(d["q"], d["k"], d["v"], d["sinks"], d["cu"],
                                         w.num_seqs, w.total_tokens, w.Hq, w.Hkv, w.D,
                                         w.window, w.scale, out, lse)
        assert rc == 0, f"{pkg.STATUS.get(rc, rc)} {pkg.tsk_last_error()}"

    w2 = inputgen.make([129, 4096], 16, 2, window=128, seed=47)

    def refill():
        _refill_from(d["k"], w2, "k")

    _check_replays(pkg, call, [out, lse], refill, s)


def test_decode_graph_replay(pkg):
    import torch
    w = inputgen.make_kvcache([1] * 5, [1, 129, 3000, 700, 20000], 16, 2, seed=48)
    d = parity.to_device(w)
    out = torch.empty((w.num_seqs, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.num_seqs, w.Hq), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def call():
        rc = pkg.tsk_mha_decode_kvcache(d["q"], d["k"], d["v"], d["sinks"], d["cu_k"],
                                        w.num_seqs, w.total_keys, max(w.seqlens_k), w.Hq,
                                        w.Hkv, w.D, w.window, w.scale, out, lse)
        assert rc == 0, f"{pkg.STATUS.get(rc, rc)} {pkg.tsk_last_error()}"

    w2 = inputgen.make_kvcache([1] * 5, [1, 129, 3000, 700, 20000], 16, 2, seed=49)

    def refill():
        _refill_from(d["q"], w2, "q")
        _refill_from(d["v"], w2, "v")

    _check_replays(pkg, call, [out, lse], refill, s)


def test_fp8_graph_replay(pkg):
    import torch
    w = inputgen.make_fp8([257, 1500], 16, 2, seed=50)
    d = parity.to_device(w)
    f = w.fp8
    q8, k8, v8 = (torch.from_numpy(np.ascontiguousarray(f[n])).to("cuda") for n in ("q", "k", "v"))
    out = torch.empty((w.total_tokens, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.total_tokens, w.Hq), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def call():
        rc = pkg.tsk_mha_prefill_fp8(q8, k8, v8, f["q_scale"], f["k_scale"], f["v_scale"], d["sinks"],
                                     d["cu"], w.num_seqs, w.total_tokens, w.Hq, w.Hkv, w.D,
                                     w.window, w.scale, out, lse)
        assert rc == 0, f"{pkg.STATUS.get(rc, rc)} {pkg.tsk_last_error()}"

    w2 = inputgen.make_fp8([257, 1500], 16, 2, seed=51)

    def refill():
        v8.copy_(torch.from_numpy(np.ascontiguousarray(w2.fp8["v"])).to("cuda"))

    _check_replays(pkg, call, [out, lse], refill, s)
