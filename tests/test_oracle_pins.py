"""The CPU oracle against its pins (no GPU)."""
import os
import tempfile

import numpy as np
import pytest

import oracle
import oracle_pins as P


@pytest.fixture(scope="module")
def lib():
    return oracle._load()


@pytest.mark.parametrize("name", list(P.ALL_PINS))
def test_pin(lib, name):
    ok, detail = P.ALL_PINS[name](lib)
    assert ok, f"pin {name}: {detail}"


# Mistakes a plausible oracle could contain; each must be caught by >= 1 pin.
MUTANTS = {
    "gqa_modulo_mapping": ("g = h / G", "g = h % p->Hkv"),
    "sink_scaled": ("has_sink ? p->sinks[h] : -INFINITY", "has_sink ? p->scale * p->sinks[h] : -INFINITY"),
    "window_off_by_one": ("lo = t - p->window + 1;", "lo = t - p->window;"),
    "sink_dropped_from_Z": ("if (has_sink) Z += exp(sink - M);", ""),
    "lse_log2": ("*lse_out = M + log(Z);", "*lse_out = M + log2(Z);"),
    "value_reads_keys": ("const uint16_t *vr = p->v +", "const uint16_t *vr = p->k +"),
    "scale_missing": ("work[j] = p->scale * acc;", "work[j] = acc;"),
    "no_causal_bound_max_missing_sink": ("if (has_sink && sink > M) M = sink;", ""),
    "kvcache_top_left_alignment": ("p->cu_k[s] + (lk - lq) + (t - p->cu[s])", "p->cu_k[s] + (t - p->cu[s])"),
}


@pytest.mark.parametrize("mutant", list(MUTANTS))
def test_planted_mistakes_are_caught(mutant):
    old, new = MUTANTS[mutant]
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found: {old!r}"
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "mut.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        so = os.path.join(d, "libmut.so")
        import subprocess
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", so, path,
                               "-lm", "-lpthread"])
        res = P.run_all(oracle.load_variant(so))
    failed = [k for k, (ok, _) in res.items() if not ok]
    if mutant == "no_causal_bound_max_missing_sink":
        # Leaving the sink out of the running maximum is mathematically harmless
        # (the max only stabilises exp); pins must still pass except where the
        # sink dominates (big_sink), and nothing else may change.
        assert set(failed) <= {"big_sink"}, failed
        return
    assert failed, f"no pin caught mutant {mutant}"


def test_oracle_rejects_bad_problem():
    q = np.zeros((2, 2, 4), np.uint16)
    k = np.zeros((2, 1, 4), np.uint16)
    with pytest.raises(ValueError):
        oracle.mha_prefill(q, k, k, None, np.array([0, 2, 1], np.int32), 2, 1, 4, 0, 1.0)
    with pytest.raises(ValueError):  # Hq not a multiple of Hkv
        oracle.mha_prefill(q, np.zeros((2, 3, 4), np.uint16), np.zeros((2, 3, 4), np.uint16),
                           None, np.array([0, 2], np.int32), 2, 3, 4, 0, 1.0)


def test_oracle_threads_deterministic():
    w = P.small_workload(seed=21, window=0)
    o1, l1, _ = oracle.run_workload(w, nthreads=1)
    o2, l2, n = oracle.run_workload(w, nthreads=4)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_zero_length_sequences():
    w = P.small_workload(seed=22, seqlens=(0, 3, 0, 0, 5, 0))
    o, l, _ = oracle.run_workload(w)
    assert o.shape[0] == 8 and np.isfinite(o).all() and np.isfinite(l).all()
    ro, rl = P.sdpa_reference(w)
    assert np.abs(o - ro).max() < 1e-10 and np.abs(l - rl).max() < 1e-10
