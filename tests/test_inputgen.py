"""Seeded input generator (no GPU)."""
import numpy as np
import pytest

import inputgen


def test_deterministic_and_slice_independent():
    a = inputgen.normal_bf16(7, inputgen.STREAM_Q, (1000,))
    b = inputgen.normal_bf16(7, inputgen.STREAM_Q, (1000,))
    assert np.array_equal(a, b)
    big = inputgen.normal_bf16(7, inputgen.STREAM_Q, (300000,))  # threaded path
    assert np.array_equal(big[:1000], a)
    c = inputgen.normal_bf16(8, inputgen.STREAM_Q, (1000,))
    d = inputgen.normal_bf16(7, inputgen.STREAM_K, (1000,))
    assert not np.array_equal(a, c) and not np.array_equal(a, d)


def test_normal_statistics():
    x = inputgen.normal_f32(1, 2, (400000,))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    y = inputgen.normal_f32(1, 2, (400000,), sigma=2.0)
    assert np.allclose(y, 2.0 * x)
    # fraction within one sigma of a normal: 0.6827
    assert abs((np.abs(x) < 1).mean() - 0.6827) < 0.005


def test_bf16_rounding_matches_round_to_nearest_even():
    f = inputgen.normal_f32(3, 9, (100000,))
    bits = inputgen.normal_bf16(3, 9, (100000,))
    assert np.array_equal(bits, inputgen.f32_to_bf16_bits(f))
    back = inputgen.bf16_bits_to_f32(bits)
    # nearest: error at most half an ulp of bf16 (8 significant bits)
    rel = np.abs(back - f) / np.maximum(np.abs(f), 1e-30)
    assert rel.max() <= 2.0 ** -8 + 1e-7
    # ties go to even
    tie = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8], np.float32)
    assert list(inputgen.f32_to_bf16_bits(tie)) == [0x3F80, 0x3F82]


def test_k_multiplier_applied_in_fp32_then_rounded():
    f = inputgen.normal_f32(5, inputgen.STREAM_K, (5000,))
    bits = inputgen.normal_bf16(5, inputgen.STREAM_K, (5000,), 3.0)
    assert np.array_equal(bits, inputgen.f32_to_bf16_bits(f * np.float32(3.0)))


def test_uniform_int_bounds_and_coverage():
    r = inputgen.uniform_int(0, 5, 200000, 512, 8192)
    assert r.min() == 512 and r.max() == 8192
    assert abs(r.mean() - (512 + 8192) / 2) < 30
    small = inputgen.uniform_int(0, 5, 10000, 0, 2)
    assert set(np.unique(small)) == {0, 1, 2}


def test_configs_shapes():
    w = inputgen.config("tiny_1x256_h4kv1")
    assert w.q.shape == (256, 4, 64) and w.k.shape == (256, 1, 64) and w.sinks.shape == (4,)
    assert w.allowed_keys() == 256 * 257 // 2
    lens = inputgen.ragged_lengths(0)
    assert len(lens) == 32 and min(lens) >= 512 and max(lens) <= 8192
    assert inputgen.ragged_lengths(0) == lens


def test_sample_rows_cover_structure():
    w = inputgen.make([300, 1, 129], 8, 2, D=8, window=128, seed=1)
    t, h = inputgen.sample_rows(w, n_target=200)
    rows = set(zip(t.tolist(), h.tolist()))
    toks = set(t.tolist())
    for s, L in enumerate(w.seqlens):
        st = int(w.cu_seqlens[s])
        assert st in toks and st + L - 1 in toks
    assert {127, 128, 255, 256}.issubset(toks)
    assert set(h.tolist()) == set(range(8))
    assert len(rows) == len(t) >= 200


def test_e4m3_decode_matches_torch():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    mine = inputgen.e4m3_to_f32(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(mine)
    assert np.array_equal(mine[ok], ref[ok])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne():
    torch = pytest.importorskip("torch")
    vals = inputgen.e4m3_to_f32(np.arange(256, dtype=np.uint8))
    vals = np.unique(vals[~np.isnan(vals)])
    mids = (vals[:-1] + vals[1:]) / 2          # ties: round to even
    x = np.concatenate([inputgen.normal_f32(3, 77, (100000,), 40.0), vals, mids]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(inputgen.f32_to_e4m3(x), ref)
    assert inputgen.f32_to_e4m3(np.array([1e6, -1e6], np.float32)).tolist() == [0x7E, 0xFE]


def test_fp8_workload_dequantizes_exactly_in_bf16():
    w = inputgen.make_fp8([100, 37], 4, 2, seed=5)
    for name in ("q", "k", "v"):
        exact = inputgen.e4m3_to_f32(w.fp8[name]) * np.float32(w.fp8[name + "_scale"])
        assert np.array_equal(inputgen.bf16_bits_to_f32(getattr(w, name)), exact)
        assert np.log2(w.fp8[name + "_scale"]) == np.round(np.log2(w.fp8[name + "_scale"]))
