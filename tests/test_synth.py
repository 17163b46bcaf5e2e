"""The shared input generator: determinism, threading independence, grid cells, bf16 rounding."""
import math

import numpy as np
import pytest

import synth


def test_bf16_round_to_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 65504.0, 1e-40, 3.0e38], np.float32)
    bits = synth.f32_to_bf16_bits(vals)
    back = synth.bf16_bits_to_f32(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa wins (1.0)
    assert back[0] == 1.0 and back[1] == 1.0
    # 1 + 3*2^-8 is a tie between 1 + 2^-7 and 1 + 2^-6: even wins (1 + 2^-6)
    assert back[2] == 1.0 + 2 ** -6
    assert back[3] == -2.5
    lib = synth._load()
    for x in vals:
        assert lib.synth_f32_to_bf16(float(x)) == synth.f32_to_bf16_bits(np.array([x], np.float32))[0]


def test_generator_deterministic_and_thread_independent():
    w = synth.WORKLOADS["tiny_1024"]
    a = synth.make_qkv(w, threads=1)
    b = synth.make_qkv(w, threads=7)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    # a prefix of tokens is the same whatever the total length (counter-based)
    c = synth.make_qkv(w, Sq=300, Sk=300, threads=3)
    for x, y in zip(a, c):
        np.testing.assert_array_equal(x[:, :300], y)


def test_noise_statistics():
    v = synth.bf16_bits_to_f32(synth.fill(3, 1, 4096, 2, 128, seed=3)).astype(np.float64)
    assert abs(v.mean()) < 0.01
    assert abs(v.std() - 1.0) < 0.01


def test_cell_structure_of_clustered_tokens():
    w = synth.WORKLOADS["tiny_1024"]   # grid 4x16x16, cells 2x4x4
    q, k, _ = synth.make_qkv(w)
    qf = synth.bf16_bits_to_f32(q)[0, :, 0].astype(np.float64)
    kf = synth.bf16_bits_to_f32(k)[0, :, 0].astype(np.float64)

    def cell(s):
        t, y, x = s // 256, (s // 16) % 16, s % 16
        return (t // 2, y // 4, x // 4)

    same = [(a, b) for a, b in [(0, 1), (0, 17), (0, 256 + 3), (5, 54)] if cell(a) == cell(b)]
    diff = [(a, b) for a, b in [(0, 4), (0, 64), (0, 512), (700, 3)] if cell(a) != cell(b)]
    assert len(same) == 4 and len(diff) == 4
    # q.k within a cell is about gamma^2 * d = 512; across cells it is O(sqrt(d) * gamma^2)
    for a, b in same:
        assert qf[a] @ kf[b] > 250
    for a, b in diff:
        assert abs(qf[a] @ kf[b]) < 250


def test_per_head_gamma_draws():
    w = synth.WORKLOADS["long_65536"]
    g = w.gammas()
    assert g.shape == (24,)
    assert np.all((g >= 0.5) & (g < 3.0))
    assert len(set(np.round(g, 6))) == 24
    r = synth.WORKLOADS["ragged_37000"].gammas()
    assert np.all(r[:32] == 0.0) and np.all(r[32:] == 3.0)


def test_workload_grids_cover_their_tokens():
    for w in synth.WORKLOADS.values():
        T, Hg, W = w.grid
        assert T * Hg * W == w.S, w.name
        assert math.isfinite(w.dense_flops())


def test_e4m3_codes_follow_the_ocp_definition():
    # hand values of the OCP FP8 e4m3 format (bias 7, 3 mantissa bits, no infinities)
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x30: 0.5, 0x3C: 1.5, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0, 0x40: 2.0}
    for code, val in cases.items():
        assert synth.e4m3_bits_to_f32(np.array([code], np.uint8))[0] == np.float32(val)
        assert synth.f32_to_e4m3_bits(np.array([val], np.float32))[0] == code or val == 0.0
    assert np.isnan(synth.e4m3_bits_to_f32(np.array([0x7F, 0xFF], np.uint8))).all()
    # ties go to the even code; out-of-range values saturate
    x = np.array([2.0 ** -10, 3 * 2.0 ** -10, 1.0625, 1.1875, 1000.0, -1e9, 464.0], np.float32)
    np.testing.assert_array_equal(synth.f32_to_e4m3_bits(x), [0x00, 0x02, 0x38, 0x3A, 0x7E, 0xFE, 0x7E])


def test_e4m3_round_trip_and_bf16_exactness():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = synth.e4m3_bits_to_f32(codes)
    np.testing.assert_array_equal(synth.f32_to_e4m3_bits(vals)[vals != 0], codes[vals != 0])
    # every finite e4m3 value is a bf16 value, so the oracle can take e4m3 inputs as bf16 bits
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(vals)), vals)


def test_e4m3_matches_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = synth.e4m3_bits_to_f32(codes)
    np.testing.assert_array_equal(np.isnan(ref), np.isnan(got))
    np.testing.assert_array_equal(ref[~np.isnan(ref)], got[~np.isnan(got)])
    rng = np.random.default_rng(1)
    fin = np.sort(ref[np.isfinite(ref)])
    x = np.concatenate([rng.standard_normal(20000) * np.exp(rng.uniform(-12, 6, 20000)),
                        (fin[:-1] + fin[1:]) / 2]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    np.testing.assert_array_equal(synth.f32_to_e4m3_bits(x),
                                  torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_quantize_e4m3_per_tensor():
    q, _, _ = synth.make_qkv("tiny_1024")
    codes, descale = synth.quantize_e4m3(q)
    x = synth.bf16_bits_to_f32(q)
    assert abs(descale * 448.0 - np.abs(x).max()) <= 1e-6 * np.abs(x).max()
    back = synth.e4m3_bits_to_f32(codes) * descale
    # relative rounding error of e4m3 is at most 2^-4 for normal values
    big = np.abs(x) > 2.0 ** -6 * descale
    assert np.all(np.abs(back[big] - x[big]) <= 2.0 ** -4 * np.abs(x[big]) * (1 + 1e-6))
