"""The shared input generator: determinism, threading independence, grid cells, bf16 rounding."""
import math

import numpy as np

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
