"""Pins for the CPU oracle, against facts fixed by the cited sources and by mathematics.

Each check below would fail on a plausible mistake in ``oracle/blasst_oracle.c``
(``test_oracle_mutants.py`` plants such mistakes and confirms it):

1. factor = 0 is dense softmax attention (the "Skip-Softmax" design doc,
   "From configuration to the kernel threshold": threshold 0 skips no tiles;
   "Algorithm": the dense pass returns O / l exactly). Compared with a
   textbook, materialised softmax written separately.
2. Closed form of the mask: for lambda <= 1 a skipped tile never raises the
   running max, so running_max before tile j is the dense prefix maximum and
   skip_j = [max_i (tile_max_j[i] - M_{j-1}[i]) < ln(lambda)]. Scores for this
   check come from numpy, not from the oracle.
3. Monotone skip sets in lambda (follows from 2).
4. Hand-built cases with exactly representable scores skip exactly the
   predicted tiles and have closed-form outputs (tests/hand_built.py and its golden
   files): the all-rows rule, a query tail, a gap of exactly ln(lambda) = 0 (the test
   is strict), and lambda > 1 with a skipped tile above the running max (a skipped
   tile does not move it).
5. The output error stays within the bound implied by the skipped mass:
   |O_skip - O_dense| <= delta * (max_k v - min_k v) per column, and
   delta < lambda * (number of skipped keys in the row)
   ("Algorithm": exp(tile_max - running_max) bounds every key weight of the tile).
"""
import math

import numpy as np
import pytest

import oracle
import synth
from tests import hand_built


def random_bf16(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return synth.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def as_f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def scores_np(q, k, scale):
    """[B, H, Sq, Sk] fp64 scores from numpy (independent of the oracle's loops)."""
    qf = as_f64(q).transpose(0, 2, 1, 3)
    kf = as_f64(k).transpose(0, 2, 1, 3)
    return scale * np.einsum("bhqd,bhkd->bhqk", qf, kf)


def oracle_rows(res, units, Sq, tile_q):
    """Scatter per-unit oracle outputs to [B, H, Sq, d] / [B, H, Sq]."""
    o, lse = res["o"], res["lse"]
    units = np.asarray(units)
    B = units[:, 0].max() + 1
    H = units[:, 1].max() + 1
    d = o.shape[2]
    O = np.full((B, H, Sq, d), np.nan)
    L = np.full((B, H, Sq), np.nan)
    for u, (b, h, qt) in enumerate(units):
        r0 = qt * tile_q
        n = min(tile_q, Sq - r0)
        O[b, h, r0:r0 + n] = o[u, :n]
        L[b, h, r0:r0 + n] = lse[u, :n]
    return O, L


SMALL_CASES = [
    # (B, H, Sq, Sk, d, tile_q, tile_k, seed)
    (1, 1, 16, 16, 8, 4, 4, 1),
    (2, 3, 37, 300, 16, 16, 32, 2),     # ragged query and key tails, d != 128
    (1, 2, 64, 129, 32, 32, 64, 3),     # one valid key in the last tile
    (1, 1, 1, 1, 4, 128, 128, 4),       # a single query against a single key
]


@pytest.mark.parametrize("B,H,Sq,Sk,d,tq,tk,seed", SMALL_CASES)
def test_factor_zero_is_dense_attention(B, H, Sq, Sk, d, tq, tk, seed):
    q = random_bf16((B, Sq, H, d), seed, 1.5)
    k = random_bf16((B, Sk, H, d), seed + 100, 1.5)
    v = random_bf16((B, Sk, H, d), seed + 200)
    scale = 1.0 / math.sqrt(d)
    units = oracle.all_units(B, H, Sq, tq)
    res = oracle.skip_softmax_attn(q, k, v, scale, 0.0, units=units, tile_q=tq, tile_k=tk)
    assert res["mask"].sum() == 0
    O, L = oracle_rows(res, units, Sq, tq)
    rows = np.array([(b, h, s) for b in range(B) for h in range(H) for s in range(Sq)])
    od, ld = oracle.dense_attn(q, k, v, scale, rows)
    np.testing.assert_allclose(O.reshape(-1, d), od, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L.reshape(-1), ld, rtol=1e-13, atol=1e-12)
    # and the materialised definition, once more through numpy
    S = scores_np(q, k, scale)
    P = np.exp(S - S.max(-1, keepdims=True))
    ref = np.einsum("bhqk,bhkd->bhqd", P / P.sum(-1, keepdims=True), as_f64(v).transpose(0, 2, 1, 3))
    np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)


def test_factor_zero_is_dense_attention_tiny_workload():
    w = synth.WORKLOADS["tiny_1024"]
    q, k, v = synth.make_qkv(w)
    scale = 1.0 / math.sqrt(w.d)
    units = oracle.all_units(w.B, w.H, w.S)
    res = oracle.skip_softmax_attn(q, k, v, scale, 0.0, units=units, threads=8)
    assert res["mask"].sum() == 0
    O, L = oracle_rows(res, units, w.S, 128)
    rows = np.array([(0, h, s) for h in range(w.H) for s in range(0, w.S, 7)])
    od, ld = oracle.dense_attn(q, k, v, scale, rows, threads=8)
    np.testing.assert_allclose(O[rows[:, 0], rows[:, 1], rows[:, 2]], od, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L[rows[:, 0], rows[:, 1], rows[:, 2]], ld, rtol=1e-13, atol=1e-12)


def closed_form_gaps(q, k, scale, tile_q, tile_k):
    """Per (b, h, qt, j): max over valid rows of tile_max_j - (dense prefix max before j)."""
    S = scores_np(q, k, scale)
    B, H, Sq, Sk = S.shape
    nQ, nK = -(-Sq // tile_q), -(-Sk // tile_k)
    tm = np.stack([S[..., j * tile_k:min(Sk, (j + 1) * tile_k)].max(-1) for j in range(nK)], -1)
    prefix = np.concatenate([np.full(tm.shape[:-1] + (1,), -np.inf),
                             np.maximum.accumulate(tm, axis=-1)[..., :-1]], -1)
    g = tm - prefix  # [B, H, Sq, nK]
    out = np.empty((B, H, nQ, nK))
    for qt in range(nQ):
        out[:, :, qt] = g[:, :, qt * tile_q:min(Sq, (qt + 1) * tile_q)].max(2)
    return out


CLOSED_FORM_CASES = [
    # (B, H, Sq, Sk, d, tile_q, tile_k, seed, factors)  -- Sq != Sk pins the lambda denominator
    (1, 2, 96, 320, 16, 32, 32, 5, (0.0, 0.5, 2.0, 8.0, 32.0, 128.0)),
    (2, 1, 150, 61, 8, 64, 8, 6, (0.0, 0.25, 1.0, 4.0, 16.0)),
]


@pytest.mark.parametrize("B,H,Sq,Sk,d,tq,tk,seed,factors", CLOSED_FORM_CASES)
def test_mask_matches_prefix_max_closed_form(B, H, Sq, Sk, d, tq, tk, seed, factors):
    # clustered keys so that the gaps spread over several units of ln(lambda)
    rng = np.random.default_rng(seed)
    centres = rng.standard_normal((4, d)) * 3.0
    qf = centres[rng.integers(0, 4, (B, Sq, H))] + rng.standard_normal((B, Sq, H, d))
    kf = centres[rng.integers(0, 4, (B, Sk, H))] + rng.standard_normal((B, Sk, H, d))
    q = synth.f32_to_bf16_bits(qf.astype(np.float32))
    k = synth.f32_to_bf16_bits(kf.astype(np.float32))
    v = random_bf16((B, Sk, H, d), seed + 7)
    scale = 1.0 / math.sqrt(d)
    expect_gap = closed_form_gaps(q, k, scale, tq, tk)
    units = oracle.all_units(B, H, Sq, tq)
    nQ, nK = -(-Sq // tq), -(-Sk // tk)
    seen_skip = 0
    for f in factors:
        lam = f / Sk
        assert lam <= 1.0
        res = oracle.skip_softmax_attn(q, k, v, scale, f, units=units, tile_q=tq, tile_k=tk)
        gap = res["gap"].reshape(B, H, nQ, nK)
        mask = res["mask"].reshape(B, H, nQ, nK)
        np.testing.assert_allclose(gap, expect_gap, rtol=0, atol=1e-9)
        ln_lam = math.log(lam) if f > 0 else -math.inf
        assert np.all(np.abs(expect_gap - ln_lam) > 1e-6), "a tile sits on the threshold; pick another seed"
        np.testing.assert_array_equal(mask, (expect_gap < ln_lam).astype(np.uint8))
        seen_skip += mask.sum()
    assert seen_skip > 0


def _factor_grid(Sk):
    return [0.0] + [2.0 ** e for e in range(-4, 8)]


@pytest.mark.parametrize("name,S,H", [("tiny_1024", 1024, 2), ("dit_8192_g2", 2048, 2), ("dit_8192_g1", 2048, 2)])
def test_skip_set_monotone_in_lambda(name, S, H):
    w = synth.WORKLOADS[name]
    q, k, v = synth.make_qkv(w, Sq=S, Sk=S)
    q, k, v = (np.ascontiguousarray(x[:, :, :H]) for x in (q, k, v))
    scale = 1.0 / math.sqrt(w.d)
    prev = None
    counts = []
    for f in _factor_grid(S):
        assert f / S <= 1.0
        res = oracle.skip_softmax_attn(q, k, v, scale, f, threads=8)
        m = res["mask"].astype(bool)
        if prev is not None:
            assert not np.any(prev & ~m), "a tile skipped at a smaller lambda is kept at a larger one"
        counts.append(int(m.sum()))
        prev = m
    assert counts == sorted(counts)
    assert counts[0] == 0


def _load_golden():
    return hand_built.load_cases()


@pytest.mark.parametrize("case", _load_golden(), ids=hand_built.case_id)
def test_hand_built_case_skips_predicted_tiles(case):
    """Masks (and the recorded gaps) of the hand-built cases, and their closed-form outputs.

    The "above_one" construction has lambda > 1: a skipped tile whose maximum exceeds the
    running max must leave it unchanged, which decides the next tile."""
    name, c = case
    q, k, v, vv = hand_built.build(name, c["Sq"])
    res = oracle.skip_softmax_attn(q, k, v, hand_built.SCALE, hand_built.factor_of(c))
    assert res["mask"][0].tolist() == c["mask"]
    if "gap" in c:
        expect = [float(x) for x in c["gap"]]
        np.testing.assert_allclose(res["gap"][0], expect, rtol=0, atol=1e-12)
    expected = hand_built.closed_form(name, c, vv)
    if expected is not None:
        o_ref, lse_ref = expected
        np.testing.assert_allclose(res["o"][0, :c["Sq"]], o_ref, rtol=0, atol=1e-13)
        np.testing.assert_allclose(res["lse"][0, :c["Sq"]], lse_ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("name,S,H,factors", [
    ("tiny_1024", 1024, 2, (0.5, 2.0, 8.0)),
    ("dit_8192_g1", 1024, 2, (1.0, 4.0, 16.0, 64.0)),
])
def test_output_error_within_skipped_mass_bound(name, S, H, factors):
    w = synth.WORKLOADS[name]
    q, k, v = synth.make_qkv(w, Sq=S, Sk=S)
    q, k, v = (np.ascontiguousarray(x[:, :, :H]) for x in (q, k, v))
    scale = 1.0 / math.sqrt(w.d)
    Sfull = scores_np(q, k, scale)[0]                   # [H, S, S]
    W = np.exp(Sfull - Sfull.max(-1, keepdims=True))     # dense weights, max weight 1
    vf = as_f64(v)[0].transpose(1, 0, 2)                 # [H, S, d]
    dense = np.einsum("hqk,hkd->hqd", W / W.sum(-1, keepdims=True), vf)
    vrange = vf.max(1) - vf.min(1)                       # [H, d]
    units = oracle.all_units(1, H, S)
    nK = S // 128
    any_skip = False
    for f in factors:
        lam = f / S
        res = oracle.skip_softmax_attn(q, k, v, scale, f, units=units, threads=8)
        O, _ = oracle_rows(res, units, S, 128)
        O = O[0]
        mask = res["mask"].reshape(H, S // 128, nK)
        any_skip |= bool(mask.any())
        # per-row skipped-key indicator
        skipped = np.repeat(np.repeat(mask, 128, axis=1), 128, axis=2).astype(bool)  # [H, S, S]
        delta = (W * skipped).sum(-1) / W.sum(-1)                                  # [H, S]
        err = np.abs(O - dense)
        assert np.all(err <= delta[..., None] * vrange[:, None, :] + 1e-12)
        n_skipped = skipped.sum(-1)
        assert np.all(delta <= lam * n_skipped + 1e-15)
    assert any_skip


@pytest.mark.parametrize("factor", [0.0, 20.0, 100.0])
def test_max_prob_is_the_largest_kept_softmax_weight(factor):
    """'video-attention' blog, 'max_prob = 1 / l_i': the row's largest softmax weight."""
    B, H, Sq, Sk, d, tq, tk = 1, 2, 70, 200, 16, 32, 32
    rng = np.random.default_rng(12)
    centres = rng.standard_normal((3, d)) * 4.0
    q = synth.f32_to_bf16_bits((centres[rng.integers(0, 3, (B, Sq, H))] + rng.standard_normal((B, Sq, H, d))).astype(np.float32))
    # keys grouped by centre along the sequence, so whole key tiles fall far below a row's max
    k = synth.f32_to_bf16_bits((centres[(np.arange(Sk) // 40) % 3][None, :, None, :] + rng.standard_normal((B, Sk, H, d))).astype(np.float32))
    v = random_bf16((B, Sk, H, d), 13)
    scale = 1.0 / math.sqrt(d)
    units = oracle.all_units(B, H, Sq, tq)
    res = oracle.skip_softmax_attn(q, k, v, scale, factor, units=units, tile_q=tq, tile_k=tk)
    S = scores_np(q, k, scale)[0]
    nK = -(-Sk // tk)
    if factor > 0:
        assert res["mask"].sum() > 0
    for u, (b, h, qt) in enumerate(units):
        for i in range(min(tq, Sq - qt * tq)):
            kept = np.concatenate([np.arange(j * tk, min(Sk, (j + 1) * tk)) for j in range(nK) if not res["mask"][u, j]])
            s = S[h, qt * tq + i, kept]
            w = np.exp(s - s.max())
            assert res["max_prob"][u, i] == pytest.approx((w / w.sum()).max(), rel=1e-12)
