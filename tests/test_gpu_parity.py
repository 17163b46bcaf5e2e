"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every workload of the benchmark table runs at its full size in the same launch
configuration the benchmark times. The oracle checks every query tile of three or
more whole heads per workload (heads 0, H/2 and H - 1; for the long workload also
the heads of the smallest and largest clustering weight; both batch entries of
the ragged one), plus sampled units at every factor, and properties that hold at
any size are checked everywhere:
skip counts equal the mask popcount, factor 0 skips nothing, the first key tile
is never skipped, and skip sets grow with lambda (lambda <= 1).
"""
import math

import numpy as np
import pytest

import synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import softmax_threshold_tile_gb300 as blasst
    blasst.build_library()
    blasst.load_library()
    yield
    torch.cuda.synchronize()


def _run_workload_sweep(w, factors, units, whole=()):
    """Run `w` at full size at every factor and compare with the oracle.

    units: sampled (b, h, query tile) units compared at every factor.
    whole: (b, h) pairs compared on EVERY query tile at factor 0 and at the largest factor
    (outputs, lse and decisions, the oracle replaying the GPU's decisions); the decisions of
    every other factor on those heads are then checked against the gap chain of the largest
    factor's replay (for lambda <= 1 the running max is the dense prefix max at any factor)."""
    q, k, v = synth.make_qkv(w)
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    fmax = max(factors)
    prev_mask = None
    stats = []
    head_masks = {}
    gaps = {}
    whole_stats = {"units": 0, "decisions": 0, "differ": 0, "max_abs": 0.0, "mean_abs": 0.0}
    for f in sorted(factors):
        o, lse, counts, mask = parity.run_gpu(qd, kd, vd, f)
        parity.check_counts(counts, mask, f)
        if prev_mask is not None and f / w.S <= 1.0:
            assert not np.any(prev_mask.astype(bool) & ~mask.astype(bool)), "skip set shrank as lambda grew"
        prev_mask = mask
        st = parity.compare_units(q, k, v, o, lse, mask, f, units)
        st["factor"] = f
        st["skip_fraction"] = float(mask.mean())
        stats.append(st)
        for b, h in whole:
            head_masks[(f, b, h)] = mask[b, h].copy()
            if f not in (0.0, fmax):
                continue
            sw = parity.compare_units(q, k, v, o, lse, mask, f, parity.whole_head_units(b, h, w.S),
                                      return_gap=True)
            if f == fmax:
                gaps[(b, h)] = sw["gap"]
            whole_stats["units"] += len(parity.whole_head_units(b, h, w.S))
            whole_stats["decisions"] += sw["decisions"]
            whole_stats["differ"] += sw["differ"]
            whole_stats["max_abs"] = max(whole_stats["max_abs"], sw["max_abs"])
            whole_stats["mean_abs"] = max(whole_stats["mean_abs"], sw["mean_abs"])
        del o, lse
    for (f, b, h), m in head_masks.items():
        if f in (0.0, fmax) or f / w.S > 1.0:
            continue
        n, differ = parity.check_decisions(gaps[(b, h)], m, f, w.S)
        whole_stats["decisions"] += n
        whole_stats["differ"] += differ
    print(w.name, stats)
    if whole:
        print(w.name, "whole heads", sorted(whole), whole_stats)
    return stats


def test_tiny_1024_every_unit():
    w = synth.WORKLOADS["tiny_1024"]
    units = parity.sample_units(w.B, w.H, w.S, heads=range(w.H), qtiles=range(w.S // 128))
    stats = _run_workload_sweep(w, w.factors, units)
    assert stats[0]["skipped"] == 0
    assert stats[-1]["skipped"] > 0


@pytest.mark.parametrize("Sq,Sk", [(1, 1), (127, 127), (129, 129), (255, 255), (1000, 1000),
                                   (300, 1000), (1000, 129), (128, 8), (8, 1000)])
@pytest.mark.parametrize("factor", [0.0, 0.5, 4.0])
def test_odd_shapes(Sq, Sk, factor):
    q, k, v = parity.clustered_inputs(2, 3, Sq, Sk, seed=Sq * 7 + Sk)
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    o, lse, counts, mask = parity.run_gpu(qd, kd, vd, factor)
    parity.check_counts(counts, mask, factor)
    units = parity.sample_units(2, 3, Sq, heads=range(3), qtiles=range(-(-Sq // 128)))
    parity.compare_units(q, k, v, o, lse, mask, factor, units)


def test_large_factor_lambda_above_one():
    """lambda > 1 is allowed and computed literally (the decision is still the design doc's test)."""
    q, k, v = parity.clustered_inputs(1, 2, 512, 512, seed=11)
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    f = 2048.0  # lambda = 4
    o, lse, counts, mask = parity.run_gpu(qd, kd, vd, f)
    parity.check_counts(counts, mask, f)
    units = parity.sample_units(1, 2, 512, heads=range(2), qtiles=range(4))
    parity.compare_units(q, k, v, o, lse, mask, f, units)


@pytest.mark.parametrize("name", ["dit_8192_g1", "dit_8192_g2", "dit_8192_g3"])
def test_dit_8192(name):
    w = synth.WORKLOADS[name]
    units = parity.sample_units(w.B, w.H, w.S, heads=(0, 11, 23), qtiles=(0, 1, 31, 63))
    stats = _run_workload_sweep(w, w.factors, units, whole=[(0, h) for h in (0, 11, 23)])
    assert stats[0]["skipped"] == 0


def test_wan_32760():
    w = synth.WORKLOADS["wan_32760"]
    units = parity.sample_units(w.B, w.H, w.S, heads=(0, 20, 39), qtiles=(0, 1, 128, 255))
    stats = _run_workload_sweep(w, w.factors, units, whole=[(0, h) for h in (0, 20, 39)])
    assert stats[-1]["skip_fraction"] > 0


def test_long_65536():
    w = synth.WORKLOADS["long_65536"]
    g = w.gammas()
    heads = (0, 12, 23, int(np.argmin(g)), int(np.argmax(g)))
    units = parity.sample_units(w.B, w.H, w.S, heads=heads, qtiles=(0, 255, 511))
    _run_workload_sweep(w, w.factors, units, whole=[(0, h) for h in sorted(set(heads))])


def test_ragged_37000():
    w = synth.WORKLOADS["ragged_37000"]
    a, b, ts = w.curve
    factors = [0.0] + [a * math.exp(b * t) for t in ts]
    units = parity.sample_units(w.B, w.H, w.S, heads=(0, 16, 31), qtiles=(0, 144, 289))
    stats = _run_workload_sweep(w, factors, units, whole=[(b, h) for b in range(w.B) for h in (0, 16, 31)])
    assert stats[-1]["skip_fraction"] > 0


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes(seed):
    """Seeded random shapes (batch, heads, ragged Sq != Sk, clustering strength, factor), every
    query tile checked against the oracle."""
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 4))
    H = int(rng.integers(1, 6))
    Sq = int(rng.integers(1, 900))
    Sk = int(rng.integers(1, 1400))
    gamma = float(rng.uniform(0.0, 3.0))
    factor = float(rng.choice([0.0, 0.25, 2.0, 16.0, 128.0]))
    g = np.full(B * H, gamma)
    q = synth.fill(1, B, Sq, H, 128, seed, (1, 1, Sq), (1, 1, 16), g)
    k = synth.fill(2, B, Sk, H, 128, seed, (1, 1, Sk), (1, 1, 16), g)
    v = synth.fill(3, B, Sk, H, 128, seed)
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    o, lse, counts, mask = parity.run_gpu(qd, kd, vd, factor)
    parity.check_counts(counts, mask, factor)
    units = parity.sample_units(B, H, Sq, heads=range(H), qtiles=range(-(-Sq // 128)))
    st = parity.compare_units(q, k, v, o, lse, mask, factor, units)
    print(dict(B=B, H=H, Sq=Sq, Sk=Sk, gamma=round(gamma, 2), factor=factor), st)
