"""Host-side controls (threshold -> factor, calibrated curve, timestep gate, dense steps,
flow-shift schedule): the C library against the golden MiniMax-H3 table printed in the
"Skip-Softmax" design doc ("Mapping the cutoff to denoising steps"), against the plain
oracle definitions, and against invariants of the formulas. No GPU needed."""
import json
import math
import os
import random
import warnings

import pytest

import oracle.host_control as ref
import softmax_threshold_tile_gb300 as blasst
from softmax_threshold_tile_gb300 import control

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "minimax_h3_schedule.json")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    blasst.build_library()
    blasst.load_library()


def golden():
    with open(GOLDEN) as fh:
        return json.load(fh)


@pytest.mark.parametrize("impl", ["library", "oracle"])
def test_minimax_h3_table(impl):
    g = golden()
    sched = (control.flow_shift_schedule if impl == "library" else ref.flow_shift_schedule)(g["shift"], g["sigma_points"])
    published = sched[:g["forwards"]]
    assert [round(x, 3) for x in published[:5]] == g["published_prefix_3dp"]
    count = control.dense_steps if impl == "library" else ref.dense_steps
    assert count(published, 0.9) == g["steps_above_0_9"]
    for row in g["table"]:
        d = count(published, row["disabled_until_timestep"])
        assert d == row["dense_steps"]
        assert len(published) - d == row["skip_softmax_steps"]


def test_schedule_endpoints_and_monotone():
    for s in (1.0, 3.0, 12.0):
        t = control.flow_shift_schedule(s, 11)
        assert t[0] == 1.0 and t[-1] == 0.0
        assert all(a > b for a, b in zip(t, t[1:]))
    # shift 1 is the identity on u
    assert control.flow_shift_schedule(1.0, 5) == pytest.approx([1.0, 0.75, 0.5, 0.25, 0.0], abs=0)


def test_threshold_control_makes_lambda_the_threshold():
    for thr in (0.0, 1e-4, 0.01, 0.5):
        for n in (1, 1024, 32760, 65536):
            f = control.factor_from_threshold(thr, n)
            assert f / n == pytest.approx(thr, rel=1e-15)
    assert control.factor_from_threshold(0.0, 32760) == 0.0  # threshold 0 skips nothing


def test_calibrated_curve_invariants():
    a, b = 2822.6209952221557, 4.388250623520793  # Wan2.2 transformer calibration (the design doc's example)
    assert control.factor_from_target_sparsity(a, b, 0.0) == a
    for s in (0.1, 0.5, 0.7):
        f0 = control.factor_from_target_sparsity(a, b, s)
        f1 = control.factor_from_target_sparsity(a, b, s + 1.0 / b)
        assert f1 / f0 == pytest.approx(math.e, rel=1e-12)
        assert control.factor_from_target_sparsity(a, b, s + 0.05) > f0
    # At the checkpoint's target sparsity 0.7 and Wan's 32760 tokens, lambda exceeds 1
    # (the operating point lies outside the (0, 1) range the doc calls meaningful).
    assert control.factor_from_target_sparsity(a, b, 0.7) / 32760 > 1.0


def test_gate_semantics():
    f = 123.0
    # sentinel 0: gate off, t never read
    assert control.gate_factor(f, 0.0, None) == (f, False)
    assert control.gate_factor(f, 0.0, 0.999) == (f, False)
    # positive cutoff: dense while t > cutoff, active once t <= cutoff
    assert control.gate_factor(f, 0.93, 0.95) == (0.0, False)
    assert control.gate_factor(f, 0.93, 0.93) == (f, False)
    assert control.gate_factor(f, 0.93, 0.5) == (f, False)
    # cutoff 1.0 on a publishing pipeline never gates (t is in [0, 1])
    assert all(control.gate_factor(f, 1.0, t)[0] == f for t in (1.0, 0.5, 0.0))
    # no published timestep: dense and warn
    assert control.gate_factor(f, 1.0, None) == (0.0, True)


def test_library_matches_oracle_definitions():
    rng = random.Random(7)
    for _ in range(200):
        thr, n = rng.uniform(0, 2), rng.randint(1, 10 ** 6)
        assert control.factor_from_threshold(thr, n) == ref.factor_from_threshold(thr, n)
        a, b, s = rng.uniform(0, 5000), rng.uniform(-5, 5), rng.uniform(0, 1)
        assert control.factor_from_target_sparsity(a, b, s) == pytest.approx(ref.factor_from_target_sparsity(a, b, s), rel=1e-15)
        d = rng.choice([0.0, rng.uniform(0, 1)])
        t = rng.choice([None, rng.uniform(0, 1)])
        assert control.gate_factor(a, d, t) == ref.gate_factor(a, d, t)
        ts = [rng.uniform(0, 1) for _ in range(rng.randint(0, 60))]
        assert control.dense_steps(ts, d) == ref.dense_steps(ts, d)
        sh, npts = rng.uniform(0.1, 20), rng.randint(2, 80)
        assert control.flow_shift_schedule(sh, npts) == pytest.approx(ref.flow_shift_schedule(sh, npts), rel=1e-15, abs=0)


@pytest.mark.parametrize("call", [
    lambda: control.factor_from_threshold(-0.1, 10),
    lambda: control.factor_from_threshold(float("nan"), 10),
    lambda: control.factor_from_threshold(0.1, 0),
    lambda: control.factor_from_target_sparsity(-1.0, 1.0, 0.5),
    lambda: control.factor_from_target_sparsity(1.0, float("inf"), 0.5),
    lambda: control.gate_factor(-1.0, 0.5, 0.1),
    lambda: control.gate_factor(1.0, -0.5, 0.1),
    lambda: control.gate_factor(1.0, 0.5, float("nan")),
    lambda: control.flow_shift_schedule(0.0, 10),
    lambda: control.flow_shift_schedule(3.0, 1),
])
def test_invalid_arguments(call):
    with pytest.raises(blasst.BlasstError):
        call()


def test_config_validation_and_single_warning():
    with pytest.raises(ValueError):
        control.SkipSoftmaxConfig()
    with pytest.raises(ValueError):
        control.SkipSoftmaxConfig(threshold=0.1, target_sparsity=0.5, coefficients={"a": 1, "b": 1})
    with pytest.raises(ValueError, match="threshold"):
        control.SkipSoftmaxConfig(target_sparsity=0.5)
    with pytest.raises(ValueError, match="formula"):
        control.SkipSoftmaxConfig(target_sparsity=0.5, coefficients={"a": 1, "b": 1}, formula="a * b")
    cfg = control.SkipSoftmaxConfig(threshold=1e-3, disabled_until_timestep=0.9)
    assert cfg.factor(32760, t=0.95) == 0.0
    assert cfg.factor(32760, t=0.5) == pytest.approx(32.76)
    with warnings.catch_warnings(record=True) as w:
        warnings.simplefilter("always")
        assert cfg.factor(32760, t=None) == 0.0
        assert cfg.factor(32760, t=None) == 0.0
    assert len(w) == 1
    cal = control.SkipSoftmaxConfig(target_sparsity=0.5, coefficients={"a": 2.0, "b": 0.0})
    assert cal.factor(1000) == 2.0
