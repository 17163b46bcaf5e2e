"""GPU: the hand-built cases through the C ABI, against their hand-derived masks.

The expected masks come from the method's rule worked out by hand (tests/hand_built.py and
its golden files), not from the oracle: one query row keeps a tile (the all-rows rule), rows
past Sq do not vote, a ragged key tail, a gap of exactly ln(lambda) = 0 is kept (the test is
strict), and with lambda > 1 a skipped tile above the running max leaves it where the kept
tiles put it. Decisions must match bit for bit; outputs are compared with the closed forms
where the case has one and with the oracle replaying the GPU's decisions in every case.
"""
import numpy as np
import pytest

from tests import hand_built, parity

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


@pytest.mark.parametrize("case", hand_built.load_cases(), ids=hand_built.case_id)
def test_hand_built_case_on_gpu(case):
    name, c = case
    Sq = c["Sq"]
    q, k, v, vv = hand_built.build(name, Sq)
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    f = hand_built.factor_of(c)
    o, lse, counts, mask = parity.run_gpu(qd, kd, vd, f, hand_built.SCALE)
    assert mask.shape == (1, 1, 1, len(c["mask"]))
    assert mask[0, 0, 0].tolist() == c["mask"]
    assert int(counts.sum()) == sum(c["mask"])
    expected = hand_built.closed_form(name, c, vv)
    if expected is not None:
        o_ref, lse_ref = expected
        err = np.abs(o[0, :Sq, 0, :].astype(np.float64) - o_ref)
        assert err.max() <= parity.MAX_ABS and err.mean() <= parity.MEAN_ABS, (err.max(), err.mean())
        assert np.abs(lse[0, 0, :Sq].astype(np.float64) - lse_ref).max() <= parity.LSE_ABS
    units = np.array([(0, 0, 0)], dtype=np.int32)
    parity.compare_units(q, k, v, o, lse, mask, f, units, scale=hand_built.SCALE)
