"""Race detection by repetition: the kernel accumulates with no atomics in its arithmetic and
every pipeline hand-off is an ordered barrier, so repeated calls on the same inputs must give
the same bits (o, lse, max_prob, skip counts and mask). A missing fence or a stage reused too
early in the warp-specialised pipeline would show here as a run-to-run difference, on the
bf16 scores with and without skipping (factor 0) and the e4m3 score product."""
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


def _repeat(call, reps):
    import torch
    import softmax_threshold_tile_gb300 as blasst
    ref = call()
    torch.cuda.synchronize()
    for r in range(reps):
        res = call()
        torch.cuda.synchronize()
        for name in ("o", "lse", "max_prob", "skip_counts", "skip_mask"):
            a, b = getattr(res, name), getattr(ref, name)
            if a is not None:
                assert torch.equal(a, b), f"{name} differs on repetition {r}"
    assert blasst.blasst_device_error(clear=True) == (blasst.BLASST_OK, 0)


@pytest.mark.parametrize("name,factor,reps", [("dit_8192_g2", 0.0, 10), ("dit_8192_g2", 64.0, 10),
                                              ("dit_8192_g1", 16.0, 10), ("tiny_1024", 2.0, 30)])
def test_repeated_calls_are_bit_identical(name, factor, reps):
    import softmax_threshold_tile_gb300 as blasst
    w = synth.WORKLOADS[name]
    q, k, v = synth.make_qkv(w)
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    _repeat(lambda: blasst.attn_fwd(qd, kd, vd, factor, want_mask=True, want_max_prob=True), reps)


def test_repeated_fp8_calls_are_bit_identical():
    import torch
    import softmax_threshold_tile_gb300 as blasst
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    w = synth.WORKLOADS["dit_8192_g2"]
    q, k, v = synth.make_qkv(w)
    q8, dq = synth.quantize_e4m3(q)
    k8, dk = synth.quantize_e4m3(k)
    qd, kd, vd = parity.to_device_e4m3(q8), parity.to_device_e4m3(k8), parity.to_device(v)
    _repeat(lambda: blasst.attn_fwd(qd, kd, vd, 64.0, q_descale=dq, k_descale=dk, want_mask=True), 10)
