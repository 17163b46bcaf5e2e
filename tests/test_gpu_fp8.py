"""GPU parity of the FP8 score product: q and k as e4m3 codes (per-tensor scales), v and the
P . V product in bf16.

The oracle runs on the decoded e4m3 values (each one is exactly a bf16 value) with the score
scale multiplied by both dequantisation factors, so the parity bar is the bf16 one: the kernel
and the oracle see the same operands and differ only in accumulation order and precision.
Free-running decisions may differ only on tiles whose log margin is below MARGIN_FP8."""
import math

import numpy as np
import pytest

import synth
from tests import parity

pytestmark = pytest.mark.gpu

MARGIN_FP8 = parity.MARGIN


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    import softmax_threshold_tile_gb300 as blasst
    blasst.build_library()
    blasst.load_library()
    yield
    torch.cuda.synchronize()


def _fp8_case(q, k, v):
    """(device q8, k8, v) and the oracle's bf16 inputs and score scale for them."""
    q8, dq = synth.quantize_e4m3(q)
    k8, dk = synth.quantize_e4m3(k)
    qo = synth.f32_to_bf16_bits(synth.e4m3_bits_to_f32(q8))
    ko = synth.f32_to_bf16_bits(synth.e4m3_bits_to_f32(k8))
    scale = float(np.float32(1 / math.sqrt(128)))
    oscale = scale * float(np.float32(dq)) * float(np.float32(dk))
    dev = (parity.to_device_e4m3(q8), parity.to_device_e4m3(k8), parity.to_device(v))
    return dev, (qo, ko, v), scale, oscale, dq, dk


def _check(w_or_inputs, factors, units_fn, S_k):
    q, k, v = w_or_inputs
    (qd, kd, vd), (qo, ko, vo), scale, oscale, dq, dk = _fp8_case(q, k, v)
    out = []
    prev = None
    for f in sorted(factors):
        o, lse, counts, mask = parity.run_gpu(qd, kd, vd, f, scale, q_descale=dq, k_descale=dk)
        parity.check_counts(counts, mask, f)
        if prev is not None and f / S_k <= 1.0:
            assert not np.any(prev.astype(bool) & ~mask.astype(bool)), "skip set shrank as lambda grew"
        prev = mask
        st = parity.compare_units(qo, ko, vo, o, lse, mask, f, units_fn(q.shape), scale=oscale,
                                  margin=MARGIN_FP8)
        st["factor"] = f
        out.append(st)
    print(out)
    return out


def test_fp8_tiny_1024_every_unit():
    w = synth.WORKLOADS["tiny_1024"]
    st = _check(synth.make_qkv(w), w.factors, lambda s: parity.sample_units(
        s[0], s[2], s[1], heads=range(s[2]), qtiles=range(s[1] // 128)), w.S)
    assert st[0]["skipped"] == 0 and st[-1]["skipped"] > 0


@pytest.mark.parametrize("Sq,Sk", [(1, 1), (129, 77), (1000, 1300), (640, 384)])
def test_fp8_ragged(Sq, Sk):
    inp = parity.clustered_inputs(2, 3, Sq, Sk, seed=Sq + Sk)
    _check(inp, [0.0, 2.0, 32.0], lambda s: parity.sample_units(
        s[0], s[2], s[1], heads=range(s[2]), qtiles=range(-(-s[1] // 128))), Sk)


@pytest.mark.parametrize("seed", range(6))
def test_fp8_random_shapes(seed):
    """Seeded random shapes for the e4m3 score product, every query tile checked."""
    rng = np.random.default_rng(700 + seed)
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 5))
    Sq, Sk = int(rng.integers(1, 900)), int(rng.integers(1, 1400))
    gamma = float(rng.uniform(0.5, 3.0))
    g = np.full(B * H, gamma)
    q = synth.fill(1, B, Sq, H, 128, seed, (1, 1, Sq), (1, 1, 16), g)
    k = synth.fill(2, B, Sk, H, 128, seed, (1, 1, Sk), (1, 1, 16), g)
    v = synth.fill(3, B, Sk, H, 128, seed)
    _check((q, k, v), [0.0, float(rng.choice([1.0, 8.0, 64.0]))], lambda s: parity.sample_units(
        s[0], s[2], s[1], heads=range(s[2]), qtiles=range(-(-s[1] // 128))), Sk)


def test_fp8_dit_8192_sampled():
    w = synth.WORKLOADS["dit_8192_g2"]
    st = _check(synth.make_qkv(w), [0.0, 16.0], lambda s: parity.sample_units(
        s[0], s[2], s[1], heads=(0, s[2] - 1), qtiles=(0, 5, 31, 63)), w.S)
    assert st[-1]["skipped"] > 0


def test_fp8_varlen_and_max_prob_equal_separate_calls():
    import torch
    import softmax_threshold_tile_gb300 as blasst
    lens = [700, 129, 1500]
    H = 2
    parts = [parity.clustered_inputs(1, H, n, n, seed=40 + i) for i, n in enumerate(lens)]
    q = np.concatenate([p[0][0] for p in parts])
    k = np.concatenate([p[1][0] for p in parts])
    v = np.concatenate([p[2][0] for p in parts])
    q8, dq = synth.quantize_e4m3(q)
    k8, dk = synth.quantize_e4m3(k)
    qd, kd, vd = parity.to_device_e4m3(q8), parity.to_device_e4m3(k8), parity.to_device(v)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    factor = 8.0
    res = blasst.attn_varlen_fwd(qd, kd, vd, cu, cu, max(lens), max(lens), factor, want_max_prob=True,
                                 q_descale=dq, k_descale=dk)
    torch.cuda.synchronize()
    assert blasst.blasst_device_error(clear=True)[1] == 0
    counts = res.skip_counts.cpu().numpy().reshape(len(lens), H)
    c = np.concatenate([[0], np.cumsum(lens)])
    for i, n in enumerate(lens):
        one = blasst.attn_fwd(qd[None, c[i]:c[i + 1]].contiguous(), kd[None, c[i]:c[i + 1]].contiguous(),
                              vd[None, c[i]:c[i + 1]].contiguous(), factor * n / max(lens), want_max_prob=True,
                              q_descale=dq, k_descale=dk)
        torch.cuda.synchronize()
        if np.array_equal(one.skip_counts.cpu().numpy(), counts[i]):
            assert torch.equal(one.o[0], res.o[c[i]:c[i + 1]])
            assert torch.equal(one.max_prob[0], res.max_prob[:, c[i]:c[i + 1]])


def test_fp8_quantisation_error_is_the_oracles():
    """The e4m3 call against the bf16 oracle differs by the quantisation error the oracle itself
    predicts (oracle on decoded e4m3 against oracle on bf16), plus at most the parity bar."""
    import torch
    import oracle
    import softmax_threshold_tile_gb300 as blasst
    w = synth.WORKLOADS["tiny_1024"]
    q, k, v = synth.make_qkv(w)
    (qd, kd, vd), (qo, ko, _), scale, oscale, dq, dk = _fp8_case(q, k, v)
    r8 = blasst.attn_fwd(qd, kd, vd, 0.0, scale, q_descale=dq, k_descale=dk)
    torch.cuda.synchronize()
    units = parity.sample_units(w.B, w.H, w.S, heads=range(w.H), qtiles=(0, 3, 7))
    ref16 = oracle.skip_softmax_attn(q, k, v, scale, 0.0, units=units, threads=parity.host_threads())
    ref8 = oracle.skip_softmax_attn(qo, ko, v, oscale, 0.0, units=units, threads=parity.host_threads())
    o8 = r8.o.float().cpu().numpy()
    got = np.stack([o8[b, t * 128:(t + 1) * 128, h] for b, h, t in units])
    quant = np.abs(ref8["o"] - ref16["o"])
    err = np.abs(got - ref16["o"])
    print("e4m3 vs bf16: kernel mean |dO|", err.mean(), "oracle's quantisation error", quant.mean())
    assert np.all(err <= quant + parity.MAX_ABS)
    assert err.mean() <= quant.mean() + parity.MEAN_ABS


def test_fp8_rejects_bad_descale():
    import torch
    import softmax_threshold_tile_gb300 as blasst
    x8 = torch.zeros((1, 128, 1, 128), dtype=torch.float8_e4m3fn, device="cuda")
    v = torch.zeros((1, 128, 1, 128), dtype=torch.bfloat16, device="cuda")
    for dq in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(blasst.BlasstError):
            blasst.attn_fwd(x8, x8, v, 1.0, q_descale=dq)
    with pytest.raises(ValueError):
        blasst.attn_fwd(x8, v, v, 1.0)  # k must be e4m3 like q
