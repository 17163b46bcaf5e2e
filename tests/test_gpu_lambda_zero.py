"""Factor 0 (lambda = 0) against a factor too small to skip anything.

With lambda = 0 the threshold ln(lambda) is -inf, so no row passes the skip test and every key
tile is kept; the kernel takes the same path as for any other factor. A factor so small that
the test cannot pass either (ln lambda below -85 while score gaps stay within a few tens) must
therefore give bit-identical outputs, for bf16 and e4m3 scores, fixed-length batches, packed
documents, and the min_seq_len gate (which turns lambda to 0 on the host). Both are also
checked against the oracle by the parity tests at factor 0."""
import math

import numpy as np
import pytest

import synth
from tests import parity

pytestmark = pytest.mark.gpu

TINY_FACTOR = 2e-38  # nothing skippable


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


def _blasst():
    import softmax_threshold_tile_gb300 as blasst
    return blasst


def _no_error():
    st, word = _blasst().blasst_device_error(clear=True)
    assert st == _blasst().BLASST_OK and word == 0, f"device error word {word:#x}"


def _same(a, b):
    import torch
    torch.cuda.synchronize()
    _no_error()
    assert int(a.skip_counts.sum()) == 0 and int(b.skip_counts.sum()) == 0
    assert torch.equal(a.o, b.o)
    assert torch.equal(a.lse, b.lse)
    if a.max_prob is not None:
        assert torch.equal(a.max_prob, b.max_prob)


@pytest.mark.parametrize("B,H,Sq,Sk", [(2, 3, 1000, 1000), (1, 2, 300, 1000), (1, 1, 1, 129), (1, 2, 129, 8)])
def test_factor_zero_equals_tiny_factor_bf16(B, H, Sq, Sk):
    q, k, v = parity.clustered_inputs(B, H, Sq, Sk, seed=Sq + 3 * Sk)
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    zero = _blasst().attn_fwd(qd, kd, vd, 0.0, want_mask=True, want_max_prob=True)
    tiny = _blasst().attn_fwd(qd, kd, vd, TINY_FACTOR, want_mask=True, want_max_prob=True)
    _same(zero, tiny)
    assert int(zero.skip_mask.sum()) == 0 and int(tiny.skip_mask.sum()) == 0


def test_factor_zero_equals_tiny_factor_wan_heads():
    """Full Wan length (the benchmark's launch shape per head) on four heads."""
    w = synth.WORKLOADS["wan_32760"]
    q, k, v = synth.make_qkv(w)
    heads = [0, 13, 26, 39]
    qd, kd, vd = (parity.to_device(np.ascontiguousarray(x[:, :, heads])) for x in (q, k, v))
    zero = _blasst().attn_fwd(qd, kd, vd, 0.0)
    tiny = _blasst().attn_fwd(qd, kd, vd, TINY_FACTOR)
    _same(zero, tiny)


def test_fp8_factor_zero_equals_tiny_factor():
    """e4m3 scores: with nothing skippable the two factors give the same bits."""
    import torch
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    q, k, v = parity.clustered_inputs(1, 3, 700, 900, seed=21)
    q8, dq = synth.quantize_e4m3(q)
    k8, dk = synth.quantize_e4m3(k)
    qd, kd, vd = parity.to_device_e4m3(q8), parity.to_device_e4m3(k8), parity.to_device(v)
    zero = _blasst().attn_fwd(qd, kd, vd, 0.0, q_descale=dq, k_descale=dk)
    tiny = _blasst().attn_fwd(qd, kd, vd, TINY_FACTOR, q_descale=dq, k_descale=dk)
    _same(zero, tiny)


def test_factor_zero_equals_tiny_factor_packed_documents():
    import torch
    lens = [1000, 37, 2048, 129, 1]
    qs, ks, vs = [], [], []
    for i, n in enumerate(lens):
        q, k, v = parity.clustered_inputs(1, 2, n, n, seed=40 + i)
        qs.append(q[0]); ks.append(k[0]); vs.append(v[0])
    q, k, v = (np.ascontiguousarray(np.concatenate(x, 0)) for x in (qs, ks, vs))
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).cuda()
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    m = max(lens)
    zero = _blasst().attn_varlen_fwd(qd, kd, vd, cu, cu, m, m, 0.0, want_max_prob=True)
    tiny = _blasst().attn_varlen_fwd(qd, kd, vd, cu, cu, m, m, TINY_FACTOR, want_max_prob=True)
    _same(zero, tiny)


def test_min_seq_len_above_the_length_runs_dense():
    """One length below min_seq_len: the host turns lambda to 0; the outputs equal the factor-0
    call's and nothing is skipped, whatever the factor."""
    q, k, v = parity.clustered_inputs(1, 2, 1000, 1000, seed=5)
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    gated = _blasst().attn_fwd(qd, kd, vd, 64.0, min_seq_len=1001, want_mask=True)
    dense = _blasst().attn_fwd(qd, kd, vd, 0.0, want_mask=True)
    _same(gated, dense)
    units = parity.sample_units(1, 2, 1000, heads=range(2), qtiles=range(8))
    parity.compare_units(q, k, v, gated.o.float().cpu().numpy(), gated.lse.cpu().numpy(),
                         gated.skip_mask.cpu().numpy(), 0.0, units)
    assert math.isfinite(float(gated.lse.min()))
