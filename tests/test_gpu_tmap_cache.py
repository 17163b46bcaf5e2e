"""GPU test of the per-process cache of TMA tensor descriptors: repeated calls on the same tensors
encode none, a changed address or shape encodes a new one, and results do not depend on whether
a descriptor came from the cache."""
import pytest

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


def test_descriptor_cache_hits_and_misses():
    import torch
    import softmax_threshold_tile_gb300 as blasst
    q, k, v = parity.clustered_inputs(1, 3, 701, 903, seed=12)  # shapes no other test uses
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    first = blasst.attn_fwd(qd, kd, vd, 4.0)
    torch.cuda.synchronize()
    n0 = blasst.blasst_tensor_map_encodes()
    for _ in range(3):                               # same tensors: every descriptor from the cache
        again = blasst.attn_fwd(qd, kd, vd, 4.0)
    torch.cuda.synchronize()
    assert blasst.blasst_tensor_map_encodes() == n0
    assert torch.equal(again.o, first.o) and torch.equal(again.lse, first.lse)

    q2 = qd.clone()                                  # a new address for q only
    moved = blasst.attn_fwd(q2, kd, vd, 4.0)
    torch.cuda.synchronize()
    assert blasst.blasst_tensor_map_encodes() == n0 + 1
    assert torch.equal(moved.o, first.o)

    # the same addresses with a shorter key length (a contiguous prefix): new shapes for k and v
    short = blasst.attn_fwd(qd, kd[:, :501], vd[:, :501], 4.0)
    torch.cuda.synchronize()
    assert blasst.blasst_tensor_map_encodes() == n0 + 3
    ref = blasst.attn_fwd(qd, kd[:, :501].clone(), vd[:, :501].clone(), 4.0)
    torch.cuda.synchronize()
    assert torch.equal(short.o, ref.o)
    assert blasst.blasst_device_error(clear=True) == (blasst.BLASST_OK, 0)
