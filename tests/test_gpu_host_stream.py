"""GPU test of the host-buffer call: heads streamed through a device workspace in groups give
outputs equal, bit for bit, to the device call on the same tensors (every head's attention is
independent of the others), for pinned and pageable host buffers and any group size."""
import numpy as np
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


@pytest.mark.parametrize("B,H,Sq,Sk,hg,pinned", [
    (2, 5, 1000, 777, 2, True), (1, 5, 1000, 777, 1, True), (2, 3, 300, 1300, 3, False), (1, 7, 129, 129, 4, True),
    (1, 13, 700, 700, 5, True), (1, 20, 256, 300, 20, True),
])
def test_host_call_equals_device_call(B, H, Sq, Sk, hg, pinned):
    import torch
    import softmax_threshold_tile_gb300 as blasst
    q, k, v = parity.clustered_inputs(B, H, Sq, Sk, seed=B * 100 + H)
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    ref = blasst.attn_fwd(qd, kd, vd, 4.0)
    torch.cuda.synchronize()

    def host(x):
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
        return t.pin_memory() if pinned else t.clone()

    qh, kh, vh = host(q), host(k), host(v)
    lse = torch.full((B, H, Sq), float("nan"), dtype=torch.float32)
    if pinned:
        lse = lse.pin_memory()
    ws = blasst.host_workspace(B, H, Sq, Sk, hg)
    stream = torch.cuda.Stream()
    o, lse = blasst.attn_fwd_host(qh, kh, vh, 4.0, lse=lse, workspace=ws, heads_per_group=hg, stream=stream)
    stream.synchronize()
    assert blasst.blasst_device_error(clear=True) == (blasst.BLASST_OK, 0)
    assert torch.equal(o, ref.o.cpu())
    assert torch.equal(lse, ref.lse.cpu())
    # a second call on the same workspace and stream gives the same bytes
    o2, _ = blasst.attn_fwd_host(qh, kh, vh, 4.0, workspace=ws, heads_per_group=hg, stream=stream)
    stream.synchronize()
    assert torch.equal(o2, o)


def test_host_call_at_factor_zero_equals_device_call():
    """Factor 0 (lambda = 0, nothing skipped) inside the head-group pipeline."""
    import torch
    import softmax_threshold_tile_gb300 as blasst
    B, H, Sq, Sk = 1, 6, 700, 900
    q, k, v = parity.clustered_inputs(B, H, Sq, Sk, seed=77)
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    ref = blasst.attn_fwd(qd, kd, vd, 0.0)
    torch.cuda.synchronize()
    qh, kh, vh = (torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).pin_memory()
                  for x in (q, k, v))
    lse = torch.empty((B, H, Sq), dtype=torch.float32).pin_memory()
    stream = torch.cuda.Stream()
    o, lse = blasst.attn_fwd_host(qh, kh, vh, 0.0, lse=lse, heads_per_group=3, stream=stream)
    stream.synchronize()
    assert blasst.blasst_device_error(clear=True) == (blasst.BLASST_OK, 0)
    assert torch.equal(o, ref.o.cpu())
    assert torch.equal(lse, ref.lse.cpu())


def test_default_workspace_outlives_the_call_on_another_stream():
    """Without a caller workspace the binding allocates one on the call's stream and drops it at
    once; work that the caller then allocates and writes on its current (different) stream must
    not receive that block while the call's copies and kernels still use it."""
    import torch
    import softmax_threshold_tile_gb300 as blasst
    B, H, Sq, Sk, hg = 1, 6, 900, 900, 2
    q, k, v = parity.clustered_inputs(B, H, Sq, Sk, seed=31)
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    ref = blasst.attn_fwd(qd, kd, vd, 4.0)
    torch.cuda.synchronize()
    qh, kh, vh = (torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).pin_memory()
                  for x in (q, k, v))
    ws_bytes = blasst.blasst_host_workspace_bytes(B, H, Sq, Sk, hg)
    side = torch.cuda.Stream()
    for _ in range(3):
        o, _ = blasst.attn_fwd_host(qh, kh, vh, 4.0, heads_per_group=hg, stream=side)
        junk = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")   # on the current stream
        junk.fill_(0xFF)
        side.synchronize()
        torch.cuda.synchronize()
        assert torch.equal(o, ref.o.cpu())
        del junk
