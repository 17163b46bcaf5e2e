"""GPU test of failure detection: a device-side wait that runs out gives up, the kernel
leaves through its abort path, the caller reads the failure from its own status word (a
stream-ordered copy, no device-wide synchronization) and from the device error word, and the
context stays usable.

The failure is made by the library's test hook blasst_debug_withhold_key_tile, under which the
producer never issues the copy of one key tile, so the waits on it run out after their time
limit. Nothing faults: every device wait in the kernel is bounded."""
import time

import numpy as np
import pytest

from tests import parity

pytestmark = pytest.mark.gpu

# Bits of the device error word: the producer, the MMA thread or the softmax gave up waiting
# (whichever role's time limit runs out first raises the abort flag; the others then leave
# without a bit of their own), and 1 << 3 for the 50 ms exit drains.
ERR_ROLES = (1 << 0) | (1 << 1) | (1 << 2)


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


@pytest.mark.parametrize("factor", [2.0, 0.0])   # skipping, and lambda = 0
@pytest.mark.parametrize("tile", [0, 1, 3])
def test_withheld_key_tile_times_out_and_context_survives(tile, factor):
    import torch
    import softmax_threshold_tile_gb300 as blasst
    q, k, v = parity.clustered_inputs(1, 2, 512, 512, seed=7)
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    stream = torch.cuda.Stream()
    status = torch.full((1,), 0x55, dtype=torch.int32, device="cuda")
    ref = blasst.attn_fwd(qd, kd, vd, factor, want_mask=True, status=status, stream=stream)
    stream.synchronize()
    assert int(status.item()) == 0          # zeroed by the call, no wait gave up
    assert blasst.blasst_device_error(clear=True) == (blasst.BLASST_OK, 0)

    assert blasst.blasst_debug_withhold_key_tile(tile) == blasst.BLASST_OK
    try:
        t0 = time.monotonic()
        blasst.attn_fwd(qd, kd, vd, factor, status=status, stream=stream)  # the failure shows on the device
        host_status = torch.empty(1, dtype=torch.int32).pin_memory()
        with torch.cuda.stream(stream):
            host_status.copy_(status, non_blocking=True)            # ordered after the kernel on its stream
        stream.synchronize()
        elapsed = time.monotonic() - t0
    finally:
        assert blasst.blasst_debug_withhold_key_tile(-1) == blasst.BLASST_OK
    word_s = int(host_status.item())
    assert word_s & ERR_ROLES, f"status word {word_s:#x}"
    assert (word_s & ~0x1f) == 0, f"status word {word_s:#x}"
    st, word = blasst.blasst_device_error(clear=True)
    assert st == blasst.BLASST_ERR_TIMEOUT
    assert word & ERR_ROLES, f"error word {word:#x}"
    assert (word & ~0x1f) == 0, f"error word {word:#x}"
    assert elapsed < 20.0

    again = blasst.attn_fwd(qd, kd, vd, factor, want_mask=True, status=status, stream=stream)
    stream.synchronize()
    assert int(status.item()) == 0          # the next call is clean
    assert blasst.blasst_device_error(clear=True) == (blasst.BLASST_OK, 0)
    assert torch.equal(again.o, ref.o) and torch.equal(again.lse, ref.lse)
    np.testing.assert_array_equal(again.skip_mask.cpu().numpy(), ref.skip_mask.cpu().numpy())
