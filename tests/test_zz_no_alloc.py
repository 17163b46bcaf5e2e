"""The host-buffer call that allocates nothing, blasst_attn_fwd_host_noalloc.

Some callers cannot call cudaMalloc. One is a plug-in inside a host application that keeps all of
the GPU's memory in its own pool. Another is a latency-critical loop that must not call cudaMalloc
or cudaFree, because they can synchronize the device. This entry point serves them. It runs the
head-group pipeline of blasst_attn_fwd_host with its device workspace in a fixed-size buffer that
the library holds itself.

The GPU test calls it through the C ABI on two calls in a row: the second is smaller and
has another shape, so stale bytes from the first call stay in the buffer. Each call's outputs
are checked against blasst_attn_fwd_host with a caller-owned workspace, within the parity
tolerances. The file name makes pytest collect it after every other test file.
"""
import math

import numpy as np
import pytest

from tests import parity


def _blasst():
    import softmax_threshold_tile_gb300 as blasst
    blasst.build_library()
    blasst.load_library()
    return blasst


def _pinned(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).pin_memory()


def test_too_large_for_the_buffer_is_rejected_before_any_cuda_call():
    blasst = _blasst()
    scale = 1 / math.sqrt(128)
    # one head of 300 000 queries and keys needs two slots of ~307 MB: more than the buffer
    B, H, S = 1, 2, 300_000
    assert blasst.blasst_host_workspace_bytes(B, H, S, S, 1) > blasst.BLASST_NOALLOC_SCRATCH_BYTES
    st = blasst.blasst_attn_fwd_host_noalloc(4096, 8192, 12288, 16384, None, B, H, S, S, 128, scale, 2.0, 1, None)
    assert st == blasst.BLASST_ERR_TOO_LARGE
    # a caller workspace is not accepted here, and the usual argument checks apply
    assert blasst.blasst_attn_fwd_host_noalloc(4096, 8192, 12288, 16384, None, 1, 2, 256, 256, 64, scale, 2.0, 1,
                                               None) == blasst.BLASST_ERR_INVALID_ARG
    assert blasst.blasst_attn_fwd_host_noalloc(4096, 8192, 12288, 16384, None, 1, 2, 256, 256, 128, scale, 2.0, 3,
                                               None) == blasst.BLASST_ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_call_matches_the_host_call_on_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    blasst = _blasst()
    scale = 1 / math.sqrt(128)
    stream = torch.cuda.Stream()
    # (B, H, Sq, Sk, largest head group, factor, seed): the first call fills more of the buffer
    # than the second, which then runs over the first call's leftover bytes.
    cases = [(2, 5, 1500, 1300, 3, 4.0, 41), (1, 3, 700, 513, 2, 16.0, 42)]
    for B, H, Sq, Sk, hg, factor, seed in cases:
        q, k, v = parity.clustered_inputs(B, H, Sq, Sk, seed=seed)
        qh, kh, vh = _pinned(q), _pinned(k), _pinned(v)

        # the existing entry point, with a workspace the caller allocates
        ws_bytes = blasst.blasst_host_workspace_bytes(B, H, Sq, Sk, hg)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        o_ref = torch.empty((B, Sq, H, 128), dtype=torch.bfloat16).pin_memory()
        lse_ref = torch.empty((B, H, Sq), dtype=torch.float32).pin_memory()
        st = blasst.blasst_attn_fwd_host(qh, kh, vh, o_ref, lse_ref, B, H, Sq, Sk, 128, scale, factor, ws, ws_bytes,
                                         hg, stream.cuda_stream)
        assert st == blasst.BLASST_OK
        stream.synchronize()

        # the entry point that allocates nothing
        o = torch.full((B, Sq, H, 128), float("nan"), dtype=torch.bfloat16).pin_memory()
        lse = torch.full((B, H, Sq), float("nan"), dtype=torch.float32).pin_memory()
        st = blasst.blasst_attn_fwd_host_noalloc(qh, kh, vh, o, lse, B, H, Sq, Sk, 128, scale, factor, hg,
                                                 stream.cuda_stream)
        assert st == blasst.BLASST_OK, blasst.blasst_status_string(st)
        stream.synchronize()
        assert blasst.blasst_device_error(clear=True) == (blasst.BLASST_OK, 0)

        err = (o.float() - o_ref.float()).abs()
        assert torch.isfinite(err).all()
        assert float(err.max()) <= parity.MAX_ABS
        assert float(err.mean()) <= parity.MEAN_ABS
        assert float((lse - lse_ref).abs().max()) <= parity.LSE_ABS
        # every head is computed on its own, so the two calls give the same bits
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
        del ws
