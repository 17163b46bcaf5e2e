"""ctypes binding of the C ABI declared in ``include/blasst.h`` (argument marshalling only).

Every step of the attention pass runs in the CUDA library; this module only
loads it, declares the C signatures and turns torch tensors into device
pointers. If the library is missing the calls raise: there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import NamedTuple

from .build import LIB_PATH

BLASST_OK = 0
BLASST_ERR_INVALID_ARG = 1
BLASST_ERR_UNSUPPORTED_DEVICE = 2
BLASST_ERR_LAUNCH = 3
BLASST_ERR_TIMEOUT = 4

TILE = 128
HEAD_DIM = 128

_lib = None


class BlasstError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {blasst_status_string(code)} (status {code})")
        self.code = code


def library_path() -> str:
    return LIB_PATH


def load_library(path: str | None = None):
    """Open the CUDA library (default: the in-tree build) and declare its signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"CUDA library {p} is not built; call softmax_threshold_tile_gb300.build.build() first")
    lib = ctypes.CDLL(p)
    vp, u32p, u8p, f32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p, ctypes.c_void_p
    lib.blasst_attn_fwd.restype = ctypes.c_int
    lib.blasst_attn_fwd.argtypes = [vp, vp, vp, vp, f32p,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_float, ctypes.c_float, vp, vp, u8p]
    lib.blasst_status_string.restype = ctypes.c_char_p
    lib.blasst_status_string.argtypes = [ctypes.c_int]
    lib.blasst_device_error.restype = ctypes.c_int
    lib.blasst_device_error.argtypes = [u32p, ctypes.c_int]
    lib.blasst_version.restype = ctypes.c_int
    lib.blasst_version.argtypes = []
    dp, ip = ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)
    lib.blasst_factor_from_threshold.restype = ctypes.c_int
    lib.blasst_factor_from_threshold.argtypes = [ctypes.c_double, ctypes.c_int64, dp]
    lib.blasst_factor_from_target_sparsity.restype = ctypes.c_int
    lib.blasst_factor_from_target_sparsity.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_double, dp]
    lib.blasst_gate_factor.restype = ctypes.c_int
    lib.blasst_gate_factor.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_int, ctypes.c_double, dp, ip]
    lib.blasst_dense_steps.restype = ctypes.c_int
    lib.blasst_dense_steps.argtypes = [dp, ctypes.c_int, ctypes.c_double, ip]
    lib.blasst_flow_shift_schedule.restype = ctypes.c_int
    lib.blasst_flow_shift_schedule.argtypes = [ctypes.c_double, ctypes.c_int, dp]
    if path is None:
        _lib = lib
    return lib


def _p(x) -> int | None:
    """A pointer argument: None / 0 -> NULL, int -> address, tensor -> data_ptr()."""
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    return x.data_ptr()


def blasst_attn_fwd(q, k, v, o, lse, B, H, Sq, Sk, d, scale, factor, stream, skip_counts,
                    skip_mask_dbg) -> int:
    """The C entry point, one to one. Pointers are ints (device addresses), tensors or None."""
    return int(load_library().blasst_attn_fwd(
        _p(q), _p(k), _p(v), _p(o), _p(lse), int(B), int(H), int(Sq), int(Sk), int(d),
        float(scale), float(factor), _p(stream), _p(skip_counts), _p(skip_mask_dbg)))


def blasst_status_string(code: int) -> str:
    try:
        return load_library().blasst_status_string(int(code)).decode()
    except RuntimeError:
        return {0: "ok", 1: "invalid argument", 2: "unsupported device", 3: "CUDA launch or set-up failure",
                4: "a device-side wait timed out"}.get(int(code), "unknown status")


def blasst_device_error(clear: bool = True) -> tuple[int, int]:
    """(status, error word) of the current device; synchronizes the device."""
    word = ctypes.c_uint32(0)
    st = int(load_library().blasst_device_error(ctypes.byref(word), 1 if clear else 0))
    return st, int(word.value)


def blasst_version() -> int:
    return int(load_library().blasst_version())


class AttnResult(NamedTuple):
    o: object
    lse: object
    skip_counts: object
    skip_mask: object


def attn_fwd(q, k, v, factor: float, scale: float | None = None, *, out=None, want_lse: bool = True,
             want_counts: bool = True, want_mask: bool = False, stream=None) -> AttnResult:
    """Skip-Softmax attention on torch CUDA tensors [B, S, H, 128] bf16 (contiguous).

    Allocates the outputs with torch (device memory only) and calls
    ``blasst_attn_fwd`` on the current (or given) stream. Raises BlasstError on
    any non-OK status.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor [B, S, H, 128]")
    B, Sq, H, d = q.shape
    Sk = k.shape[1]
    if k.shape != (B, Sk, H, d) or v.shape != k.shape:
        raise ValueError("q [B,Sq,H,d] and k, v [B,Sk,H,d] shapes disagree")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = q.device
    o = out if out is not None else torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=dev) if want_lse else None
    counts = torch.empty((B * H,), dtype=torch.int32, device=dev) if want_counts else None
    nQ, nK = -(-Sq // TILE), -(-Sk // TILE)
    mask = torch.empty((B, H, nQ, nK), dtype=torch.uint8, device=dev) if want_mask else None
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    st = blasst_attn_fwd(q, k, v, o, lse, B, H, Sq, Sk, d, scale, factor, stream.cuda_stream, counts, mask)
    if st != BLASST_OK:
        raise BlasstError(st, "blasst_attn_fwd")
    return AttnResult(o, lse, counts, mask)
