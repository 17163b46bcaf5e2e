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
BLASST_ERR_TOO_LARGE = 5

# Size of the library's own device buffer used by blasst_attn_fwd_host_noalloc.
BLASST_NOALLOC_SCRATCH_BYTES = 256 << 20

BLASST_QK_BF16 = 0
BLASST_QK_E4M3 = 1

TILE = 128
HEAD_DIM = 128

_lib = None


class FwdArgs(ctypes.Structure):
    """Mirror of ``blasst_fwd_args`` (include/blasst.h)."""
    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("max_prob", ctypes.c_void_p),
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("Sq", ctypes.c_int), ("Sk", ctypes.c_int), ("d", ctypes.c_int),
        ("scale", ctypes.c_float), ("factor", ctypes.c_float),
        ("stream", ctypes.c_void_p),
        ("skip_counts", ctypes.c_void_p), ("skip_mask_dbg", ctypes.c_void_p),
        ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
        ("max_seqlen_q", ctypes.c_int), ("max_seqlen_k", ctypes.c_int),
        ("min_seq_len", ctypes.c_int),
        ("qk_format", ctypes.c_int),
        ("q_descale", ctypes.c_float), ("k_descale", ctypes.c_float),
        ("status", ctypes.c_void_p),
    ]


class HostArgs(ctypes.Structure):
    """Mirror of ``blasst_host_args`` (include/blasst.h)."""
    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("Sq", ctypes.c_int), ("Sk", ctypes.c_int), ("d", ctypes.c_int),
        ("scale", ctypes.c_float), ("factor", ctypes.c_float),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("heads_per_group", ctypes.c_int),
        ("stream", ctypes.c_void_p),
    ]


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
    lib.blasst_attn_fwd_ex.restype = ctypes.c_int
    lib.blasst_attn_fwd_ex.argtypes = [ctypes.POINTER(FwdArgs)]
    lib.blasst_attn_fwd_host.restype = ctypes.c_int
    lib.blasst_attn_fwd_host.argtypes = [ctypes.POINTER(HostArgs)]
    lib.blasst_host_workspace_bytes.restype = ctypes.c_size_t
    lib.blasst_host_workspace_bytes.argtypes = [ctypes.c_int] * 5
    lib.blasst_status_string.restype = ctypes.c_char_p
    lib.blasst_status_string.argtypes = [ctypes.c_int]
    lib.blasst_device_error.restype = ctypes.c_int
    lib.blasst_device_error.argtypes = [u32p, ctypes.c_int]
    lib.blasst_version.restype = ctypes.c_int
    lib.blasst_version.argtypes = []
    lib.blasst_debug_withhold_key_tile.restype = ctypes.c_int
    lib.blasst_debug_withhold_key_tile.argtypes = [ctypes.c_int]
    lib.blasst_tensor_map_encodes.restype = ctypes.c_uint64
    lib.blasst_tensor_map_encodes.argtypes = []
    lib.blasst_attn_fwd_host_noalloc.restype = ctypes.c_int
    lib.blasst_attn_fwd_host_noalloc.argtypes = [ctypes.POINTER(HostArgs)]
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


def blasst_attn_fwd_ex(q, k, v, o, lse, max_prob, B, H, Sq, Sk, d, scale, factor, stream, skip_counts,
                       skip_mask_dbg, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=0, max_seqlen_k=0,
                       min_seq_len=0, qk_format=BLASST_QK_BF16, q_descale=1.0, k_descale=1.0,
                       status=None) -> int:
    """The extended C entry point: fills a ``blasst_fwd_args`` and calls it."""
    a = FwdArgs()
    a.struct_size = ctypes.sizeof(FwdArgs)
    a.q, a.k, a.v, a.o, a.lse, a.max_prob = _p(q), _p(k), _p(v), _p(o), _p(lse), _p(max_prob)
    a.B, a.H, a.Sq, a.Sk, a.d = int(B), int(H), int(Sq), int(Sk), int(d)
    a.scale, a.factor = float(scale), float(factor)
    a.stream = _p(stream)
    a.skip_counts, a.skip_mask_dbg = _p(skip_counts), _p(skip_mask_dbg)
    a.cu_seqlens_q, a.cu_seqlens_k = _p(cu_seqlens_q), _p(cu_seqlens_k)
    a.max_seqlen_q, a.max_seqlen_k, a.min_seq_len = int(max_seqlen_q), int(max_seqlen_k), int(min_seq_len)
    a.qk_format, a.q_descale, a.k_descale = int(qk_format), float(q_descale), float(k_descale)
    a.status = _p(status)
    return int(load_library().blasst_attn_fwd_ex(ctypes.byref(a)))


def blasst_host_workspace_bytes(B, H, Sq, Sk, heads_per_group) -> int:
    return int(load_library().blasst_host_workspace_bytes(int(B), int(H), int(Sq), int(Sk), int(heads_per_group)))


def blasst_attn_fwd_host(q, k, v, o, lse, B, H, Sq, Sk, d, scale, factor, workspace, workspace_bytes,
                         heads_per_group, stream) -> int:
    """The host-buffer C entry point: q / k / v / o / lse are HOST addresses (or CPU tensors),
    workspace a device address (or CUDA tensor)."""
    a = HostArgs()
    a.struct_size = ctypes.sizeof(HostArgs)
    a.q, a.k, a.v, a.o, a.lse = _p(q), _p(k), _p(v), _p(o), _p(lse)
    a.B, a.H, a.Sq, a.Sk, a.d = int(B), int(H), int(Sq), int(Sk), int(d)
    a.scale, a.factor = float(scale), float(factor)
    a.workspace, a.workspace_bytes = _p(workspace), int(workspace_bytes)
    a.heads_per_group = int(heads_per_group)
    a.stream = _p(stream)
    return int(load_library().blasst_attn_fwd_host(ctypes.byref(a)))


def blasst_attn_fwd_host_noalloc(q, k, v, o, lse, B, H, Sq, Sk, d, scale, factor, heads_per_group,
                                 stream) -> int:
    """The host-buffer C entry point that allocates nothing (its workspace is the library's own
    fixed device buffer); q / k / v / o / lse are HOST addresses (or CPU tensors)."""
    a = HostArgs()
    a.struct_size = ctypes.sizeof(HostArgs)
    a.q, a.k, a.v, a.o, a.lse = _p(q), _p(k), _p(v), _p(o), _p(lse)
    a.B, a.H, a.Sq, a.Sk, a.d = int(B), int(H), int(Sq), int(Sk), int(d)
    a.scale, a.factor = float(scale), float(factor)
    a.workspace, a.workspace_bytes = None, 0
    a.heads_per_group = int(heads_per_group)
    a.stream = _p(stream)
    return int(load_library().blasst_attn_fwd_host_noalloc(ctypes.byref(a)))


def blasst_debug_withhold_key_tile(tile: int) -> int:
    """Test hook of the bounded device waits: the producer withholds the copy of key tile `tile`
    in every launch from now on (-1: off)."""
    return int(load_library().blasst_debug_withhold_key_tile(int(tile)))


def blasst_tensor_map_encodes() -> int:
    """TMA tensor descriptors encoded by this process so far (the cache's misses)."""
    return int(load_library().blasst_tensor_map_encodes())


def blasst_status_string(code: int) -> str:
    try:
        return load_library().blasst_status_string(int(code)).decode()
    except RuntimeError:
        return {0: "ok", 1: "invalid argument", 2: "unsupported device", 3: "CUDA launch or set-up failure",
                4: "a device-side wait timed out", 5: "too large for the library's fixed buffer"}.get(
                    int(code), "unknown status")


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
    max_prob: object = None


def _check_qkv(q, k, v, packed: bool) -> int:
    """Validate the operands; returns the qk format (bf16 q / k, or e4m3 q / k with bf16 v)."""
    import torch
    nd = 3 if packed else 4
    shape = "[S, H, 128]" if packed else "[B, S, H, 128]"
    fp8 = getattr(torch, "float8_e4m3fn", None)
    qk_format = BLASST_QK_E4M3 if fp8 is not None and q.dtype == fp8 else BLASST_QK_BF16
    qk_dtype = fp8 if qk_format == BLASST_QK_E4M3 else torch.bfloat16
    for name, t, want in (("q", q, qk_dtype), ("k", k, qk_dtype), ("v", v, torch.bfloat16)):
        if t.dtype != want or t.dim() != nd or not t.is_contiguous() or not t.is_cuda:
            kind = "bf16" if want == torch.bfloat16 else "float8_e4m3fn (like q)"
            raise ValueError(f"{name} must be a contiguous CUDA {kind} tensor {shape}")
    if packed:
        bad = k.shape != v.shape or k.shape[1:] != q.shape[1:]
    else:
        bad = k.shape != v.shape or k.shape[0] != q.shape[0] or k.shape[2:] != q.shape[2:]
    if bad:
        raise ValueError("q, k and v shapes disagree")
    return qk_format


def attn_fwd(q, k, v, factor: float, scale: float | None = None, *, out=None, want_lse: bool = True,
             want_counts: bool = True, want_mask: bool = False, want_max_prob: bool = False,
             min_seq_len: int = 0, q_descale: float = 1.0, k_descale: float = 1.0,
             status=None, stream=None) -> AttnResult:
    """Skip-Softmax attention on torch CUDA tensors [B, S, H, 128] (contiguous): q / k / v bf16,
    or q / k float8_e4m3fn with v bf16 (scores then carry q_descale * k_descale).

    Allocates the outputs with torch (device memory only) and calls the C entry point on the
    current (or given) stream. `status` (optional CUDA int32 tensor of one element) receives the
    error bits of CTAs whose device waits gave up, zeroed by the call first. Raises BlasstError on
    any non-OK status.
    """
    import torch

    qk_format = _check_qkv(q, k, v, packed=False)
    B, Sq, H, d = q.shape
    Sk = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = q.device
    o = out if out is not None else torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=dev) if want_lse else None
    mp = torch.empty((B, H, Sq), dtype=torch.float32, device=dev) if want_max_prob else None
    counts = torch.empty((B * H,), dtype=torch.int32, device=dev) if want_counts else None
    nQ, nK = -(-Sq // TILE), -(-Sk // TILE)
    mask = torch.empty((B, H, nQ, nK), dtype=torch.uint8, device=dev) if want_mask else None
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if mp is None and min_seq_len == 0 and qk_format == BLASST_QK_BF16 and status is None:
        st = blasst_attn_fwd(q, k, v, o, lse, B, H, Sq, Sk, d, scale, factor, stream.cuda_stream, counts, mask)
    else:
        st = blasst_attn_fwd_ex(q, k, v, o, lse, mp, B, H, Sq, Sk, d, scale, factor, stream.cuda_stream, counts,
                                mask, min_seq_len=min_seq_len, qk_format=qk_format, q_descale=q_descale,
                                k_descale=k_descale, status=status)
    if st != BLASST_OK:
        raise BlasstError(st, "blasst_attn_fwd")
    return AttnResult(o, lse, counts, mask, mp)


def attn_varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int, factor: float,
                    scale: float | None = None, *, out=None, want_lse: bool = True, want_counts: bool = True,
                    want_max_prob: bool = False, min_seq_len: int = 0, q_descale: float = 1.0,
                    k_descale: float = 1.0, stream=None) -> AttnResult:
    """Packed documents: q / o [Tq, H, 128], k / v [Tk, H, 128] (bf16, or e4m3 q / k as in
    attn_fwd) and int32 CUDA offset tables of B + 1 entries. lambda = factor / max_seqlen_k
    for every document."""
    import torch

    qk_format = _check_qkv(q, k, v, packed=True)
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or t.dim() != 1 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA int32 vector")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k need the same B + 1 >= 2 entries")
    Tq, H, d = q.shape
    Tk = k.shape[0]
    B = cu_seqlens_q.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = q.device
    o = out if out is not None else torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((H, Tq), dtype=torch.float32, device=dev) if want_lse else None
    mp = torch.empty((H, Tq), dtype=torch.float32, device=dev) if want_max_prob else None
    counts = torch.empty((B * H,), dtype=torch.int32, device=dev) if want_counts else None
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    st = blasst_attn_fwd_ex(q, k, v, o, lse, mp, B, H, Tq, Tk, d, scale, factor, stream.cuda_stream, counts, None,
                            cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, min_seq_len, qk_format,
                            q_descale, k_descale)
    if st != BLASST_OK:
        raise BlasstError(st, "blasst_attn_fwd_ex")
    return AttnResult(o, lse, counts, None, mp)


def host_workspace(B: int, H: int, Sq: int, Sk: int, heads_per_group: int, device=None):
    """A device workspace (uint8 CUDA tensor) large enough for attn_fwd_host."""
    import torch
    n = blasst_host_workspace_bytes(B, H, Sq, Sk, heads_per_group)
    if n == 0:
        raise ValueError("invalid sizes for the host-buffer call")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def attn_fwd_host(q, k, v, factor: float, scale: float | None = None, *, out=None, lse=None, workspace=None,
                  heads_per_group: int | None = None, stream=None):
    """Skip-Softmax attention on HOST tensors [B, S, H, 128] bf16 (contiguous CPU tensors; pinned for
    overlap), streamed through a device workspace by head groups. Returns (o, lse) CPU tensors; they
    are complete once `stream` (default: the current stream) has reached the end of the call."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous() or t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CPU bf16 tensor [B, S, H, 128]")
    B, Sq, H, d = q.shape
    Sk = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if heads_per_group is None:
        heads_per_group = max(1, H // 5)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=q.is_pinned())
    if stream is None:
        stream = torch.cuda.current_stream()
    if workspace is None:
        # Allocated on `stream`, the stream the call's last step joins: once this tensor is
        # released, the caching allocator hands its block only to work ordered after the call.
        with torch.cuda.stream(stream):
            workspace = host_workspace(B, H, Sq, Sk, heads_per_group)
    st = blasst_attn_fwd_host(q, k, v, out, lse, B, H, Sq, Sk, d, scale, factor, workspace,
                              workspace.numel() * workspace.element_size(), heads_per_group, stream.cuda_stream)
    if st != BLASST_OK:
        raise BlasstError(st, "blasst_attn_fwd_host")
    return out, lse
