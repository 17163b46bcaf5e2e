"""Skip-Softmax (BLASST) attention forward for GB300 (sm_103a).

All compute runs in the hand-written CUDA library built from ``csrc/`` (see
``build.build()``); this package is its C ABI (``include/blasst.h``) exposed
through ctypes, plus host-side helpers. PyTorch is only used for device memory
and streams. Nothing here falls back to a CPU or library implementation.
"""
from ._binding import (  # noqa: F401
    BLASST_ERR_INVALID_ARG,
    BLASST_ERR_LAUNCH,
    BLASST_ERR_TIMEOUT,
    BLASST_ERR_TOO_LARGE,
    BLASST_ERR_UNSUPPORTED_DEVICE,
    BLASST_NOALLOC_SCRATCH_BYTES,
    BLASST_OK,
    BLASST_QK_BF16,
    BLASST_QK_E4M3,
    HEAD_DIM,
    TILE,
    AttnResult,
    BlasstError,
    FwdArgs,
    HostArgs,
    attn_fwd,
    attn_fwd_host,
    host_workspace,
    blasst_attn_fwd_host,
    blasst_attn_fwd_host_noalloc,
    blasst_debug_withhold_key_tile,
    blasst_host_workspace_bytes,
    blasst_tensor_map_encodes,
    attn_varlen_fwd,
    blasst_attn_fwd_ex,
    blasst_attn_fwd,
    blasst_device_error,
    blasst_status_string,
    blasst_version,
    library_path,
    load_library,
)
from .build import build as build_library  # noqa: F401
from . import control  # noqa: F401,E402
