"""Host-side checks of the C ABI: the library loads, exports every declared symbol, and
rejects invalid arguments before any CUDA call. No GPU is needed."""
import math
import os
import re
import subprocess

import pytest

import softmax_threshold_tile_gb300 as blasst

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    blasst.build_library()
    return blasst.load_library()


def declared_functions():
    names = set()
    for fn in os.listdir(INCLUDE):
        if fn.endswith(".h"):
            text = open(os.path.join(INCLUDE, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(blasst_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "blasst_attn_fwd" in names and len(names) >= 4
    out = subprocess.run(["nm", "-D", "--defined-only", blasst.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (\w+)$", out, flags=re.M))
    for n in names:
        assert n in exported, f"{n} is declared in include/ but not exported"
        assert hasattr(lib, n)


def test_status_strings(lib):
    for code in range(6):
        assert blasst.blasst_status_string(code)
    assert blasst.blasst_version() >= 100


GOOD = dict(q=256, k=512, v=768, o=1024, lse=None, B=1, H=2, Sq=1024, Sk=1024, d=128,
            scale=1 / math.sqrt(128), factor=2.0, stream=None, skip_counts=None, skip_mask_dbg=None)


def call(**kw):
    a = dict(GOOD)
    a.update(kw)
    return blasst.blasst_attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Sq"],
                                  a["Sk"], a["d"], a["scale"], a["factor"], a["stream"],
                                  a["skip_counts"], a["skip_mask_dbg"])


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(k=None), dict(v=None), dict(o=None),
    dict(B=0), dict(H=0), dict(Sq=0), dict(Sk=0), dict(B=-1), dict(H=70000), dict(B=65536),
    dict(d=64), dict(d=256),
    dict(scale=0.0), dict(scale=-0.1), dict(scale=float("nan")), dict(scale=float("inf")),
    dict(factor=-1.0), dict(factor=float("nan")), dict(factor=float("inf")),
    dict(q=258), dict(k=8), dict(v=1032), dict(o=1000), dict(lse=1026),
    dict(H=65535, Sq=2 ** 31 - 1),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_invalid_arguments_rejected_before_any_cuda_call(lib, kw):
    assert call(**kw) == blasst.BLASST_ERR_INVALID_ARG


def test_valid_call_without_gb300_reports_unsupported_device(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the GPU tests cover this path")
    # Pointers are never dereferenced: the device check fails first.
    assert call() == blasst.BLASST_ERR_UNSUPPORTED_DEVICE


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        blasst.load_library(str(tmp_path / "absent.so"))


def test_package_has_no_cpu_fallback():
    """The product package imports nothing from the oracle and has no CPU compute path."""
    pkg = os.path.join(ROOT, "softmax_threshold_tile_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith(".py"):
                src = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", src, flags=re.M), fn
                assert "softmax(" not in src, fn


def test_extended_args_struct_matches_header(tmp_path):
    import ctypes
    src = tmp_path / "size.c"
    src.write_text('#include <stdio.h>\n#include "blasst.h"\nint main(void){printf("%zu\\n", sizeof(blasst_fwd_args));return 0;}\n')
    exe = tmp_path / "size"
    subprocess.check_call(["gcc", "-I", INCLUDE, str(src), "-o", str(exe)])
    size = int(subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout)
    assert size == ctypes.sizeof(blasst.FwdArgs)


def call_ex(**kw):
    a = dict(q=256, k=512, v=768, o=1024, lse=None, max_prob=None, B=2, H=2, Sq=1000, Sk=1000, d=128,
             scale=1 / math.sqrt(128), factor=2.0, stream=None, skip_counts=None, skip_mask_dbg=None,
             cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=0, max_seqlen_k=0, min_seq_len=0)
    a.update(kw)
    return blasst.blasst_attn_fwd_ex(**a)


@pytest.mark.parametrize("kw", [
    dict(cu_seqlens_q=4096),                           # only one offset table
    dict(cu_seqlens_k=4096),
    dict(cu_seqlens_q=4096, cu_seqlens_k=8192, max_seqlen_q=600, max_seqlen_k=600, skip_mask_dbg=64),
    dict(cu_seqlens_q=4096, cu_seqlens_k=8192, max_seqlen_q=0, max_seqlen_k=600),
    dict(cu_seqlens_q=4096, cu_seqlens_k=8192, max_seqlen_q=600, max_seqlen_k=1001),
    dict(cu_seqlens_q=4098, cu_seqlens_k=8192, max_seqlen_q=600, max_seqlen_k=600),
    dict(max_prob=1026), dict(min_seq_len=-1), dict(d=64),
    dict(qk_format=2), dict(qk_format=-1),                  # unknown score-operand format
    dict(qk_format=1, q_descale=0.0), dict(qk_format=1, k_descale=-2.0),
    dict(qk_format=1, q_descale=float("nan")), dict(qk_format=1, k_descale=float("inf")),
    dict(qk_format=1, q=264),                               # e4m3 q must still be 16-byte aligned
    dict(status=4098),                                      # the status word must be 4-byte aligned
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_extended_invalid_arguments(lib, kw):
    assert call_ex(**kw) == blasst.BLASST_ERR_INVALID_ARG


def test_extended_rejects_wrong_struct_size(lib):
    import ctypes
    a = blasst.FwdArgs()
    a.struct_size = ctypes.sizeof(blasst.FwdArgs) - 4
    assert lib.blasst_attn_fwd_ex(ctypes.byref(a)) == blasst.BLASST_ERR_INVALID_ARG
    assert lib.blasst_attn_fwd_ex(None) == blasst.BLASST_ERR_INVALID_ARG


def test_extended_accepts_the_layout_without_status(lib):
    """A caller built against the layout before the status word passes that smaller struct_size:
    its arguments are read (an invalid one is still rejected) and status counts as NULL."""
    import ctypes
    old = blasst.FwdArgs.status.offset
    a = blasst.FwdArgs()
    a.struct_size = old
    a.q, a.k, a.v, a.o = 256, 512, 768, 1024
    a.B, a.H, a.Sq, a.Sk, a.d = 1, 2, 300, 300, 128
    a.scale, a.factor = 1 / math.sqrt(128), 2.0
    a.status = 4098  # past the caller's struct: never read
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert lib.blasst_attn_fwd_ex(ctypes.byref(a)) == blasst.BLASST_ERR_UNSUPPORTED_DEVICE
    a.d = 64
    assert lib.blasst_attn_fwd_ex(ctypes.byref(a)) == blasst.BLASST_ERR_INVALID_ARG


def test_debug_hooks(lib):
    assert blasst.blasst_debug_withhold_key_tile(-2) == blasst.BLASST_ERR_INVALID_ARG
    assert blasst.blasst_debug_withhold_key_tile(-1) == blasst.BLASST_OK
    assert blasst.blasst_tensor_map_encodes() >= 0


def test_host_args_struct_matches_header(tmp_path):
    import ctypes
    src = tmp_path / "hsize.c"
    src.write_text('#include <stdio.h>\n#include "blasst.h"\nint main(void){printf("%zu\\n", sizeof(blasst_host_args));return 0;}\n')
    exe = tmp_path / "hsize"
    subprocess.check_call(["gcc", "-I", INCLUDE, str(src), "-o", str(exe)])
    size = int(subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout)
    assert size == ctypes.sizeof(blasst.HostArgs)


def test_host_workspace_bytes(lib):
    B, H, Sq, Sk, hg = 2, 5, 1000, 777, 2
    n = blasst.blasst_host_workspace_bytes(B, H, Sq, Sk, hg)
    # two slots, each holding q, o (B Sq hg 256 B), k, v (B Sk hg 256 B) and lse (B hg Sq 4 B), 256-B aligned
    per = 2 * B * Sq * hg * 256 + 2 * B * Sk * hg * 256 + B * hg * Sq * 4
    assert 2 * per <= n <= 2 * (per + 5 * 256) and n % 256 == 0
    assert blasst.blasst_host_workspace_bytes(B, H, Sq, Sk, H) > n
    for bad in ((0, H, Sq, Sk, hg), (B, H, Sq, Sk, 0), (B, H, Sq, Sk, H + 1), (B, H, 0, Sk, hg)):
        assert blasst.blasst_host_workspace_bytes(*bad) == 0


def call_host(**kw):
    B, H, Sq, Sk = 2, 3, 500, 400
    a = dict(q=4096, k=8192, v=12288, o=16384, lse=None, B=B, H=H, Sq=Sq, Sk=Sk, d=128,
             scale=1 / math.sqrt(128), factor=2.0, workspace=1 << 20,
             workspace_bytes=blasst.blasst_host_workspace_bytes(B, H, Sq, Sk, 2), heads_per_group=2, stream=None)
    a.update(kw)
    return blasst.blasst_attn_fwd_host(**a)


@pytest.mark.parametrize("kw", [
    dict(q=0), dict(o=0), dict(workspace=0), dict(d=64), dict(B=0), dict(Sk=0),
    dict(heads_per_group=0), dict(heads_per_group=4),
    dict(workspace=(1 << 20) + 16),                      # not 256-byte aligned
    dict(workspace_bytes=1000),                          # too small
    dict(scale=0.0), dict(factor=-1.0), dict(factor=float("nan")),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_host_call_invalid_arguments(lib, kw):
    assert call_host(**kw) == blasst.BLASST_ERR_INVALID_ARG


def test_host_call_rejects_wrong_struct_size(lib):
    import ctypes
    a = blasst.HostArgs()
    a.struct_size = ctypes.sizeof(blasst.HostArgs) + 8
    assert lib.blasst_attn_fwd_host(ctypes.byref(a)) == blasst.BLASST_ERR_INVALID_ARG
