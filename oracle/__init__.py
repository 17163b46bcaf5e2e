"""Plain CPU definition of Skip-Softmax (BLASST) attention forward.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` import this package. The CUDA library and its Python
binding never import it, and it imports nothing from them.

The arithmetic lives in ``blasst_oracle.c`` (scalar C, fp64); this module only
compiles it with gcc, marshals numpy arrays and optionally spreads independent
units over host threads (ctypes releases the GIL during each call).

Sources: the "Skip-Softmax" design doc (vLLM-Omni), sections "Algorithm" and
"From configuration to the kernel threshold"; "Skip-Softmax" on docs.vllm.ai,
section "The online-softmax pass".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "blasst_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/liboracle.so`` and return its path."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fPIC", "-shared",
            _SRC, "-o", tmp, "-lm",
        ])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i32p = ctypes.POINTER(ctypes.c_int32)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    f64p = ctypes.POINTER(ctypes.c_double)
    lib.oracle_skip_softmax_attn.restype = ctypes.c_int
    lib.oracle_skip_softmax_attn.argtypes = [
        u16p, u16p, u16p,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, ctypes.c_double, ctypes.c_int, ctypes.c_int,
        i32p, ctypes.c_int, u8p, f64p, f64p, u8p, f64p, f64p,
    ]
    lib.oracle_dense_attn.restype = ctypes.c_int
    lib.oracle_dense_attn.argtypes = [
        u16p, u16p, u16p,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, i32p, ctypes.c_int, f64p, f64p,
    ]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _check_bshd(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != np.uint16 or t.ndim != 4 or not t.flags.c_contiguous:
            raise ValueError(f"{name} must be a C-contiguous uint16 (bf16 bits) array [B,S,H,d]")
    B, Sq, H, d = q.shape
    if k.shape[0] != B or k.shape[2] != H or k.shape[3] != d or v.shape != k.shape:
        raise ValueError("q [B,Sq,H,d], k and v [B,Sk,H,d] shapes disagree")
    return B, Sq, k.shape[1], H, d


def all_units(B: int, H: int, Sq: int, tile_q: int = 128) -> np.ndarray:
    """Every (b, h, qt) triple, in b-major, then h, then qt order."""
    nQ = -(-Sq // tile_q)
    b, h, qt = np.meshgrid(np.arange(B), np.arange(H), np.arange(nQ), indexing="ij")
    return np.stack([b.ravel(), h.ravel(), qt.ravel()], axis=1).astype(np.int32)


def skip_softmax_attn(q, k, v, scale: float, factor: float, units=None, mask_in=None,
                      tile_q: int = 128, tile_k: int = 128, threads: int = 1):
    """Skip-Softmax attention on the listed (b, h, qt) units.

    Returns a dict with, per unit: ``o`` [n, tile_q, d] (NaN past Sq), ``lse``
    [n, tile_q], ``max_prob`` [n, tile_q] (1 / l), ``mask`` [n, nK] (1 = skipped),
    ``gap`` [n, nK] (max over rows of tile_max - running_max, natural-log units),
    plus ``units`` and ``nK``.
    ``mask_in`` [n, nK] replays given decisions instead of running the test.
    """
    lib = _load()
    B, Sq, Sk, H, d = _check_bshd(q, k, v)
    if units is None:
        units = all_units(B, H, Sq, tile_q)
    units = np.ascontiguousarray(units, dtype=np.int32).reshape(-1, 3)
    n = units.shape[0]
    nK = -(-Sk // tile_k)
    o = np.full((n, tile_q, d), np.nan)
    lse = np.full((n, tile_q), np.nan)
    mask = np.zeros((n, nK), dtype=np.uint8)
    gap = np.zeros((n, nK))
    maxp = np.full((n, tile_q), np.nan)
    if mask_in is not None:
        mask_in = np.ascontiguousarray(mask_in, dtype=np.uint8).reshape(n, nK)

    def run(lo, hi):
        if hi <= lo:
            return 0
        return lib.oracle_skip_softmax_attn(
            _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
            B, H, Sq, Sk, d, float(scale), float(factor), tile_q, tile_k,
            _ptr(units[lo:hi], ctypes.c_int32), hi - lo,
            None if mask_in is None else _ptr(mask_in[lo:hi], ctypes.c_uint8),
            _ptr(o[lo:hi], ctypes.c_double), _ptr(lse[lo:hi], ctypes.c_double),
            _ptr(mask[lo:hi], ctypes.c_uint8), _ptr(gap[lo:hi], ctypes.c_double),
            _ptr(maxp[lo:hi], ctypes.c_double))

    threads = max(1, min(int(threads), n)) if n else 1
    if threads == 1:
        rcs = [run(0, n)]
    else:
        bounds = np.linspace(0, n, threads + 1).astype(int)
        with ThreadPoolExecutor(threads) as ex:
            rcs = list(ex.map(lambda i: run(bounds[i], bounds[i + 1]), range(threads)))
    if any(rcs):
        raise ValueError(f"oracle_skip_softmax_attn rejected its arguments (codes {rcs})")
    return {"o": o, "lse": lse, "mask": mask, "gap": gap, "max_prob": maxp, "units": units, "nK": nK}


def dense_attn(q, k, v, scale: float, rows, threads: int = 1):
    """Textbook softmax(scale * q k^T) v for the listed (b, h, s) rows: (o [n,d], lse [n])."""
    lib = _load()
    B, Sq, Sk, H, d = _check_bshd(q, k, v)
    rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
    n = rows.shape[0]
    o = np.zeros((n, d))
    lse = np.zeros(n)

    def run(lo, hi):
        if hi <= lo:
            return 0
        return lib.oracle_dense_attn(
            _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
            B, H, Sq, Sk, d, float(scale), _ptr(rows[lo:hi], ctypes.c_int32), hi - lo,
            _ptr(o[lo:hi], ctypes.c_double), _ptr(lse[lo:hi], ctypes.c_double))

    threads = max(1, min(int(threads), n)) if n else 1
    bounds = np.linspace(0, n, threads + 1).astype(int)
    with ThreadPoolExecutor(threads) as ex:
        rcs = list(ex.map(lambda i: run(bounds[i], bounds[i + 1]), range(threads)))
    if any(rcs):
        raise ValueError(f"oracle_dense_attn rejected its arguments (codes {rcs})")
    return o, lse


def unit_rows(units, Sq: int, tile_q: int = 128):
    """For oracle outputs laid out per unit: (unit index, row-in-tile, b, h, s) of every valid row."""
    out = []
    for u, (b, h, qt) in enumerate(np.asarray(units).reshape(-1, 3)):
        r0 = int(qt) * tile_q
        for i in range(min(tile_q, Sq - r0)):
            out.append((u, i, int(b), int(h), r0 + i))
    return np.array(out, dtype=np.int64).reshape(-1, 5)
