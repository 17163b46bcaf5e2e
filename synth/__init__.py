"""Seeded synthetic inputs for Skip-Softmax attention, and the workload table.

This module draws inputs only; it holds no step of the attention method. Both the
CPU oracle (through the tests) and the CUDA path (tests and benchmark) consume the
same bf16 bytes it produces. The generator itself is ``gen.c`` (counter-based
SplitMix64 + Box-Muller, defined in that file's header); this wrapper compiles it
with gcc and spreads token ranges over host threads.

Workloads follow the video-DiT token-grid shapes of the attention benchmarks: a
T x H x W latent grid flattened in raster order, tokens clustered by grid cell
(Q = K-side structure gamma * c_cell + noise), V pure noise.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None
_lock = threading.Lock()

GAMMA_STREAM = 0x7A  # stream id for per-head gamma draws (tensor ids 0..3 use the high bits)


def build(force: bool = False) -> str:
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fPIC",
                               "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.synth_fill.restype = ctypes.c_int
            lib.synth_fill.argtypes = [
                ctypes.POINTER(ctypes.c_uint16), ctypes.c_int, ctypes.c_uint64,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.POINTER(ctypes.c_double), ctypes.c_int, ctypes.c_int,
            ]
            lib.synth_uniform.restype = ctypes.c_double
            lib.synth_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
            lib.synth_f32_to_bf16.restype = ctypes.c_uint16
            lib.synth_f32_to_bf16.argtypes = [ctypes.c_float]
            _lib = lib
    return _lib


def uniform(seed: int, stream: int, index: int) -> float:
    return float(_load().synth_uniform(seed, stream, index))


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 bit patterns, nearest-even (vectorised, same rule as gen.c)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = ((u & 0x7F800000) == 0x7F800000) & ((u & 0x007FFFFF) != 0)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF
    r = np.where(nan, ((u >> 16) | 0x40) & 0xFFFF, r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)



E4M3_MAX = 448.0  # largest finite OCP FP8 e4m3 ("e4m3fn") value: 1.75 * 2^8


def f32_to_e4m3_bits(x) -> np.ndarray:
    """Round float32 values to OCP FP8 e4m3 bit patterns (1 sign, 4 exponent bits with bias 7,
    3 mantissa bits; no infinities), nearest-even, saturating to +-448. Codes 0x7F / 0xFF (NaN)
    are produced only for NaN input."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.uint8) << 7
    a = np.minimum(np.abs(np.nan_to_num(x, nan=0.0)), E4M3_MAX)
    _, ex = np.frexp(a)                     # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)              # unbiased exponent; below 2^-6 the subnormal step
    q = np.rint(a / np.ldexp(1.0, e - 3))   # mantissa with the leading one, in steps of 1/8
    # normal: code = (e + 7) * 8 + (q - 8); q == 16 carries into the exponent on its own.
    # subnormal (e == -6, q < 8): code = q.
    code = np.where(q >= 8, (e + 7) * 8 + (q - 8), q).astype(np.int64)
    out = (code.astype(np.uint8) | sign).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), out).astype(np.uint8)


def e4m3_bits_to_f32(bits) -> np.ndarray:
    """Decode OCP FP8 e4m3 bit patterns (0x7F / 0xFF are NaN)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    e = (b >> 3) & 0xF
    m = b & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    val = np.where(b & 0x80, -mag, mag)
    val = np.where((b & 0x7F) == 0x7F, np.nan, val)
    return val.astype(np.float32)


def quantize_e4m3(bits_bf16):
    """Per-tensor FP8 quantisation of a bf16 tensor, as a caller would do before an e4m3 call:
    descale = amax / 448, codes = e4m3(x / descale). Returns (uint8 codes, descale)."""
    x = bf16_bits_to_f32(bits_bf16).astype(np.float64)
    amax = float(np.abs(x).max()) if x.size else 0.0
    descale = amax / E4M3_MAX if amax > 0 else 1.0
    descale = float(np.float32(descale))
    return f32_to_e4m3_bits((x / descale).astype(np.float32)), descale

@dataclass
class Workload:
    """One synthetic attention problem: shapes, token grid, clustering and factor sweep."""
    name: str
    B: int
    H: int
    S: int
    d: int = 128
    grid: tuple = (0, 0, 0)       # T, Hg, W of the latent token grid (0: no structure)
    cell: tuple = (1, 1, 1)       # ct, ch, cw
    gamma: float | None = 2.0     # one weight for every (b, h) ...
    gamma_per_batch: tuple | None = None   # ... or one per batch entry ...
    gamma_range: tuple | None = None       # ... or per head, uniform in [lo, hi) (seeded)
    factors: tuple = (0.0,)
    curve: tuple | None = None    # (a, b, (t, ...)): factor = a * exp(b * t) per point
    seed: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def Sq(self):
        return self.S

    @property
    def Sk(self):
        return self.S

    def gammas(self) -> np.ndarray:
        """[B * H] centre weights, b-major."""
        if self.gamma_per_batch is not None:
            g = np.repeat(np.asarray(self.gamma_per_batch, dtype=np.float64), self.H)
        elif self.gamma_range is not None:
            lo, hi = self.gamma_range
            g = np.array([lo + (hi - lo) * uniform(self.seed, GAMMA_STREAM, b * self.H + h)
                          for b in range(self.B) for h in range(self.H)])
        else:
            g = np.full(self.B * self.H, float(self.gamma))
        return g

    def dense_flops(self) -> float:
        return 4.0 * self.B * self.H * self.S * self.S * self.d


WORKLOADS = {
    "tiny_1024": Workload("tiny_1024", B=1, H=2, S=1024, grid=(4, 16, 16), cell=(2, 4, 4),
                          gamma=2.0, factors=(0.0, 0.5, 2.0, 8.0)),
    "dit_8192_g1": Workload("dit_8192_g1", B=1, H=24, S=8192, grid=(8, 32, 32), cell=(2, 8, 8),
                            gamma=1.0, factors=(0.0, 1.0, 4.0, 16.0, 64.0)),
    "dit_8192_g2": Workload("dit_8192_g2", B=1, H=24, S=8192, grid=(8, 32, 32), cell=(2, 8, 8),
                            gamma=2.0, factors=(0.0, 1.0, 4.0, 16.0, 64.0)),
    "dit_8192_g3": Workload("dit_8192_g3", B=1, H=24, S=8192, grid=(8, 32, 32), cell=(2, 8, 8),
                            gamma=3.0, factors=(0.0, 1.0, 4.0, 16.0, 64.0)),
    "wan_32760": Workload("wan_32760", B=1, H=40, S=32760, grid=(21, 30, 52), cell=(3, 6, 6),
                          gamma=2.0, factors=(0.0, 2.0, 8.0, 32.0)),
    "long_65536": Workload("long_65536", B=1, H=24, S=65536, grid=(16, 64, 64), cell=(2, 8, 8),
                           gamma=None, gamma_range=(0.5, 3.0), factors=(0.0, 4.0, 16.0)),
    "ragged_37000": Workload("ragged_37000", B=2, H=32, S=37000, grid=(37, 25, 40), cell=(2, 8, 8),
                             gamma=None, gamma_per_batch=(0.0, 3.0),
                             curve=(1.0, 4.0, (0.5, 0.75, 0.9)),
                             notes="batch 0 i.i.d. noise, batch 1 clustered (gamma 3)"),
}


def fill(tensor: int, B: int, S: int, H: int, d: int, seed: int = 0, grid=(0, 0, 0), cell=(1, 1, 1),
         gammas=None, threads: int | None = None) -> np.ndarray:
    """A [B, S, H, d] uint16 (bf16 bits) array for tensor 1 (Q), 2 (K) or 3 (V)."""
    lib = _load()
    out = np.empty((B, S, H, d), dtype=np.uint16)
    g = None if gammas is None else np.ascontiguousarray(gammas, dtype=np.float64)
    gp = None if g is None else g.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    threads = threads or min(32, os.cpu_count() or 1)
    bounds = np.linspace(0, S, max(1, min(threads, S)) + 1).astype(int)

    def run(i):
        return lib.synth_fill(out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), tensor, seed,
                              B, S, H, d, grid[0], grid[1], grid[2], cell[0], cell[1], cell[2],
                              gp, int(bounds[i]), int(bounds[i + 1]))

    with ThreadPoolExecutor(len(bounds) - 1) as ex:
        rcs = list(ex.map(run, range(len(bounds) - 1)))
    if any(rcs):
        raise ValueError("synth_fill rejected its arguments")
    return out


def make_qkv(w: Workload | str, threads: int | None = None, Sq: int | None = None, Sk: int | None = None):
    """(q, k, v) uint16 arrays [B, S, H, d] for a workload (optionally truncated to Sq / Sk tokens)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    g = w.gammas()
    sq = w.S if Sq is None else Sq
    sk = w.S if Sk is None else Sk
    q = fill(1, w.B, sq, w.H, w.d, w.seed, w.grid, w.cell, g, threads)
    k = fill(2, w.B, sk, w.H, w.d, w.seed, w.grid, w.cell, g, threads)
    v = fill(3, w.B, sk, w.H, w.d, w.seed, (0, 0, 0), (1, 1, 1), None, threads)
    return q, k, v
