"""Host-side controls: from user settings to the factor the kernel takes.

The arithmetic is in the C library (``blasst_factor_from_threshold``,
``blasst_factor_from_target_sparsity``, ``blasst_gate_factor``, ``blasst_dense_steps``,
``blasst_flow_shift_schedule``); this module marshals arguments and adds the settings
checks of the "Skip-Softmax" design doc (vLLM-Omni), sections "From configuration to the
kernel threshold" and "Timestep gating": ``threshold`` and ``target_sparsity`` are
mutually exclusive, only the curve ``a * exp(b * target_sparsity)`` is accepted, a
``target_sparsity`` without calibration is an error pointing to ``threshold``, and a
pipeline that does not publish its timestep stays dense with one warning.
"""
from __future__ import annotations

import ctypes
import warnings

from ._binding import BLASST_OK, BlasstError, load_library

CURVE_FORMULA = "a * exp(b * target_sparsity)"


def _check(st: int, what: str):
    if st != BLASST_OK:
        raise BlasstError(st, what)


def factor_from_threshold(threshold: float, max_kv_len: int) -> float:
    out = ctypes.c_double()
    _check(load_library().blasst_factor_from_threshold(float(threshold), int(max_kv_len), ctypes.byref(out)),
           "blasst_factor_from_threshold")
    return out.value


def factor_from_target_sparsity(a: float, b: float, target_sparsity: float) -> float:
    out = ctypes.c_double()
    _check(load_library().blasst_factor_from_target_sparsity(float(a), float(b), float(target_sparsity),
                                                              ctypes.byref(out)),
           "blasst_factor_from_target_sparsity")
    return out.value


def gate_factor(factor: float, disabled_until_timestep: float, t: float | None) -> tuple[float, bool]:
    """(factor for this call, whether the caller should warn that no timestep is published)."""
    out, warn = ctypes.c_double(), ctypes.c_int()
    _check(load_library().blasst_gate_factor(float(factor), float(disabled_until_timestep), 0 if t is None else 1,
                                             0.0 if t is None else float(t), ctypes.byref(out), ctypes.byref(warn)),
           "blasst_gate_factor")
    return out.value, bool(warn.value)


def dense_steps(ts, disabled_until_timestep: float) -> int:
    vals = [float(x) for x in ts]
    arr = (ctypes.c_double * max(1, len(vals)))(*vals)
    out = ctypes.c_int()
    _check(load_library().blasst_dense_steps(arr, len(vals), float(disabled_until_timestep), ctypes.byref(out)),
           "blasst_dense_steps")
    return out.value


def flow_shift_schedule(shift: float, num_points: int) -> list[float]:
    arr = (ctypes.c_double * int(num_points))()
    _check(load_library().blasst_flow_shift_schedule(float(shift), int(num_points), arr), "blasst_flow_shift_schedule")
    return list(arr)


class SkipSoftmaxConfig:
    """Per-layer settings: exactly one of ``threshold`` or ``target_sparsity`` (with calibration
    ``coefficients = {"a": .., "b": ..}`` and ``formula``), plus ``disabled_until_timestep``."""

    def __init__(self, threshold=None, target_sparsity=None, coefficients=None,
                 formula: str = CURVE_FORMULA, disabled_until_timestep: float = 0.0):
        if (threshold is None) == (target_sparsity is None):
            raise ValueError("set exactly one of threshold or target_sparsity")
        if target_sparsity is not None:
            if formula != CURVE_FORMULA:
                raise ValueError(f"unsupported calibration formula {formula!r}; only {CURVE_FORMULA!r} is accepted")
            if not coefficients or "a" not in coefficients or "b" not in coefficients:
                raise ValueError("target_sparsity needs calibration coefficients a and b; "
                                 "use threshold for a calibration-free setting")
        self.threshold = threshold
        self.target_sparsity = target_sparsity
        self.coefficients = coefficients
        self.disabled_until_timestep = float(disabled_until_timestep)
        self._warned = False

    def factor(self, max_kv_len: int, t: float | None = None) -> float:
        """The threshold_scale_factor for one attention call (0 means dense)."""
        if self.threshold is not None:
            f = factor_from_threshold(self.threshold, max_kv_len)
        else:
            f = factor_from_target_sparsity(self.coefficients["a"], self.coefficients["b"], self.target_sparsity)
        g, warn = gate_factor(f, self.disabled_until_timestep, t)
        if warn and not self._warned:
            warnings.warn("disabled_until_timestep is set but no timestep was published; running dense")
            self._warned = True
        return g
