"""Plain definitions of the host-side controls that turn user settings into the kernel's
threshold_scale_factor. TEST INFRASTRUCTURE, like the rest of ``oracle/``.

Sources: the "Skip-Softmax" design doc (vLLM-Omni), sections "From configuration to the
kernel threshold" (threshold -> factor, the calibrated curve), "Timestep gating" and
"Mapping the cutoff to denoising steps" (the gate, dense-step count, flow-shift schedule).
"""
from __future__ import annotations

import math


def factor_from_threshold(threshold: float, max_kv_len: int) -> float:
    """The direct control: the kernel gets threshold * max_kv_len, so lambda == threshold."""
    if not (math.isfinite(threshold) and threshold >= 0.0) or max_kv_len <= 0:
        raise ValueError("threshold must be finite and >= 0, max_kv_len > 0")
    return threshold * max_kv_len


def factor_from_target_sparsity(a: float, b: float, target_sparsity: float) -> float:
    """The calibrated control: factor = a * exp(b * target_sparsity)."""
    f = a * math.exp(b * target_sparsity)
    if not (math.isfinite(f) and f >= 0.0):
        raise ValueError("the calibrated curve gives no finite non-negative factor")
    return f


def gate_factor(factor: float, disabled_until_timestep: float, t: float | None):
    """(factor passed to the kernel, warn) for one attention call.

    disabled_until_timestep == 0 is the 'gate off' sentinel: t is never read. Otherwise the
    call is dense (factor 0) while t > cutoff, and also when no t is published (with a
    warning); skipping is active once t <= cutoff.
    """
    if disabled_until_timestep == 0.0:
        return factor, False
    if t is None:
        return 0.0, True
    return (0.0 if t > disabled_until_timestep else factor), False


def dense_steps(ts, disabled_until_timestep: float) -> int:
    """count(t[i] > disabled_until_timestep) over a published sequence."""
    return sum(1 for t in ts if t > disabled_until_timestep)


def flow_shift_schedule(shift: float, num_points: int):
    """t = s*u / (1 + (s-1)*u) at num_points uniform positions u from 1 down to 0."""
    if num_points < 2:
        raise ValueError("need at least two positions")
    out = []
    for i in range(num_points):
        u = 1.0 - i / (num_points - 1)
        out.append(shift * u / (1.0 + (shift - 1.0) * u))
    return out
