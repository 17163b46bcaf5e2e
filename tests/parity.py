"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle on the same seeded bf16 inputs.

Tolerances (bf16 output O, per the parity bar of the method):
  * decisions replayed in the oracle: max |O_gpu - O_oracle| <= 2e-2 and
    mean |O_gpu - O_oracle| <= 2e-3; lse within 1e-2;
  * free-running decisions may differ from the oracle's only on tiles whose
    log margin |gap - ln(lambda)| is below 1e-3.
"""
from __future__ import annotations

import math
import os

import numpy as np

import oracle
import synth

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_ABS = 1e-2
MARGIN = 1e-3
TILE = 128


def to_device(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def to_device_e4m3(codes):
    import torch
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).cuda().view(torch.float8_e4m3fn)


def run_gpu(qd, kd, vd, factor, scale=None, **kw):
    """Call the CUDA path through the C ABI; returns numpy (o fp32 [B,Sq,H,d], lse, counts, mask)."""
    import torch
    import softmax_threshold_tile_gb300 as blasst

    res = blasst.attn_fwd(qd, kd, vd, factor, scale, want_mask=True, **kw)
    torch.cuda.synchronize()
    st, word = blasst.blasst_device_error(clear=True)
    assert st == blasst.BLASST_OK and word == 0, f"device error word {word:#x}"
    o = res.o.float().cpu().numpy()
    lse = res.lse.cpu().numpy()
    counts = res.skip_counts.cpu().numpy().astype(np.int64)
    mask = res.skip_mask.cpu().numpy()
    return o, lse, counts, mask


def check_counts(counts, mask, factor):
    B, H = mask.shape[:2]
    np.testing.assert_array_equal(counts.reshape(B, H), mask.reshape(B, H, -1).sum(-1))
    assert np.all(mask[..., 0] == 0), "the first key tile of a query tile was skipped"
    if factor == 0:
        assert counts.sum() == 0


def sample_units(B, H, Sq, heads=None, qtiles=None, batches=None):
    nQ = -(-Sq // TILE)
    heads = sorted(set(heads if heads is not None else (0, H // 2, H - 1)))
    qtiles = sorted(set(qtiles if qtiles is not None else (0, 1, nQ // 2, nQ - 1)))
    batches = sorted(set(batches if batches is not None else range(B)))
    return np.array([(b, h, t) for b in batches for h in heads for t in qtiles if 0 <= t < nQ],
                     dtype=np.int32)


def host_threads():
    """Every host core: the oracle's units are independent."""
    return os.cpu_count() or 1


def compare_units(q, k, v, o_gpu, lse_gpu, mask_gpu, factor, units, scale=None, threads=None, margin=MARGIN,
                  return_gap=False):
    """Replay the GPU's decisions in the oracle on `units`; assert the parity bar.

    Returns a dict of the observed errors and decision agreement; with return_gap, its "gap"
    entry holds the oracle's per-(unit, key tile) log margins max_i(tile_max - running_max)."""
    threads = host_threads() if threads is None else threads
    B, Sq, H, d = q.shape
    Sk = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    nK = -(-Sk // TILE)
    m_in = np.stack([mask_gpu[b, h, t] for b, h, t in units]).astype(np.uint8)
    ref = oracle.skip_softmax_attn(q, k, v, scale, factor, units=units, mask_in=m_in, threads=threads)
    errs, lse_errs = [], []
    for u, (b, h, t) in enumerate(units):
        r0 = t * TILE
        n = min(TILE, Sq - r0)
        diff = np.abs(o_gpu[b, r0:r0 + n, h, :].astype(np.float64) - ref["o"][u, :n])
        errs.append(diff)
        lse_errs.append(np.abs(lse_gpu[b, h, r0:r0 + n].astype(np.float64) - ref["lse"][u, :n]))
    err = np.concatenate([e.ravel() for e in errs])
    lerr = np.concatenate(lse_errs)
    assert np.all(np.isfinite(err)), "non-finite output"
    max_abs, mean_abs = float(err.max()), float(err.mean())
    assert max_abs <= MAX_ABS, f"max |dO| {max_abs:.3g} > {MAX_ABS}"
    assert mean_abs <= MEAN_ABS, f"mean |dO| {mean_abs:.3g} > {MEAN_ABS}"
    assert float(lerr.max()) <= LSE_ABS, f"max |dlse| {float(lerr.max()):.3g} > {LSE_ABS}"
    # Free-running agreement: with lambda <= 1 the replayed run has the same running-max chain
    # as a free run, so the oracle's own decision on every tile is gap < ln(lambda).
    ln_lam = math.log(factor / Sk) if factor > 0 else -math.inf
    free = (ref["gap"] < ln_lam).astype(np.uint8)
    differ = free != m_in
    if factor / Sk <= 1.0:
        margins = np.abs(ref["gap"][differ] - ln_lam)
        assert np.all(margins < margin), f"decision differs on a tile with margin {margins.max():.3g}"
    out = {"max_abs": max_abs, "mean_abs": mean_abs, "lse_max_abs": float(lerr.max()),
           "decisions": int(m_in.size), "differ": int(differ.sum()), "skipped": int(m_in.sum())}
    if return_gap:
        out["gap"] = ref["gap"]
    return out


def check_decisions(gap, mask, factor, Sk, margin=MARGIN):
    """Decisions of a run at `factor` against the oracle's gap chain of the same units.

    For lambda <= 1 a skipped tile never raises the running max, so the running max before key
    tile j is the dense prefix max at every factor, and one oracle pass gives the gap of every
    tile for all factors. The free-running decision is gap < ln(lambda); the GPU's may differ
    only where |gap - ln(lambda)| < margin. Returns (decisions, differ)."""
    assert factor / Sk <= 1.0
    ln_lam = math.log(factor / Sk) if factor > 0 else -math.inf
    free = gap < ln_lam
    differ = free != mask.astype(bool)
    if differ.any():
        margins = np.abs(gap[differ] - ln_lam)
        assert np.all(margins < margin), f"decision differs on a tile with margin {margins.max():.3g}"
    return int(mask.size), int(differ.sum())


def whole_head_units(b, h, Sq):
    """Every query tile of one (batch, head)."""
    return np.array([(b, h, t) for t in range(-(-Sq // TILE))], dtype=np.int32)


def clustered_inputs(B, H, Sq, Sk, seed=0, gamma=2.0, cell=16):
    """Clustered Q/K along a 1 x 1 x S token line (cells of `cell` tokens), V noise."""
    g = np.full(B * H, gamma)
    q = synth.fill(1, B, Sq, H, 128, seed, (1, 1, Sq), (1, 1, cell), g)
    k = synth.fill(2, B, Sk, H, 128, seed, (1, 1, Sk), (1, 1, cell), g)
    v = synth.fill(3, B, Sk, H, 128, seed)
    return q, k, v
