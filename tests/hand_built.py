"""Hand-built cases with exactly representable scores, whose skip masks and outputs follow
by hand from the method's rule ("Skip-Softmax" design doc, vLLM-Omni, section
"Algorithm": a key tile is skipped only when tile_max - running_max < ln(lambda) holds
for every query row, and a skipped tile leaves the running max, l and O untouched;
"From configuration to the kernel threshold": lambda = factor / Sk).

Two constructions, each with its golden file under tests/golden/ (construction,
derivation and the expected masks):

* ``tiles``: hand_built_tiles.json — one query row decides a tile (the all-rows rule),
  a query tail that must not vote, a ragged key tail, and a gap of exactly 0 at
  lambda = 1 (the test is strict).
* ``above_one``: hand_built_lambda_above_one.json — lambda > 1, where a skipped tile's
  maximum exceeds the running max and the next tile's decision depends on the running
  max staying where the kept tiles left it.

Inputs are [1, S, 1, 128] bf16 bit patterns; the closed forms below are written from the
derivations, in fp64, and share nothing with the oracle or the CUDA path.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D = 128
SCALE = 1.0 / math.sqrt(D)
FILES = {"tiles": "hand_built_tiles.json", "above_one": "hand_built_lambda_above_one.json"}


def hadamard(n):
    h = np.array([[1]], dtype=np.int64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def values(Sk):
    """V[c][t] = ((7c + 3t) mod 5) - 2: small integers, exact in bf16."""
    c = np.arange(Sk)[:, None]
    t = np.arange(D)[None, :]
    return ((7 * c + 3 * t) % 5 - 2).astype(np.float64)


def build(name, Sq):
    """(q, k, v) bf16 bits [1, S, 1, 128] and V as fp64 [Sk, 128]."""
    h = hadamard(D)
    Sk = 520 if name == "tiles" else 384
    q = np.zeros((1, Sq, 1, D), np.float32)
    q[0, :, 0] = h[:Sq]
    k = np.zeros((1, Sk, 1, D), np.float32)
    if name == "tiles":
        k[0, :128, 0] = 2 * h           # tile 0: row i scores 2 * 128 * scale on key i
        k[0, 256, 0] = 2 * h[5]         # tile 2: one key aligned with query row 5 only
    else:
        k[0, :128, 0] = 1.0 * h         # tile 0: 1 * sqrt(128) on the row's own key
        k[0, 128:256, 0] = 1.25 * h     # tile 1: 1.25 * sqrt(128)
        k[0, 256:384, 0] = 1.5 * h      # tile 2: 1.5 * sqrt(128)
    vv = values(Sk)
    v = vv.astype(np.float32)[None, :, None, :].copy()
    conv = synth.f32_to_bf16_bits
    return conv(q), conv(k), conv(v), vv


def load_cases():
    """[(construction name, case dict)] from both golden files."""
    out = []
    for name, fn in FILES.items():
        with open(os.path.join(GOLDEN, fn)) as fh:
            out += [(name, c) for c in json.load(fh)["cases"]]
    return out


def case_id(nc):
    name, c = nc
    return f"{name}_Sq{c['Sq']}_lnlam{c['ln_lambda']}"


def factor_of(case):
    """lambda = factor / Sk, so factor = Sk * lambda (0 for ln(lambda) = -inf)."""
    ln_lam = float(case["ln_lambda"])
    return 0.0 if ln_lam == -math.inf else case["Sk"] * math.exp(ln_lam)


def closed_form(name, case, vv):
    """Expected O [Sq, 128] and lse [Sq] over the kept keys, or None where the case has none.

    Every row's weights are exp(score) over the kept keys: a handful of large scores on
    the row's own keys and weight 1 (score 0) on every other kept key."""
    Sq, mask = case["Sq"], case["mask"]
    rows_o, rows_lse = [], []
    if name == "tiles" and mask == [0, 1, 0, 1, 1]:
        # kept: tile 0 (row i: 256 * scale on key i) and tile 2 (row 5: 256 * scale on key 256)
        E = math.exp(256 * SCALE)
        tile0, tile2 = vv[0:128], vv[256:384]
        for i in range(Sq):
            if i != 5:
                num = E * tile0[i] + (tile0.sum(0) - tile0[i]) + tile2.sum(0)
                den = E + 127 + 128
            else:
                num = E * tile0[5] + E * tile2[0] + (tile0.sum(0) - tile0[5]) + (tile2.sum(0) - tile2[0])
                den = 2 * E + 127 + 127
            rows_o.append(num / den)
            rows_lse.append(math.log(den))
    elif name == "above_one" and mask == [0, 1, 0]:
        # kept: tile 0 (row i: sqrt(128) on key i) and tile 2 (1.5 sqrt(128) on key 256 + i)
        E0 = math.exp(math.sqrt(128.0))
        E2 = math.exp(1.5 * math.sqrt(128.0))
        tile0, tile2 = vv[0:128], vv[256:384]
        for i in range(Sq):
            num = E0 * tile0[i] + E2 * tile2[i] + (tile0.sum(0) - tile0[i]) + (tile2.sum(0) - tile2[i])
            den = E0 + E2 + 254
            rows_o.append(num / den)
            rows_lse.append(math.log(den))
    else:
        return None
    return np.array(rows_o), np.array(rows_lse)
