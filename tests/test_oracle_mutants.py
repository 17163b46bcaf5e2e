"""Plant plausible mistakes in a copy of the CPU oracle and check that the pins catch each.

Every mutant is the oracle's C source with one textual change, compiled into a
temporary library on the CPU. The pins of ``test_oracle_pins.py`` are then run
against it; at least one must fail. The real oracle is never modified.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "blasst_oracle.c")

MUTANTS = {
    # skip when ANY row passes instead of every row ("Algorithm": all rows)
    "any_row_rule": ("if (g > worst)", "if (g < worst || worst == -INFINITY)"),
    # scores without the scale (docs.vllm.ai: Q . K_j^T . scale)
    "drop_scale": ("scale * dot_row(qrow", "dot_row(qrow"),
    # lambda normalised by the query length instead of the KV length
    "lambda_over_sq": ("log(factor / (double)Sk)", "log(factor / (double)Sq)"),
    # rescale factor with the wrong sign
    "alpha_sign": ("exp(m[i] - m_new)", "exp(m_new - m[i])"),
    # forget to rescale the running numerator when m grows
    "no_o_rescale": ("acc[(size_t)i * d + t] *= alpha;", ";"),
    # V read from K
    "v_from_k": ("const uint16_t *vr = v + row_offset", "const uint16_t *vr = k + row_offset"),
    # log-sum-exp in base 2
    "lse_log2": ("m[i] + log(l[i])", "m[i] + log2(l[i])"),
    # inverted test
    "inverted_test": ("(worst < ln_lambda)", "(worst > ln_lambda)"),
    # max_prob as l instead of 1 / l
    "max_prob_inverted": ("= 1.0 / l[i];", "= l[i];"),
    # a non-strict test: a gap equal to ln(lambda) would skip ("Algorithm": strictly below)
    "non_strict_test": ("(worst < ln_lambda)", "(worst <= ln_lambda)"),
    # a skipped tile raises the running max ("Algorithm": a skipped tile changes nothing);
    # visible only for lambda > 1, where a skipped tile's maximum can exceed it
    "skipped_tile_moves_max": ("continue; /* the tile's contribution to l and O is omitted */",
                               "{ for (int i2 = 0; i2 < nr; ++i2) if (tile_max[i2] > m[i2]) m[i2] = tile_max[i2]; "
                               "continue; }"),
}


def _compile_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path_c = tmp_path / f"{name}.c"
    path_so = tmp_path / f"{name}.so"
    path_c.write_text(src.replace(old, new))
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           str(path_c), "-o", str(path_so), "-lm"])
    return oracle.load_library(str(path_so))


def _pin_checks():
    yield lambda: pins.test_factor_zero_is_dense_attention(*pins.SMALL_CASES[1])
    yield lambda: pins.test_factor_zero_is_dense_attention(*pins.SMALL_CASES[2])
    yield lambda: pins.test_mask_matches_prefix_max_closed_form(*pins.CLOSED_FORM_CASES[0])
    for case in pins._load_golden():
        yield lambda case=case: pins.test_hand_built_case_skips_predicted_tiles(case)
    yield lambda: pins.test_max_prob_is_the_largest_kept_softmax_weight(20.0)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, monkeypatch, name):
    monkeypatch.setattr(oracle, "_lib", _compile_mutant(tmp_path, name))
    caught = 0
    with np.errstate(all="ignore"):
        for check in _pin_checks():
            try:
                check()
            except (AssertionError, ValueError, FloatingPointError):
                caught += 1
    assert caught > 0, f"no pin detects the planted mistake '{name}'"


def test_unmutated_copy_passes_every_pin(tmp_path, monkeypatch):
    path_so = tmp_path / "clean.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           SRC, "-o", str(path_so), "-lm"])
    monkeypatch.setattr(oracle, "_lib", oracle.load_library(str(path_so)))
    for check in _pin_checks():
        check()
