"""Planted mistakes in the oracle must each fail at least one pin (CPU only).

Each mutant is a copy of ``oracle/conv2d_direct.c`` with one textual change,
compiled to a temporary library and run through the pin battery of
``tests/oracle_pins.py`` in a subprocess (so a mutant that reads out of bounds
cannot take the test process down).  The oracle itself is never modified.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "conv2d_direct.c")
PINS = os.path.join(ROOT, "tests", "oracle_pins.py")

MUTANTS = {
    "padding_sign_h": ("p * sp->sh - sp->ph + r * sp->dh", "p * sp->sh + sp->ph + r * sp->dh"),
    "stride_for_dilation_w": ("q * sp->sw - sp->pw + s * sp->dw", "q * sp->sw - sp->pw + s * sp->sw"),
    "dilation_for_stride_h": ("p * sp->sh - sp->ph + r * sp->dh", "p * sp->dh - sp->ph + r * sp->dh"),
    "filter_transposed": ("((k * sp->r + r) * sp->s + s)", "((k * sp->r + s) * sp->s + r)"),
    "filter_flipped": ("((k * sp->r + r) * sp->s + s)",
                       "((k * sp->r + (sp->r - 1 - r)) * sp->s + (sp->s - 1 - s))"),
    "input_hw_swapped": ("((n * sp->h + ih) * sp->w + iw)", "((n * sp->w + iw) * sp->h + ih)"),
    "bias_dropped": ("bias ? (double)bias[k] : 0.0", "0.0"),
    "bias_wrong_channel": ("bias ? (double)bias[k] : 0.0", "bias ? (double)bias[0] : 0.0"),
    "first_channel_dropped": ("for (int64_t c = 0; c < cg; ++c)", "for (int64_t c = 1; c < cg; ++c)"),
    "group_channel_offset_dropped": ("* sp->c + group * cg;", "* sp->c;"),
    "group_weight_row_stride_full_c": ("* sp->s + s) * cg;", "* sp->s + s) * sp->c;"),
    "groups_interleaved": ("k / (sp->k / sp->g)", "k % sp->g"),
    "border_off_by_one": ("if (ih < 0 || ih >= sp->h) continue;", "if (ih <= 0 || ih >= sp->h) continue;"),
    "extent_missing_plus_one": ("return room / stride + 1;", "return room / stride;"),
    "extent_span_wrong": ("int64_t span = dil * (ker - 1) + 1;", "int64_t span = dil * ker;"),
    "bf16_shift_wrong": ("(uint32_t)b << 16", "(uint32_t)b << 15"),
    "thread_block_gap": ("jobs[t].row_end = rows * (t + 1) / threads;",
                         "jobs[t].row_end = rows * (t + 1) / threads - (t == 1);"),
    "points_q_index": ("int64_t q = m % sp->q;", "int64_t q = m % sp->p;"),
    "output_k_stride": ("* sp->q + q) * sp->k + k]", "* sp->q + q) * sp->k + (k + 1) % sp->k]"),
}


def test_unmutated_oracle_passes_battery(tmp_path):
    lib = oracle.compile_library(SRC, str(tmp_path / "orig.so"))
    res = subprocess.run([sys.executable, PINS, lib], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} no longer unique in the oracle"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(mutated), str(tmp_path / "mutant.so"))
    res = subprocess.run([sys.executable, PINS, lib], capture_output=True, text=True, timeout=300)
    assert res.returncode != 0, f"mutant {name} survived every pin:\n{res.stdout}{res.stderr}"
