"""The weight-gradient oracle against its pins, and planted mistakes in it that the
pins must each catch (CPU only; mutants run in a subprocess)."""
import os
import subprocess
import sys

import pytest

from oracle import wgrad as ow
from tests import oracle_wgrad_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "conv2d_wgrad.c")
PINS = os.path.join(ROOT, "tests", "oracle_wgrad_pins.py")


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_wgrad_pin(pin):
    pin(ow.load())


MUTANTS = {
    "padding_sign_h": ("p * sp->sh - sp->ph + r * sp->dh", "p * sp->sh + sp->ph + r * sp->dh"),
    "stride_for_dilation_w": ("q * sp->sw - sp->pw + s * sp->dw", "q * sp->sw - sp->pw + s * sp->sw"),
    "dy_channel_shifted": ("* sp->q + q) * sp->k + k]", "* sp->q + q) * sp->k + (k + 1) % sp->k]"),
    "group_offset_dropped": ("(k / (sp->k / sp->g)) * (sp->c / sp->g) + c", "c"),
    "border_off_by_one": ("if (ih < 0 || ih >= sp->h) continue;", "if (ih < 0 || ih > sp->h - 2) continue;"),
    "gradient_r_s_swapped": ("((k * sp->r + r) * sp->s + s) * cg + c", "((k * sp->r + s) * sp->s + r) * cg + c"),
    "thread_block_gap": ("jobs[t].k_end = sp.k * (t + 1) / threads;",
                         "jobs[t].k_end = sp.k * (t + 1) / threads - (t == 1);"),
    "bf16_shift_wrong": ("(uint32_t)b << 16", "(uint32_t)b << 15"),
    "points_tap_decode": ("rs / sp.s, rs % sp.s", "rs % sp.s, rs / sp.s"),
    "mass_signed": ("mass += t < 0 ? -t : t;", "mass += t;"),
    "extent_missing_plus_one": ("return room < 0 ? 0 : room / stride + 1;", "return room < 0 ? 0 : room / stride;"),
    "input_row_for_column": ("x[((n * sp->h + ih) * sp->w + iw) * sp->c + cin]",
                             "x[((n * sp->h + iw % sp->h) * sp->w + ih % sp->w) * sp->c + cin]"),
}


def test_unmutated_wgrad_oracle_passes_battery(tmp_path):
    lib = ow.compile_library(SRC, str(tmp_path / "orig.so"))
    res = subprocess.run([sys.executable, PINS, lib], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_wgrad_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} no longer unique in the oracle"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = ow.compile_library(str(mutated), str(tmp_path / "mutant.so"))
    res = subprocess.run([sys.executable, PINS, lib], capture_output=True, text=True, timeout=300)
    assert res.returncode != 0, f"mutant {name} survived every pin:\n{res.stdout}{res.stderr}"
