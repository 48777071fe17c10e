"""The data-gradient oracle against its pins, and planted mistakes in it that the
pins must each catch (CPU only; mutants run in a subprocess)."""
import os
import subprocess
import sys

import pytest

from oracle import dgrad as od
from tests import oracle_dgrad_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "conv2d_dgrad.c")
PINS = os.path.join(ROOT, "tests", "oracle_dgrad_pins.py")


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_dgrad_pin(pin):
    pin(od.load())


MUTANTS = {
    "padding_sign_h": ("const int64_t th = h + sp->ph - r * sp->dh;", "const int64_t th = h - sp->ph - r * sp->dh;"),
    "tap_not_flipped_w": ("const int64_t tw = w + sp->pw - s * sp->dw;",
                          "const int64_t tw = w + sp->pw - (sp->s - 1 - s) * sp->dw;"),
    "stride_divisibility_ignored": ("if (th < 0 || th % sp->sh != 0) continue;", "if (th < 0) continue;"),
    "stride_not_divided": ("const int64_t p = th / sp->sh;", "const int64_t p = th;"),
    "upper_bound_off_by_one": ("if (q >= sp->q) continue;", "if (q >= sp->q - 1) continue;"),
    "group_k_range_whole": ("for (int64_t kk = grp * kg; kk < (grp + 1) * kg; ++kk)",
                            "for (int64_t kk = 0; kk < kg; ++kk)"),
    "group_from_output_channel_count": ("const int64_t grp = ci / cg;", "const int64_t grp = ci / kg;"),
    "weight_r_s_swapped": ("wt[((kk * sp->r + r) * sp->s + s) * cg + cw]", "wt[((kk * sp->r + s % sp->r) * sp->s + r % sp->s) * cg + cw]"),
    "thread_block_gap": ("jobs[t].row_end = rows * (t + 1) / threads;",
                         "jobs[t].row_end = rows * (t + 1) / threads - (t == 1);"),
    "bf16_shift_wrong": ("(uint32_t)b << 16", "(uint32_t)b << 15"),
    "points_h_decode": ("h = (m / sp.w) % sp.h", "h = (m / sp.w) % sp.w % sp.h"),
    "mass_signed": ("mass += t < 0 ? -t : t;", "mass += t;"),
}


def test_unmutated_dgrad_oracle_passes_battery(tmp_path):
    lib = od.compile_library(SRC, str(tmp_path / "orig.so"))
    res = subprocess.run([sys.executable, PINS, lib], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_dgrad_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} no longer unique in the oracle"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = od.compile_library(str(mutated), str(tmp_path / "mutant.so"))
    res = subprocess.run([sys.executable, PINS, lib], capture_output=True, text=True, timeout=300)
    assert res.returncode != 0, f"mutant {name} survived every pin:\n{res.stdout}{res.stderr}"
