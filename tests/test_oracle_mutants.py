"""Plant single mistakes in copies of the oracle and check that the pins
catch each one (CPU only).  Shows the pins constrain every part of the
recurrence: decay index, update order, skip term, group map, B/C roles,
input scaling, state orientation and the snapshots."""
import functools
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")

MUTANTS = {
    "decay_uses_previous_dt": ("const double a = exp(dtv * a_h);",
                               "const double a = exp((t > 0 ? dt[(b * L + t - 1) * H + hd] : dtv) * a_h);"),
    "decay_without_dt": ("const double a = exp(dtv * a_h);", "const double a = exp(a_h);"),
    "output_reads_old_state": ("h[n] = a * h[n] + u * Bt[n];\n                    acc += Ct[n] * h[n];",
                               "acc += Ct[n] * h[n];\n                    h[n] = a * h[n] + u * Bt[n];"),
    "skip_term_dropped": ("y[((b * L + t) * H + hd) * P + p] = acc + d_h * xv;",
                          "y[((b * L + t) * H + hd) * P + p] = acc;"),
    "group_map_interleaved": ("const int64_t g = hd * G / H;", "const int64_t g = hd % G;"),
    "b_c_swapped": ("const double *Bt = B + ((b * L + t) * G + g) * N;\n                const double *Ct = C + ((b * L + t) * G + g) * N;",
                    "const double *Bt = C + ((b * L + t) * G + g) * N;\n                const double *Ct = B + ((b * L + t) * G + g) * N;"),
    "input_without_dt": ("const double u = dtv * xv;", "const double u = xv;"),
    "init_transposed": ("h[n] = init ? init[((b * H + hd) * P + p) * N + n] : 0.0;",
                        "h[n] = init ? init[((b * H + hd) * N + n) * P + p] : 0.0;"),
    "snapshot_after_update": ("if (snap && t % snap_every == 0) {", "if (snap && (t + 1) % snap_every == 0) {"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, mutant_dir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path_c = os.path.join(mutant_dir, f"{name}.c")
    path_so = os.path.join(mutant_dir, f"lib{name}.so")
    open(path_c, "w").write(src.replace(old, new))
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-shared", "-fPIC", path_c, "-o", path_so, "-lm"],
                   check=True)
    rec = functools.partial(oracle.ssd_recurrence, lib=oracle.open_library(path_so))
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(rec)
        except (AssertionError, FloatingPointError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
