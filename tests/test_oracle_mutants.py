"""Planted mistakes: each plausible error in the oracle's arithmetic must make at least
one of its pins fail.  Every mutant is a copy of oracle/kda_oracle.c with one textual
change, compiled on the CPU into a temporary library that the oracle module is pointed
at for the duration of the check; the committed oracle is never touched.  Mutants stay
memory-safe (they never write more than the buffers the pins allocate)."""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

# (name, original text, planted text)
MUTANTS = [
    ("residual sign", "u[j] -= ki * row[j];", "u[j] += ki * row[j];"),
    ("decay dropped", "const double a = exp(log_alpha[i]);", "const double a = 1.0;"),
    ("output read before the update", "    /* o = S^T q */\n    if (o) {",
     "    /* o = S^T q */\n    if (o) { for (int i = 0; i < Dk; ++i) { const double c = beta * k[i]; "
     "double* row = S + (size_t)i * Dv; for (int j = 0; j < Dv; ++j) row[j] -= c * u[j]; }"),
    ("beta dropped from the write", "const double c = beta * k[i];", "const double c = k[i];"),
    ("transposed read", "o[j] += qi * row[j];", "o[j] += q[j] * S[(size_t)j * Dv + i];"),
    # (memory-safe: a mutant may write fewer checkpoint slots than the count, never more)
    ("checkpoint slot not advanced", "sizeof(double) * SS);\n                ++slot;", "sizeof(double) * SS);"),
]

# pins that exercise the recurrence and the checkpoint policy end to end
PIN_CHECKS = [
    pins.test_hand_worked_example_dk2_dv1,
    pins.test_hand_worked_example_scalar,
    lambda: pins.test_dense_brute_force(0),
    pins.test_delta_rule_exact_write,
    pins.test_beta_zero_is_pure_decay,
    pins.test_varlen_packing_and_checkpoints,
    pins.test_checkpoints_on_the_absolute_grid_enumerated,
]


def _build_mutant(tmp_path, original, planted):
    src = open(SRC).read()
    assert src.count(original) == 1, f"mutation anchor not unique: {original!r}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(original, planted))
    so = tmp_path / "mutant.so"
    # serial build (no OpenMP runtime shared with the real oracle)
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", str(so), str(path), "-lm"],
                   check=True)
    return oracle._declare(ctypes.CDLL(str(so)))


@pytest.mark.parametrize("name,original,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_each_planted_mistake_fails_a_pin(tmp_path, monkeypatch, name, original, planted):
    monkeypatch.setattr(oracle, "_lib", _build_mutant(tmp_path, original, planted))
    failed = []
    for check in PIN_CHECKS:
        try:
            check()
        except AssertionError:
            failed.append(getattr(check, "__name__", "brute force"))
    assert failed, f"no pin caught the planted mistake: {name}"


def test_the_unmutated_copy_passes(tmp_path, monkeypatch):
    """The same harness with no change: every pin passes (the harness itself is sound)."""
    monkeypatch.setattr(oracle, "_lib", _build_mutant(tmp_path, "u[j] -= ki * row[j];", "u[j] -= ki * row[j];"))
    for check in PIN_CHECKS:
        check()
