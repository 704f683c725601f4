"""The pins have teeth: copies of the C oracle with one planted mistake each
(compiled into a temporary directory, on the CPU) must each fail at least one
pin. The committed oracle is never modified."""
import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")

# (name, text in the committed source, planted replacement)
MUTANTS = [
    ("drop_D_term", "acc + D[h] * xt[p]", "acc"),
    ("D_times_u", "acc + D[h] * xt[p]", "acc + D[h] * u"),
    ("A_sign_flipped", "exp(dtv * A[h])", "exp(-dtv * A[h])"),
    ("no_dt_on_input", "const double u = dtv * xt[p];", "const double u = xt[p];"),
    ("exact_zoh_input", "const double u = dtv * xt[p];", "const double u = (a - 1.0) / A[h] * xt[p];"),
    ("y_before_update", "row[n] = a * row[n] + u * Bt[n];\n                        acc += Ct[n] * row[n];",
     "acc += Ct[n] * row[n];\n                        row[n] = a * row[n] + u * Bt[n];"),
    ("B_C_swapped_in_update", "u * Bt[n]", "u * Ct[n]"),
    ("snapshot_off_by_one", "t + 1 == j", "t == j"),
    ("group_interleaved", "h / heads_per_group", "h % G"),
    ("dt_layout_transposed", "dt[(b * K + t) * H + h]", "dt[(b * H + h) * K + t]"),
    ("no_restore_on_reject", "memcpy(S, S0, slice * sizeof(double)); /* j = 0, or invalid j */",
     "memset(S, 0, slice * sizeof(double));"),
    ("decay_not_applied", "row[n] = a * row[n] + u * Bt[n];", "row[n] = row[n] + u * Bt[n];"),
    ("C_from_next_group", "Cm + ((b * K + t) * G + g) * N", "Cm + ((b * K + t) * G + (g + 1) % G) * N"),
    ("invalid_j_not_reported", "int valid = (j >= 0 && j <= K);", "int valid = (j >= 0);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/present"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(lib), str(mpath),
                           "-lm"])
    run = oracle.Oracle(str(lib)).verify_commit
    failed = []
    for pin in ALL_PINS:
        try:
            pin(run)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
