"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them (CPU only; the real oracle is never modified).

Each mutant replaces one exact snippet of ``oracle/gmm_oracle.c``; the test
first checks that the snippet is present, so a change to the oracle that
silently disarms a mutant fails here too."""
import os
import subprocess

import pytest

import oracle
import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "gmm_oracle.c")

MUTANTS = {
    "drop_log_2pi": ("s += log(v) + LOG_2PI + diff * diff / v;",
                     "s += log(v) + diff * diff / v;"),
    "drop_log_det": ("s += log(v) + LOG_2PI + diff * diff / v;",
                     "s += LOG_2PI + diff * diff / v;"),
    "sign_of_difference": ("double diff = (double)x[d] - means[k * D + d];",
                           "double diff = (double)x[d] + means[k * D + d];"),
    "wrong_dimension_index": ("double diff = (double)x[d] - means[k * D + d];",
                              "double diff = (double)x[0] - means[k * D + d];"),
    "missing_half": ("return log_weights[k] - 0.5 * s;",
                     "return log_weights[k] - s;"),
    "diag_reads_spherical_slot": ("cov == ORACLE_SPHERICAL ? vars[k] : vars[k * D + d];",
                                  "vars[k];"),
    "lse_without_max": ("return mx + log(sum);", "return log(sum);"),
    "responsibility_sign": ("double r = exp(ell[k] - lse);\n                Nk[k] += r;",
                            "double r = exp(lse - ell[k]);\n                Nk[k] += r;"),
    "variance_about_old_mean": ("double diff = (double)x[d] - new_means[(int64_t)k * D + d];",
                                "double diff = (double)x[d] - means[(int64_t)k * D + d];"),
    "spherical_not_per_dimension": ("SV_t[k] / ((double)D * Nk[k])", "SV_t[k] / Nk[k]"),
    "weights_not_normalised": ("log(Nk[k] / (double)N)", "log(Nk[k])"),
    "reg_before_floor": ("v = (v > var_floor ? v : var_floor) + reg_covar;\n                new_vars[j] = v;",
                         "v = (v + reg_covar > var_floor ? v + reg_covar : var_floor);\n                new_vars[j] = v;"),
    "empty_rule_missing": ("new_means[j] = Nk[k] < ORACLE_EMPTY_NK ? means[j] : S1_t[j] / Nk[k];",
                           "new_means[j] = S1_t[j] / Nk[k];"),
    "topm_ascending": ("if (!taken[k] && (best < 0 || ell[k] > ell[best])) best = k;",
                       "if (!taken[k] && (best < 0 || ell[k] < ell[best])) best = k;"),
    "topm_ties_to_higher_index": ("if (!taken[k] && (best < 0 || ell[k] > ell[best])) best = k;",
                                  "if (!taken[k] && (best < 0 || ell[k] >= ell[best])) best = k;"),
    "first_moment_unweighted": ("S1[(int64_t)k * D + d] += r * (double)x[d];",
                                "S1[(int64_t)k * D + d] += (double)x[d] / K;"),
}


def _build_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"snippet for mutant {name} not found in the oracle"
    path_c = tmp_path / f"{name}.c"
    path_so = tmp_path / f"{name}.so"
    path_c.write_text(src.replace(old, new, 1))
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-o", str(path_so), str(path_c), "-lm"])
    return oracle.Oracle(str(path_so))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    mutant = _build_mutant(name, tmp_path)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, FloatingPointError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {name}"
