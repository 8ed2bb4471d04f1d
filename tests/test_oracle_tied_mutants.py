"""Plant plausible mistakes in a copy of the tied-covariance oracle and check
that its pins catch every one of them (CPU only; the real oracle is never
modified).  Each mutant replaces one exact snippet of ``oracle/tied.py``; the
test first checks that the snippet is present."""
import importlib.util
import os

import numpy as np
import pytest

import oracle
import oracle_tied_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "tied.py")

MUTANTS = {
    "drop_log_det": ("D * LOG_2PI + logdet + (z * z).sum(0)", "D * LOG_2PI + (z * z).sum(0)"),
    "missing_half": ("ell[:, k] = lw[k] - 0.5 * (", "ell[:, k] = lw[k] - 1.0 * ("),
    "upper_factor_solve": ("z = solve_triangular(L, (X - mu[k]).T, lower=True)",
                           "z = solve_triangular(L.T, (X - mu[k]).T, lower=False)"),
    "responsibility_sign": ("r = np.exp(ell - lse[:, None])\n    Nk", "r = np.exp(lse[:, None] - ell)\n    Nk"),
    "weights_not_normalised": ("np.log(np.maximum(Nk, EMPTY_NK) / N)", "np.log(np.maximum(Nk, EMPTY_NK))"),
    "first_moment_unweighted": ("new_mu[live] = (r[:, live].T @ X) / Nk[live, None]",
                                "new_mu[live] = X.mean(0)"),
    "covariance_about_old_mean": ("diff = X - new_mu[k]", "diff = X - mu[k]"),
    "covariance_unbiased": ("S /= N", "S /= N - 1"),
    "covariance_unweighted": ("S += (diff * r[:, k:k + 1]).T @ diff", "S += diff.T @ diff / len(Nk)"),
    "reg_on_every_entry": ("S[d, d] = np.maximum(S[d, d], var_floor) + reg_covar",
                           "S = np.maximum(S, var_floor) + reg_covar"),
}


def _load_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"snippet for mutant {name} not found in the tied oracle"
    path = tmp_path / f"tied_{name}.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"tied_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_tied_mutant_is_caught(name, tmp_path):
    mutant = _load_mutant(name, tmp_path)
    caught = []
    for pin in P.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mutant)
        except (AssertionError, FloatingPointError, ValueError, np.linalg.LinAlgError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {name}"
