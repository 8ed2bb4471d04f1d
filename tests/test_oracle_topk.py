"""The approximate top-k EM oracle against its pins, and planted mistakes in
a copy of it that must each fail a pin (CPU only)."""
import importlib.util
import os

import numpy as np
import pytest

import oracle
import oracle_topk_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "topk_em.py")


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_topk_oracle_pin(pin):
    pin(oracle.topk_em)


MUTANTS = {
    "largest_k_reversed": ("np.lexsort((np.broadcast_to(np.arange(K), ell.shape), -ell), axis=1)[:, :k]",
                           "np.lexsort((np.broadcast_to(np.arange(K), ell.shape), ell), axis=1)[:, :k]"),
    "ties_to_higher_index": ("np.lexsort((np.broadcast_to(np.arange(K), ell.shape), -ell), axis=1)[:, :k]",
                             "np.lexsort((-np.broadcast_to(np.arange(K), ell.shape), -ell), axis=1)[:, :k]"),
    "normalised_over_all": ("r = np.where(keep, np.exp(sub - lse_k[:, None]), 0.0)",
                            "r = np.where(keep, np.exp(sub - lse_all[:, None]), 0.0)"),
    "k_plus_one_kept": ("axis=1)[:, :k]", "axis=1)[:, :k + 1]"),
    "loglik_of_the_subset": ("return r, lse_all\n\n\ndef em_step", "return r, lse_k\n\n\ndef em_step"),
    "variance_about_old_mean": ("diff = X - new_mu[j]", "diff = X - mu[j]"),
    "weights_not_normalised": ("np.log(np.maximum(Nk, EMPTY_NK) / N)", "np.log(np.maximum(Nk, EMPTY_NK))"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_topk_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / f"topk_{name}.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"topk_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    caught = []
    for pin in P.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {name}"
