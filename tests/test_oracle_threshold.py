"""Pins of the oracle's threshold multi-assignment (CPU only).  The function
restates its definition ("Flash-GMM", conclusion: border vectors assigned to
several clusters from the responsibilities); these checks tie it to a
hand-computed case with ties and to properties that follow from the
responsibilities of a point summing to one.  Each pin also runs on copies of
the function with a planted mistake, and every copy must fail one of them."""
import inspect

import numpy as np
import pytest

import oracle
import workloads as W


def pin_hand_computed_case_with_ties(fn):
    r = np.array([[0.5, 0.5, 0.0],
                  [0.2, 0.3, 0.5],
                  [0.1, 0.1, 0.8]])
    off, idx, resp = fn(r, 0.3, 16)
    assert off.tolist() == [0, 2, 4, 5]
    assert idx.tolist() == [0, 1, 2, 1, 2]           # equal values: lower index first
    assert np.allclose(resp, [0.5, 0.5, 0.5, 0.3, 0.8])
    off, idx, _ = fn(r, 0.3, 1)  # capped at one per point
    assert off.tolist() == [0, 1, 2, 3] and idx.tolist() == [0, 2, 2]


def _resp(seed=0, N=300, D=6, K=9):
    w = W.generic(N, D, K, "diag", "f32", seed=seed)
    X = W.make_data(w)
    lw, mu, var = W.make_init(w, X)
    return oracle.responsibilities(X.numpy(), lw, mu, var, "diag")[0]


def pin_properties_on_real_responsibilities(fn):
    r = _resp()
    N, K = r.shape
    for tau, m in ((0.05, 16), (0.2, 4), (0.34, 2), (0.6, 1)):
        off, idx, resp = fn(r, tau, m)
        assert off[0] == 0 and np.all(np.diff(off) >= 0) and off[-1] == len(idx)
        for i in range(N):
            ks = idx[off[i]:off[i + 1]]
            assert len(ks) <= m and np.all(r[i, ks] >= tau)
            assert np.all(np.diff(r[i, ks]) <= 0)                     # descending
            if tau > 1.0 / (m + 1):                                  # nothing is cut by the cap
                assert set(ks.tolist()) == set(np.nonzero(r[i] >= tau)[0].tolist())
            assert np.allclose(resp[off[i]:off[i + 1]], r[i, ks])


def pin_tiny_threshold_gives_every_component_in_order(fn):
    r = _resp(seed=1, N=50, K=7)
    off, idx, _ = fn(r, 1e-300, 7)
    kept = r >= 1e-300
    assert off[-1] == kept.sum()
    for i in range(len(r)):
        ks = idx[off[i]:off[i + 1]]
        order = [k for k in np.lexsort((np.arange(7), -r[i])) if kept[i, k]]
        assert ks.tolist() == order


def pin_threshold_above_one_half_keeps_the_argmax_or_nothing(fn):
    r = _resp(seed=2)
    off, idx, _ = fn(r, 0.5 + 1e-9, 16)
    for i in range(len(r)):
        ks = idx[off[i]:off[i + 1]]
        if r[i].max() >= 0.5 + 1e-9:
            assert ks.tolist() == [int(np.argmax(r[i]))]
        else:
            assert len(ks) == 0


PINS = [pin_hand_computed_case_with_ties, pin_properties_on_real_responsibilities,
        pin_tiny_threshold_gives_every_component_in_order, pin_threshold_above_one_half_keeps_the_argmax_or_nothing]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_threshold_oracle_pin(pin):
    pin(oracle.threshold_assign)


MUTANTS = {
    "strict_threshold": ("if row[k] >= tau", "if row[k] > tau"),
    "ties_to_higher_index": ("key=lambda k: (-row[k], k)", "key=lambda k: (-row[k], -k)"),
    "ascending_order": ("key=lambda k: (-row[k], k)", "key=lambda k: (row[k], k)"),
    "cap_ignored": ("[:max_per_point]", ""),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_threshold_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = inspect.getsource(oracle.threshold_assign)
    assert src.count(old) == 1, name
    ns = {"np": np}
    exec(src.replace(old, new), ns)
    caught = []
    for pin in PINS:
        try:
            pin(ns["threshold_assign"])
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {name}"
