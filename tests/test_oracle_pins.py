"""The oracle against what the method and the mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
import oracle_pins as P
import workloads as W


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


# EM never decreases the likelihood, on a prefix of every workload with its
# own K, D, covariance type and starting parameters (reg_covar = 0, variance
# floor at 1e-3 of the data's mean per-dimension variance).
@pytest.mark.parametrize("name,rows,iters", [
    ("tiny_diag", 4096, 20),
    ("spherical_1m", 4000, 10),
    ("embed_10m", 2000, 6),
    ("descriptor_100m", 2000, 6),
    ("largek_2m", 8192, 2),
])
def test_monotone_on_workloads(orc, name, rows, iters):
    w = W.WORKLOADS[name].scaled(rows)
    X = W.make_data(w)
    init = W.make_init(w, X)
    Xf = X.float().numpy()
    floor = 1e-3 * float(Xf.astype(np.float64).var(0).mean())
    lls = P.pin_monotone(orc, Xf, init, w.cov, iters, var_floor=floor)
    assert lls[-1] > lls[0]


def test_prefix_property():
    w = W.WORKLOADS["embed_10m"]
    a = W.make_data(w, 300)
    b = W.make_data(w, 1000)
    assert a.dtype == b.dtype and bool((a == b[:300]).all())


def test_threads_reported(orc):
    assert orc.threads() >= 1
    assert orc.threads(2) == 2


def test_oracle_rejects_bad_args(orc):
    X = np.zeros((4, 2), np.float32)
    with pytest.raises(AssertionError):
        orc.topm(X, [0.0], np.zeros((1, 2)), np.ones((1, 2)), "diag", 2)  # m > K
