"""Checks that pin the float64 oracle to facts fixed outside the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` instance and raises
AssertionError when the oracle disagrees with the fact it checks.  They are
run against the real oracle (test_oracle_pins.py) and against deliberately
broken copies of it (test_oracle_mutants.py), which shows that a plausible
slip anywhere in the oracle is caught by at least one of them.

What pins what:
  pin_bayes        E-step and log-likelihood against Bayes' rule with the
                   Gaussian density written as a product of 1-D pdfs, summed
                   in 40-digit arithmetic (no logs, no max shift).
  pin_sum_to_one   responsibilities form a probability vector per point
                   ("ML0094 GMM vs K-Means", hard vs soft assignment).
  pin_k1           K = 1: the M-step is the sample mean and the biased sample
                   variance (numpy.mean / numpy.var); the log-likelihood is a
                   sum of scipy.stats.norm.logpdf values.
  pin_moments      conservation laws that hold for any responsibilities
                   summing to 1: sum_k pi_k = 1, sum_k N_k mu_k = sum_i x_i,
                   sum_k N_k (s2_k + mu_k^2) = sum_i x_i^2 (variance about the
                   new mean).
  pin_kmeans       the k-means limit ("ML0094 GMM vs K-Means": shared spherical
                   variance going to zero, equal weights): argmax r equals the
                   nearest centre, and the M-step mean is Lloyd's update.
  pin_sklearn      one warm-started iteration of scikit-learn's
                   GaussianMixture (an independent implementation).
  pin_monotone     EM never decreases the log-likelihood (reg_covar = 0).
  pin_recovery     a well separated mixture is recovered to within a few
                   standard errors.
  pin_topm         top-m selection equals a full stable sort of the
                   responsibilities; equal responsibilities go to the lower
                   component index.
  pin_empty        a component with weight 0 keeps its parameters and does not
                   change the others' update.
  pin_floor        var_floor is applied before reg_covar.
"""
from __future__ import annotations

import warnings

import numpy as np

RNG_SEED = 12345


def _problem(N, D, K, seed, spread=(0.6, 1.4), scale=2.0, spherical=False):
    rng = np.random.default_rng(seed)
    centres = rng.normal(0.0, scale, size=(K, D))
    lab = rng.integers(0, K, size=N)
    sd = rng.uniform(*spread, size=(K, D))
    X = (centres[lab] + sd[lab] * rng.normal(size=(N, D))).astype(np.float32)
    means = centres + rng.normal(0.0, 0.5, size=(K, D))
    w = rng.dirichlet(np.ones(K))
    if spherical:
        var = rng.uniform(0.5, 2.0, size=K)
    else:
        var = rng.uniform(0.5, 2.0, size=(K, D))
    return X, np.log(w), means, var


# ---------------------------------------------------------------------------
def pin_bayes(o):
    import mpmath as mp
    mp.mp.dps = 40
    for cov in ("diag", "spherical"):
        X, lw, mu, var = _problem(10, 3, 4, RNG_SEED + 1, spherical=(cov == "spherical"),
                                  scale=0.8)
        N, D = X.shape
        K = mu.shape[0]
        r_ref = np.zeros((N, K))
        ll_ref = mp.mpf(0)
        for i in range(N):
            joint = []
            for k in range(K):
                dens = mp.mpf(1)
                for d in range(D):
                    v = mp.mpf(float(var[k] if cov == "spherical" else var[k, d]))
                    diff = mp.mpf(float(X[i, d])) - mp.mpf(float(mu[k, d]))
                    dens *= mp.exp(-diff * diff / (2 * v)) / mp.sqrt(2 * mp.pi * v)
                joint.append(mp.exp(mp.mpf(float(lw[k]))) * dens)
            p = mp.fsum(joint)
            ll_ref += mp.log(p)
            for k in range(K):
                r_ref[i, k] = float(joint[k] / p)
        r, lse = o.responsibilities(X, lw, mu, var, cov)
        np.testing.assert_allclose(r, r_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse.sum(), float(ll_ref), rtol=1e-12)
        _, _, _, ll = o.em_step(X, lw, mu, var, cov)
        np.testing.assert_allclose(ll, float(ll_ref), rtol=1e-12)


def pin_sum_to_one(o):
    for cov in ("diag", "spherical"):
        X, lw, mu, var = _problem(500, 5, 7, RNG_SEED + 2, spherical=(cov == "spherical"))
        r, _ = o.responsibilities(X, lw, mu, var, cov)
        assert np.all(r >= 0)
        np.testing.assert_allclose(r.sum(1), 1.0, rtol=0, atol=1e-12)


def pin_k1(o):
    from scipy.stats import norm
    rng = np.random.default_rng(RNG_SEED + 3)
    X = (rng.normal(size=(1000, 6)) * [1, 2, 3, 0.5, 1, 4] + [1, -2, 3, 0, 5, -1]).astype(np.float32)
    Xd = X.astype(np.float64)
    reg = 1e-6
    mu0 = rng.normal(size=(1, 6))
    # diagonal
    var0 = rng.uniform(0.5, 3.0, size=(1, 6))
    lw, mu, var, ll = o.em_step(X, [0.0], mu0, var0, "diag", reg_covar=reg)
    np.testing.assert_allclose(lw, [0.0], atol=1e-12)
    np.testing.assert_allclose(mu[0], np.mean(Xd, axis=0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(var[0], np.var(Xd, axis=0) + reg, rtol=1e-10)
    ll_ref = norm.logpdf(Xd, loc=mu0[0], scale=np.sqrt(var0[0])).sum()
    np.testing.assert_allclose(ll, ll_ref, rtol=1e-12)
    # spherical
    s0 = np.array([1.7])
    lw, mu, var, ll = o.em_step(X, [0.0], mu0, s0, "spherical", reg_covar=reg)
    np.testing.assert_allclose(mu[0], np.mean(Xd, axis=0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(var[0], np.var(Xd - np.mean(Xd, axis=0)) + reg, rtol=1e-10)
    ll_ref = norm.logpdf(Xd, loc=mu0[0], scale=np.sqrt(s0[0])).sum()
    np.testing.assert_allclose(ll, ll_ref, rtol=1e-12)


def pin_moments(o):
    reg = 1e-3
    for cov in ("diag", "spherical"):
        X, lw, mu, var = _problem(800, 5, 6, RNG_SEED + 4, spherical=(cov == "spherical"))
        Xd = X.astype(np.float64)
        N, D = X.shape
        lw2, mu2, var2, _ = o.em_step(X, lw, mu, var, cov, reg_covar=reg)
        Nk = np.exp(lw2) * N
        np.testing.assert_allclose(np.exp(lw2).sum(), 1.0, rtol=1e-12)
        np.testing.assert_allclose((Nk[:, None] * mu2).sum(0), Xd.sum(0), rtol=1e-10, atol=1e-8)
        if cov == "diag":
            second = (Nk[:, None] * (var2 - reg + mu2 ** 2)).sum(0)
            np.testing.assert_allclose(second, (Xd ** 2).sum(0), rtol=1e-10)
        else:
            second = (Nk * (D * (var2 - reg) + (mu2 ** 2).sum(1))).sum()
            np.testing.assert_allclose(second, (Xd ** 2).sum(), rtol=1e-10)


def pin_kmeans(o):
    rng = np.random.default_rng(RNG_SEED + 5)
    K, D, N = 5, 4, 600
    X = rng.normal(0, 3.0, size=(N, D)).astype(np.float32)
    Xd = X.astype(np.float64)
    mu = rng.normal(0, 3.0, size=(K, D))
    lw = np.full(K, -np.log(K))
    var = np.full(K, 1e-6 * 9.0)
    r, _ = o.responsibilities(X, lw, mu, var, "spherical")
    dist = ((Xd[:, None, :] - mu[None]) ** 2).sum(-1)
    near = dist.argmin(1)
    np.testing.assert_array_equal(r.argmax(1), near)
    lw2, mu2, _, _ = o.em_step(X, lw, mu, var, "spherical")
    counts = np.bincount(near, minlength=K)
    np.testing.assert_allclose(np.exp(lw2) * N, counts, rtol=1e-9)
    for k in range(K):
        if counts[k]:
            np.testing.assert_allclose(mu2[k], Xd[near == k].mean(0), rtol=1e-9, atol=1e-9)


def pin_sklearn(o):
    from sklearn.exceptions import ConvergenceWarning
    from sklearn.mixture import GaussianMixture
    for cov in ("diag", "spherical"):
        X, lw, mu, var = _problem(2000, 4, 5, RNG_SEED + 6, spherical=(cov == "spherical"))
        lw = lw - np.log(np.exp(lw).sum())
        reg = 1e-6
        gm = GaussianMixture(n_components=5, covariance_type=cov, max_iter=1, tol=0.0,
                             reg_covar=reg, weights_init=np.exp(lw), means_init=mu,
                             precisions_init=1.0 / var, init_params="random")
        with warnings.catch_warnings():
            warnings.simplefilter("ignore", ConvergenceWarning)
            gm.fit(X.astype(np.float64))
        lw2, mu2, var2, ll = o.em_step(X, lw, mu, var, cov, reg_covar=reg)
        np.testing.assert_allclose(np.exp(lw2), gm.weights_, rtol=1e-9)
        np.testing.assert_allclose(mu2, gm.means_, rtol=1e-9, atol=1e-10)
        np.testing.assert_allclose(var2, gm.covariances_, rtol=1e-9)
        np.testing.assert_allclose(ll / X.shape[0], gm.lower_bound_, rtol=1e-9)


def pin_monotone(o, X=None, init=None, cov="diag", iters=20, var_floor=1e-3):
    # reg_covar = 0 and a variance floor: the floored update is still the exact
    # maximiser of the EM auxiliary function over variances >= var_floor, so the
    # monotone property holds without exception.
    if X is None:
        X, lw, mu, var = _problem(1500, 3, 6, RNG_SEED + 7)
        init = (lw, mu, var)
    *_, lls = o.em_run(X, *init, cov, iters, reg_covar=0.0, var_floor=var_floor)
    lls = np.asarray(lls)
    assert np.all(np.isfinite(lls))
    drops = lls[:-1] - lls[1:]
    assert np.all(drops <= 1e-10 * np.abs(lls[:-1])), (lls, drops.max())
    return lls


def pin_recovery(o):
    rng = np.random.default_rng(RNG_SEED + 8)
    K, D, n_per = 6, 5, 4000
    centres = rng.uniform(-30, 30, size=(K, D))
    sd = rng.uniform(0.5, 2.0, size=(K, D))
    lab = np.repeat(np.arange(K), n_per)
    X = (centres[lab] + sd[lab] * rng.normal(size=(K * n_per, D))).astype(np.float32)
    # one data point of each true component as its starting mean
    first = np.array([np.flatnonzero(lab == k)[7] for k in range(K)])
    init = (np.full(K, -np.log(K)), X[first].astype(np.float64), np.ones((K, D)))
    lw, mu, var, _ = o.em_run(X, *init, "diag", 20)
    se = sd / np.sqrt(n_per)
    z = np.abs(mu - centres) / se
    assert z.max() < 6.0, z.max()                       # means within 6 standard errors
    np.testing.assert_allclose(np.sqrt(var), sd, rtol=0.1)  # spreads within 10%
    np.testing.assert_allclose(np.exp(lw), 1.0 / K, rtol=0.01)


def pin_topm(o):
    import mpmath as mp
    mp.mp.dps = 30
    X, lw, mu, var = _problem(300, 4, 9, RNG_SEED + 9, scale=1.0)
    r_full, lse = o.responsibilities(X, lw, mu, var, "diag")
    for m in (1, 3, 9):
        r, idx, ll = o.topm(X, lw, mu, var, "diag", m)
        order = np.argsort(-r_full, axis=1, kind="stable")[:, :m]
        np.testing.assert_array_equal(idx, order)
        np.testing.assert_allclose(r, np.take_along_axis(r_full, order, 1), rtol=1e-14, atol=0)
        np.testing.assert_allclose(ll, lse.sum(), rtol=1e-14)
        assert np.all(np.diff(r, axis=1) <= 0)
    # equal components: components 1, 3 and 4 are copies of one another
    mu2, var2, lw2 = mu.copy(), var.copy(), lw.copy()
    for k in (3, 4):
        mu2[k], var2[k], lw2[k] = mu2[1], var2[1], lw2[1]
    r, idx, _ = o.topm(X, lw2, mu2, var2, "diag", 9)
    for i in range(X.shape[0]):
        pos = [list(idx[i]).index(k) for k in (1, 3, 4)]
        assert pos == sorted(pos) and pos[2] - pos[0] == 2, (idx[i], pos)
        assert r[i, pos[0]] == r[i, pos[1]] == r[i, pos[2]]


def pin_empty(o):
    X, lw, mu, var = _problem(700, 3, 5, RNG_SEED + 10)
    lw_dead = lw.copy()
    lw_dead[2] = -np.inf
    lw2, mu2, var2, ll = o.em_step(X, lw_dead, mu, var, "diag")
    assert lw2[2] == -np.inf
    np.testing.assert_array_equal(mu2[2], mu[2])
    np.testing.assert_array_equal(var2[2], var[2])
    keep = [0, 1, 3, 4]
    lw3, mu3, var3, ll3 = o.em_step(X, lw[keep], mu[keep], var[keep], "diag")
    np.testing.assert_allclose(lw2[keep], lw3, rtol=1e-12)
    np.testing.assert_allclose(mu2[keep], mu3, rtol=1e-12)
    np.testing.assert_allclose(var2[keep], var3, rtol=1e-12)
    np.testing.assert_allclose(ll, ll3, rtol=1e-12)


def pin_floor(o):
    X, lw, mu, var = _problem(400, 3, 4, RNG_SEED + 11)
    _, _, v0, _ = o.em_step(X, lw, mu, var, "diag", reg_covar=1e-3, var_floor=0.0)
    floor = float(np.median(v0))
    _, _, v1, _ = o.em_step(X, lw, mu, var, "diag", reg_covar=1e-3, var_floor=floor)
    np.testing.assert_allclose(v1, np.maximum(v0 - 1e-3, floor) + 1e-3, rtol=1e-12)


ALL_PINS = [pin_bayes, pin_sum_to_one, pin_k1, pin_moments, pin_kmeans, pin_sklearn,
            pin_monotone, pin_recovery, pin_topm, pin_empty, pin_floor]
