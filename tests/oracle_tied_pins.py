"""Pins of the oracle's tied-covariance EM step, as functions of the module
that implements it (the real ``oracle.tied`` in test_oracle_tied.py, planted
mistakes in test_oracle_tied_mutants.py): special cases that reduce to
textbook routines or to the oracle's independent C paths, an invariance that
only a correct full-covariance treatment has, brute force on a tiny case, and
the monotone log-likelihood of EM."""
import numpy as np
from scipy.stats import multivariate_normal

import oracle


def _data(seed=0, N=400, D=4):
    rng = np.random.default_rng(seed)
    A = rng.normal(size=(D, D))
    X = rng.normal(size=(N, D)) @ A.T + rng.normal(size=D)
    return X


def _spd(D, seed=1):
    rng = np.random.default_rng(seed)
    A = rng.normal(size=(D, D))
    return A @ A.T + D * np.eye(D)


def pin_one_component_is_the_sample_mean_and_covariance(tied):
    X = _data()
    N, D = X.shape
    lw, mu, S, ll = tied.em_step(X, [0.0], X[:1], _spd(D), reg_covar=1e-6)
    assert lw[0] == 0.0
    assert np.allclose(mu[0], X.mean(0), rtol=1e-12, atol=1e-12)
    assert np.allclose(S, np.cov(X.T, bias=True) + 1e-6 * np.eye(D), rtol=1e-10, atol=1e-12)
    ll_ref = multivariate_normal(mean=X[0], cov=_spd(D)).logpdf(X).sum()
    assert abs(ll - ll_ref) <= 1e-9 * abs(ll_ref)


def pin_isotropic_and_diagonal_covariance_match_the_c_oracle(tied):
    X = _data(seed=2)
    N, D = X.shape
    K = 5
    lw = np.log(np.random.default_rng(3).dirichlet(np.ones(K)))
    mu = X[:K]
    # sigma^2 I: the spherical path with every sigma_k^2 = sigma^2
    r_s, lse_s = oracle.responsibilities(X.astype(np.float32), lw, mu, np.full(K, 2.5), "spherical")
    Xf = X.astype(np.float32).astype(np.float64)          # the C oracle reads float32 X
    r_t, lse_t = tied.responsibilities(Xf, lw, mu, 2.5 * np.eye(D))
    assert np.allclose(r_t, r_s, atol=1e-12) and np.allclose(lse_t, lse_s, rtol=1e-12)
    # a diagonal Sigma: the diagonal path with every row of variances = diag(Sigma)
    v = np.array([0.5, 1.0, 2.0, 4.0])
    r_t, lse_t = tied.responsibilities(Xf, lw, mu, np.diag(v))
    r_d, lse_d = oracle.responsibilities(X.astype(np.float32), lw, mu, np.tile(v, (K, 1)), "diag")
    assert np.allclose(r_t, r_d, atol=1e-12) and np.allclose(lse_t, lse_d, rtol=1e-12)


def pin_rotation_invariance(tied):
    X = _data(seed=4)
    N, D = X.shape
    K = 4
    lw = np.log(np.full(K, 1.0 / K))
    mu = X[:K] + 0.1
    S = _spd(D, seed=5)
    Q, _ = np.linalg.qr(np.random.default_rng(6).normal(size=(D, D)))
    a = tied.em_step(X, lw, mu, S)
    b = tied.em_step(X @ Q.T, lw, mu @ Q.T, Q @ S @ Q.T)
    assert np.allclose(a[0], b[0], atol=1e-10)
    assert np.allclose(a[1] @ Q.T, b[1], atol=1e-9)
    reg = 1e-6 * np.eye(D)
    assert np.allclose(Q @ (a[2] - reg) @ Q.T, b[2] - reg, atol=1e-9)
    assert abs(a[3] - b[3]) <= 1e-9 * abs(a[3])


def pin_brute_force_tiny_case(tied):
    X = _data(seed=7, N=12, D=3)
    K = 3
    lw = np.log([0.2, 0.3, 0.5])
    mu = X[:K] * 0.5
    S = _spd(3, seed=8)
    Si, det = np.linalg.inv(S), np.linalg.det(S)
    p = np.empty((12, K))
    for i in range(12):
        for k in range(K):
            d = X[i] - mu[k]
            p[i, k] = np.exp(lw[k]) * np.exp(-0.5 * d @ Si @ d) / np.sqrt((2 * np.pi) ** 3 * det)
    r_ref = p / p.sum(1, keepdims=True)
    r, lse = tied.responsibilities(X, lw, mu, S)
    assert np.allclose(r, r_ref, rtol=1e-12, atol=1e-15)
    assert np.allclose(lse, np.log(p.sum(1)), rtol=1e-12)
    Nk = r_ref.sum(0)
    mu2 = (r_ref.T @ X) / Nk[:, None]
    S2 = sum(r_ref[i, k] * np.outer(X[i] - mu2[k], X[i] - mu2[k]) for i in range(12) for k in range(K)) / 12
    lw_o, mu_o, S_o, _ = tied.em_step(X, lw, mu, S, reg_covar=0.0)
    assert np.allclose(mu_o, mu2, rtol=1e-12) and np.allclose(S_o, S2, rtol=1e-11)
    assert np.allclose(np.exp(lw_o), Nk / 12, rtol=1e-12)


def pin_loglik_is_non_decreasing(tied):
    X = _data(seed=9, N=600, D=5)
    K = 6
    lw, mu, S = np.log(np.full(K, 1.0 / K)), X[:K].copy(), np.cov(X.T)
    lls = []
    for _ in range(15):
        lw, mu, S, ll = tied.em_step(X, lw, mu, S, reg_covar=1e-9)
        lls.append(ll)
    assert all(b >= a - 1e-9 * abs(a) for a, b in zip(lls, lls[1:]))


ALL_PINS = [pin_one_component_is_the_sample_mean_and_covariance,
            pin_isotropic_and_diagonal_covariance_match_the_c_oracle,
            pin_rotation_invariance, pin_brute_force_tiny_case, pin_loglik_is_non_decreasing]
