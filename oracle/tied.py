"""Tied-covariance EM step of the oracle: every component shares one full
D x D covariance Sigma.  Plain float64 numpy, written from the definitions
(direct difference form, no expansion).  TEST INFRASTRUCTURE ONLY, like the
rest of this folder.

Sources: the EM step of "Flash-GMM: A Memory-Efficient Kernel for Scalable
Soft Clustering", section 2 (mixture density, responsibilities by
log-sum-exp, M-step), with the covariance shared by all components as in the
"GMMXX" README ("Covariance Coverage": covariance_type "tied", parameter
shape (D, D)).

  log score   l_ik = log pi_k - 1/2 (D log 2 pi + log|Sigma|
                                    + (x_i - mu_k)^T Sigma^-1 (x_i - mu_k))
  E-step      r_ik = exp(l_ik - lse_i),  lse_i = log sum_k exp(l_ik)
  M-step      N_k = sum_i r_ik,  log pi_k' = log(N_k / N),
              mu_k' = sum_i r_ik x_i / N_k,
              Sigma' = sum_k sum_i r_ik (x_i - mu_k')(x_i - mu_k')^T / N,
              then on the diagonal: max(Sigma'_dd, var_floor) + reg_covar.
A component with N_k < 1e-30 keeps its mean, gets log-weight -inf and adds
nothing to Sigma'.  The log-likelihood is sum_i lse_i at the input
parameters.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular

EMPTY_NK = 1e-30
LOG_2PI = float(np.log(2.0 * np.pi))


def log_scores(X, log_weights, means, cov):
    """l (N x K) and lse (N) for a shared covariance `cov` (D x D)."""
    X = np.asarray(X, np.float64)
    mu = np.asarray(means, np.float64)
    lw = np.asarray(log_weights, np.float64).reshape(-1)
    S = np.asarray(cov, np.float64)
    N, D = X.shape
    L = np.linalg.cholesky(S)
    logdet = 2.0 * np.log(np.diag(L)).sum()
    ell = np.empty((N, len(lw)))
    for k in range(len(lw)):
        z = solve_triangular(L, (X - mu[k]).T, lower=True)     # L z = x - mu_k
        ell[:, k] = lw[k] - 0.5 * (D * LOG_2PI + logdet + (z * z).sum(0))
    mx = ell.max(1)
    with np.errstate(invalid="ignore"):
        lse = mx + np.log(np.exp(ell - mx[:, None]).sum(1))
    lse[mx == -np.inf] = -np.inf
    return ell, lse


def em_step(X, log_weights, means, cov, reg_covar=1e-6, var_floor=0.0):
    """One EM iteration.  Returns (new_log_weights, new_means, new_cov, total_loglik)."""
    X = np.asarray(X, np.float64)
    mu = np.asarray(means, np.float64)
    N, D = X.shape
    ell, lse = log_scores(X, log_weights, mu, cov)
    r = np.exp(ell - lse[:, None])
    Nk = r.sum(0)
    empty = Nk < EMPTY_NK
    new_lw = np.where(empty, -np.inf, np.log(np.maximum(Nk, EMPTY_NK) / N))
    new_mu = mu.copy()
    live = ~empty
    new_mu[live] = (r[:, live].T @ X) / Nk[live, None]
    S = np.zeros((D, D))
    for k in np.nonzero(live)[0]:
        diff = X - new_mu[k]
        S += (diff * r[:, k:k + 1]).T @ diff
    S /= N
    d = np.arange(D)
    S[d, d] = np.maximum(S[d, d], var_floor) + reg_covar
    return new_lw, new_mu, S, float(lse.sum())


def responsibilities(X, log_weights, means, cov):
    ell, lse = log_scores(X, log_weights, means, cov)
    return np.exp(ell - lse[:, None]), lse
