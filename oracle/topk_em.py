"""Approximate top-k EM step of the oracle (spherical or diagonal
covariance): each point keeps only its k largest log scores in the E-step and
normalises its responsibilities over that subset; the M-step is the usual
one with those responsibilities.  k >= K is exact EM.  Plain float64 numpy
from the definition.  TEST INFRASTRUCTURE ONLY, like the rest of this folder.

Source: the "GMMXX" README's training option approx_top_k (each E-step keeps
the top k component logits per sample and normalises over that subset; values
>= K are exact EM), on the EM step of "Flash-GMM: A Memory-Efficient Kernel
for Scalable Soft Clustering", section 2.

Reading where the page is silent: the subset is the k largest log scores
with equal values ordered by the lower component index; the reported
log-likelihood stays the exact one at the input parameters (log-sum-exp over
all K), so that runs with different k remain comparable.
"""
from __future__ import annotations

import numpy as np

EMPTY_NK = 1e-30
LOG_2PI = float(np.log(2.0 * np.pi))


def log_scores(X, log_weights, means, vars_, cov):
    """l (N x K): log pi_k + log N(x_i | mu_k, Sigma_k) in the direct form."""
    X = np.asarray(X, np.float64)
    mu = np.asarray(means, np.float64)
    lw = np.asarray(log_weights, np.float64).reshape(-1)
    K, D = mu.shape
    v = np.asarray(vars_, np.float64)
    v = np.repeat(v.reshape(K, 1), D, 1) if cov == "spherical" else v.reshape(K, D)
    ell = np.empty((X.shape[0], K))
    for k in range(K):
        diff = X - mu[k]
        ell[:, k] = lw[k] - 0.5 * (np.log(2.0 * np.pi * v[k]).sum() + (diff * diff / v[k]).sum(1))
    return ell


def _lse(a, axis=1):
    mx = a.max(axis)
    with np.errstate(invalid="ignore"):
        out = mx + np.log(np.exp(a - np.expand_dims(mx, axis)).sum(axis))
    out[mx == -np.inf] = -np.inf
    return out


def responsibilities(X, log_weights, means, vars_, cov, k):
    """r (N x K) with at most k nonzeros per row, and the exact lse (N)."""
    ell = log_scores(X, log_weights, means, vars_, cov)
    N, K = ell.shape
    lse_all = _lse(ell)
    if k >= K:
        return np.exp(ell - lse_all[:, None]), lse_all
    # the k largest scores of each row; equal values: lower index first
    order = np.lexsort((np.broadcast_to(np.arange(K), ell.shape), -ell), axis=1)[:, :k]
    keep = np.zeros_like(ell, dtype=bool)
    np.put_along_axis(keep, order, True, axis=1)
    sub = np.where(keep, ell, -np.inf)
    lse_k = _lse(sub)
    r = np.where(keep, np.exp(sub - lse_k[:, None]), 0.0)
    return r, lse_all


def em_step(X, log_weights, means, vars_, cov, k, reg_covar=1e-6, var_floor=0.0):
    """One approximate top-k EM iteration.  Returns (new_log_weights,
    new_means, new_vars, total_loglik) like the exact oracle."""
    X = np.asarray(X, np.float64)
    mu = np.asarray(means, np.float64)
    N, D = X.shape
    K = mu.shape[0]
    r, lse = responsibilities(X, log_weights, mu, vars_, cov, k)
    Nk = r.sum(0)
    empty = Nk < EMPTY_NK
    new_lw = np.where(empty, -np.inf, np.log(np.maximum(Nk, EMPTY_NK) / N))
    new_mu = mu.copy()
    new_mu[~empty] = (r[:, ~empty].T @ X) / Nk[~empty, None]
    old_v = np.asarray(vars_, np.float64)
    if cov == "spherical":
        new_v = old_v.reshape(K).copy()
    else:
        new_v = old_v.reshape(K, D).copy()
    for j in np.nonzero(~empty)[0]:
        diff = X - new_mu[j]
        sv = (r[:, j:j + 1] * diff * diff).sum(0) / Nk[j]
        if cov == "spherical":
            new_v[j] = max(sv.mean(), var_floor) + reg_covar
        else:
            new_v[j] = np.maximum(sv, var_floor) + reg_covar
    return new_lw, new_mu, new_v, float(lse.sum())
