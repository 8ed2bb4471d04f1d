"""Plain float64 CPU oracle for one EM step of a spherical / diagonal GMM.

TEST INFRASTRUCTURE ONLY: the parity tests, the smoke check and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library never
imports, links or runs anything in this folder, and this folder imports
nothing from the library.

The arithmetic lives in ``gmm_oracle.c`` (direct difference form, double
precision, OpenMP over points).  This module compiles it with gcc on first use
and wraps it with numpy-friendly functions.

Sources: "Flash-GMM: A Memory-Efficient Kernel for Scalable Soft Clustering",
section 2 (mixture density, E-step, log-sum-exp, M-step) and its multi-assignment
use of the final responsibilities; "ML0094 GMM vs K-Means" (EM steps and the
k-means limit).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gmm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()

SPHERICAL = 0
DIAG = 1
COV = {"spherical": SPHERICAL, "diag": DIAG}


def build(force: bool = False) -> str:
    """Compile ``gmm_oracle.c`` into ``liboracle.so`` (plain -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-std=c11", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Oracle:
    """ctypes wrapper around one compiled copy of the oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        dp = ctypes.POINTER(ctypes.c_double)
        fp = ctypes.POINTER(ctypes.c_float)
        ip = ctypes.POINTER(ctypes.c_int32)
        i64, i32 = ctypes.c_int64, ctypes.c_int
        lib.oracle_threads.argtypes = [i32]
        lib.oracle_threads.restype = i32
        lib.oracle_log_scores.argtypes = [fp, i64, i32, i32, i32, dp, dp, dp,
                                          dp, dp, i32]
        lib.oracle_log_scores.restype = i32
        lib.oracle_em_step.argtypes = [fp, i64, i32, i32, i32, dp, dp, dp,
                                       ctypes.c_double, ctypes.c_double,
                                       dp, dp, dp, dp, i32]
        lib.oracle_em_step.restype = i32
        lib.oracle_topm.argtypes = [fp, i64, i32, i32, i32, dp, dp, dp, i32,
                                    dp, ip, dp, i32]
        lib.oracle_topm.restype = i32
        self.lib = lib
        self.path = lib_path

    def threads(self, nthreads: int = 0) -> int:
        """Threads the oracle uses for a request of ``nthreads`` (0 = all)."""
        return int(self.lib.oracle_threads(nthreads))

    def log_scores(self, X, log_weights, means, vars_, cov, nthreads=0):
        """Per-point per-component log(pi_k N(x_i|mu_k,Sigma_k)) and per-point log p(x_i)."""
        X, N, D, K, lw, mu, var = _check(X, log_weights, means, vars_, cov)
        ell = np.empty((N, K), np.float64)
        lse = np.empty((N,), np.float64)
        rc = self.lib.oracle_log_scores(_ptr(X, ctypes.c_float), N, D, K, _cov(cov),
                                       _ptr(lw, ctypes.c_double), _ptr(mu, ctypes.c_double),
                                       _ptr(var, ctypes.c_double), _ptr(ell, ctypes.c_double),
                                       _ptr(lse, ctypes.c_double), nthreads)
        assert rc == 0, rc
        return ell, lse

    def responsibilities(self, X, log_weights, means, vars_, cov, nthreads=0):
        """Full N x K responsibility matrix (small inputs only)."""
        ell, lse = self.log_scores(X, log_weights, means, vars_, cov, nthreads)
        return np.exp(ell - lse[:, None]), lse

    def em_step(self, X, log_weights, means, vars_, cov, reg_covar=1e-6, var_floor=0.0,
                nthreads=0):
        """One EM iteration.  Returns (new_log_weights, new_means, new_vars, total_loglik)."""
        X, N, D, K, lw, mu, var = _check(X, log_weights, means, vars_, cov)
        out_lw = np.empty(K, np.float64)
        out_mu = np.empty((K, D), np.float64)
        out_var = np.empty_like(var)
        ll = np.zeros(1, np.float64)
        rc = self.lib.oracle_em_step(_ptr(X, ctypes.c_float), N, D, K, _cov(cov),
                                    _ptr(lw, ctypes.c_double), _ptr(mu, ctypes.c_double),
                                    _ptr(var, ctypes.c_double), float(reg_covar),
                                    float(var_floor), _ptr(out_lw, ctypes.c_double),
                                    _ptr(out_mu, ctypes.c_double),
                                    _ptr(out_var, ctypes.c_double),
                                    _ptr(ll, ctypes.c_double), nthreads)
        assert rc == 0, rc
        return out_lw, out_mu, out_var, float(ll[0])

    def em_run(self, X, log_weights, means, vars_, cov, iters, reg_covar=1e-6,
               var_floor=0.0, nthreads=0):
        """``iters`` EM iterations; returns the final parameters and the list of
        log-likelihoods (entry t is evaluated at the parameters entering step t)."""
        lls = []
        lw, mu, var = _f64(log_weights), _f64(means), _f64(vars_)
        for _ in range(iters):
            lw, mu, var, ll = self.em_step(X, lw, mu, var, cov, reg_covar, var_floor, nthreads)
            lls.append(ll)
        return lw, mu, var, lls

    def topm(self, X, log_weights, means, vars_, cov, m, nthreads=0):
        """Top-m responsibilities (N x m, descending) and indices (N x m int32),
        plus the total log-likelihood."""
        X, N, D, K, lw, mu, var = _check(X, log_weights, means, vars_, cov)
        r = np.empty((N, m), np.float64)
        idx = np.empty((N, m), np.int32)
        ll = np.zeros(1, np.float64)
        rc = self.lib.oracle_topm(_ptr(X, ctypes.c_float), N, D, K, _cov(cov),
                                 _ptr(lw, ctypes.c_double), _ptr(mu, ctypes.c_double),
                                 _ptr(var, ctypes.c_double), int(m),
                                 _ptr(r, ctypes.c_double), _ptr(idx, ctypes.c_int32),
                                 _ptr(ll, ctypes.c_double), nthreads)
        assert rc == 0, rc
        return r, idx, float(ll[0])


from . import tied  # noqa: E402  (tied-covariance EM, numpy)
from . import topk_em  # noqa: E402  (approximate top-k EM, numpy)


def threshold_assign(r, tau, max_per_point):
    """Threshold multi-assignment written from its definition: for every
    point (row of the N x K responsibility matrix r), the components with
    r >= tau in descending order of r (equal values: lower index first), at
    most max_per_point of them; as compressed rows (offsets N+1, idx, resp)."""
    r = np.asarray(r, np.float64)
    offsets = [0]
    idx, resp = [], []
    for row in r:
        order = sorted(range(len(row)), key=lambda k: (-row[k], k))
        kept = [k for k in order if row[k] >= tau][:max_per_point]
        idx.extend(kept)
        resp.extend(row[k] for k in kept)
        offsets.append(len(idx))
    return np.array(offsets, np.int64), np.array(idx, np.int32), np.array(resp, np.float64)


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _cov(cov):
    return COV[cov] if isinstance(cov, str) else int(cov)


def _check(X, log_weights, means, vars_, cov):
    X = _f32(X)
    N, D = X.shape
    means = _f64(means)
    K = means.shape[0]
    assert means.shape == (K, D)
    log_weights = _f64(log_weights).reshape(K)
    vars_ = _f64(vars_)
    vars_ = vars_.reshape(K) if _cov(cov) == SPHERICAL else vars_.reshape(K, D)
    return X, N, D, K, log_weights, means, vars_


_default = None


def default() -> Oracle:
    """The oracle built from ``gmm_oracle.c`` in this folder."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def threads(nthreads: int = 0) -> int:
    return default().threads(nthreads)


def log_scores(*a, **k):
    return default().log_scores(*a, **k)


def responsibilities(*a, **k):
    return default().responsibilities(*a, **k)


def em_step(*a, **k):
    return default().em_step(*a, **k)


def em_run(*a, **k):
    return default().em_run(*a, **k)


def topm(*a, **k):
    return default().topm(*a, **k)
