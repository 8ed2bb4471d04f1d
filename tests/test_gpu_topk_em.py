"""Parity of approximate top-k EM on the GPU (gmm_em_step with
opts.approx_top_k = k, through the C ABI) with the float64 oracle
(oracle/topk_em.py).

Approximate top-k EM (the "GMMXX" README's training option approx_top_k): in
the E-step every point keeps its k largest logits and normalises its
responsibilities over those k; the M-step is the usual one with them; the
reported log-likelihood stays the exact one over all K components.

The bounds are the EM step's (gpu_util.elementwise_errors; FAST 2e-2,
PRECISE 1e-4).  Whether a component is kept can flip where the k-th and
(k+1)-th logits of a point are closer than the path's rounding; a flip moves
the point's renormalised responsibility r'_(k) from one component to the
other.  At broad starting parameters (every variance the data's) many
components share each point and r'_(k) is about 1/k, so under FAST rounding
(logit error ~2^-12 times the size of the expanded form's terms) flips
move whole fractions of a point; the FAST cases therefore run at fitted
parameters (oracle EM iterations, as in test_gpu_fitted), where each point's
mass sits on few components and r'_(k) at the boundary is small.  PRECISE
resolves the selection at the starting parameters.

Cases cover: both covariance types, both paths, the two-team top-m kernel
(FAST, k <= 8) and the general one (PRECISE, k = 16), the two-pass plan
(K > 1024), k = 1 (hard EM), components with more than one chunk of pairs,
point counts that leave a ragged last tile of the counting sort, dead
components, k >= K (exact EM, bit-identical to the exact call) and
bit-identical repetition.
"""
import numpy as np
import pytest
import torch

import em_gmm_step_02_b300 as G
import workloads as W
from gpu_util import elementwise_errors, params_to_device
from oracle import topk_em
from test_gpu_fitted import fitted

TOL = {"fast": (2e-2, 1e-2), "precise": (1e-4, 1e-4)}

CASES = [
    # N, D, K, cov, x_dtype, path, k
    (5000, 16, 64, "diag", "f32", "precise", 4),
    (4000, 33, 50, "spherical", "f32", "precise", 3),
    (9001, 8, 16, "diag", "f32", "precise", 1),
    (3000, 8, 40, "diag", "f32", "precise", 16),
    (20000, 4, 6, "diag", "f32", "precise", 2),
    (6000, 64, 128, "spherical", "bf16", "fast", 2),
]

FITTED_CASES = [
    # workload, rows, oracle iterations, k (FAST: bf16 data)
    ("embed_10m", 20000, 10, 4),
    ("largek_2m", 8192, 4, 8),
]


def _run(X, lw, mu, var, cov, path, k, **kw):
    p = params_to_device(lw, mu, var)
    out = G.gmm_em_step(X.cuda(), *p, cov, precision=path, approx_top_k=k, **kw)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    return [t.cpu().numpy() for t in out[:3]] + [float(out[3].item())]


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,K,cov,xd,path,k", CASES)
def test_topk_em_against_oracle(N, D, K, cov, xd, path, k):
    w = W.generic(N, D, K, cov, xd, seed=N + D + K + k)
    X = W.make_data(w)
    lw, mu, var = W.make_init(w, X)
    got = _run(X, lw, mu, var, cov, path, k)
    ref = topk_em.em_step(X.float().numpy(), lw, mu, var, cov, k)
    tol, tol_ll = TOL[path]
    e_w, e_mu, e_v, msg = elementwise_errors(got[:3], ref, N, cov, path, tol, xd, mu)
    e_ll = abs(got[3] - ref[3]) / N
    msg += f" ll/N {e_ll:.2e}"
    print(msg)
    assert e_w <= 1 and e_mu <= 1 and e_v <= 1 and e_ll <= tol_ll, msg


@pytest.mark.gpu
@pytest.mark.parametrize("name,rows,iters,k", FITTED_CASES)
def test_topk_em_at_fitted_parameters(name, rows, iters, k):
    w, X, (lw, mu, var), reg = fitted(name, rows, iters, 0.0)
    got = _run(X, lw, mu, var, w.cov, "fast", k, reg_covar=reg)
    ref = topk_em.em_step(X.float().numpy(), lw, mu, var, w.cov, k, reg_covar=reg)
    tol, tol_ll = TOL["fast"]
    e_w, e_mu, e_v, msg = elementwise_errors(got[:3], ref, rows, w.cov, "fast", tol, w.x_dtype, mu)
    e_ll = abs(got[3] - ref[3]) / rows
    msg += f" ll/N {e_ll:.2e}"
    print(msg)
    assert e_w <= 1 and e_mu <= 1 and e_v <= 1, msg
    if name == "embed_10m":
        assert e_ll <= tol_ll, msg


@pytest.mark.gpu
def test_topk_em_dead_components_and_repeat():
    N, D, K, k = 7000, 12, 30, 3
    w = W.generic(N, D, K, "diag", "f32", seed=5)
    X = W.make_data(w)
    lw, mu, var = W.make_init(w, X)
    lw = lw.copy()
    lw[[0, 7, 29]] = -np.inf
    got = _run(X, lw, mu, var, "diag", "precise", k)
    again = _run(X, lw, mu, var, "diag", "precise", k)
    for a, b in zip(got, again):
        assert np.array_equal(np.asarray(a), np.asarray(b))
    ref = topk_em.em_step(X.float().numpy(), lw, mu, var, "diag", k)
    assert np.all(np.isneginf(got[0][[0, 7, 29]]))
    assert np.array_equal(got[1][[0, 7, 29]], mu[[0, 7, 29]])
    assert np.array_equal(got[2][[0, 7, 29]], var[[0, 7, 29]])
    e_w, e_mu, e_v, msg = elementwise_errors(got[:3], ref, N, "diag", "precise", 1e-4, "f32", mu)
    assert e_w <= 1 and e_mu <= 1 and e_v <= 1, msg


@pytest.mark.gpu
def test_topk_em_k_at_least_K_is_exact_em():
    N, D, K = 3000, 16, 8
    w = W.generic(N, D, K, "diag", "bf16", seed=9)
    X = W.make_data(w)
    lw, mu, var = W.make_init(w, X)
    exact = _run(X, lw, mu, var, "diag", "fast", 0)
    for k in (K, K + 5):
        got = _run(X, lw, mu, var, "diag", "fast", k)
        for a, b in zip(got, exact):
            assert np.array_equal(np.asarray(a), np.asarray(b))


@pytest.mark.gpu
def test_topk_em_rejections():
    w = W.generic(500, 8, 8, "diag", "f32", seed=1)
    X = W.make_data(w).cuda()
    lw, mu, var = params_to_device(*W.make_init(w, X.cpu()))
    with pytest.raises(G.GmmError) as e:
        G.gmm_em_step(X, lw, mu, var, "diag", approx_top_k=-1)
    assert e.value.code == -1
    w = W.generic(500, 8, 40, "diag", "f32", seed=1)
    X = W.make_data(w).cuda()
    lw, mu, var = params_to_device(*W.make_init(w, X.cpu()))
    with pytest.raises(G.GmmError) as e:
        G.gmm_em_step(X, lw, mu, var, "diag", approx_top_k=17)
    assert e.value.code == -2
