"""Pins of the oracle's approximate top-k EM step, as functions of the module
that implements it (the real ``oracle.topk_em`` in test_oracle_topk.py,
planted mistakes in the mutant test there): k >= K is the exact EM step of
the independent C oracle, k = 1 is hard-assignment EM computed by grouping,
and properties of the kept subset on a case with ties."""
import numpy as np

import oracle
import workloads as W


def _case(cov="diag", seed=0, N=500, D=5, K=9):
    w = W.generic(N, D, K, cov, "f32", seed=seed)
    X = W.make_data(w)
    lw, mu, var = W.make_init(w, X)
    lw = np.log(np.random.default_rng(seed).dirichlet(np.ones(K))).astype(np.float32)
    return X.numpy(), lw, mu, var


def pin_all_components_is_exact_em(topk):
    for cov in ("diag", "spherical"):
        X, lw, mu, var = _case(cov, seed=1)
        K = len(lw)
        a = topk.em_step(X, lw, mu, var, cov, K)
        b = oracle.em_step(X, lw, mu, var, cov)
        for u, v in zip(a[:3], b[:3]):
            assert np.allclose(u, v, rtol=1e-10, atol=1e-12)
        assert abs(a[3] - b[3]) <= 1e-10 * abs(b[3])
        c = topk.em_step(X, lw, mu, var, cov, K + 5)     # k > K is exact too
        assert np.allclose(c[1], b[1], rtol=1e-10)


def pin_one_component_is_hard_assignment_em(topk):
    X, lw, mu, var = _case(seed=2)
    X64 = X.astype(np.float64)
    N, D = X.shape
    K = len(lw)
    ell = oracle.log_scores(X, lw, mu, var, "diag")[0]
    lab = np.argmax(ell, 1)                               # ties: the first (lowest) index
    lw2, mu2, v2, _ = topk.em_step(X, lw, mu, var, "diag", 1, reg_covar=0.0)
    for k in range(K):
        sel = X64[lab == k]
        if len(sel) == 0:
            assert lw2[k] == -np.inf
            continue
        assert abs(np.exp(lw2[k]) - len(sel) / N) <= 1e-12
        assert np.allclose(mu2[k], sel.mean(0), rtol=1e-12, atol=1e-12)
        assert np.allclose(v2[k], sel.var(0), rtol=1e-10, atol=1e-14)


def pin_subset_properties(topk):
    X, lw, mu, var = _case(seed=3)
    r_all, lse_all = topk.responsibilities(X, lw, mu, var, "diag", 100)
    for k in (2, 4):
        r, lse = topk.responsibilities(X, lw, mu, var, "diag", k)
        assert np.allclose(lse, lse_all)                  # the exact log-likelihood
        assert np.allclose(r.sum(1), 1.0, rtol=1e-12)
        assert ((r > 0).sum(1) <= k).all()
        for i in range(len(r)):
            top = np.lexsort((np.arange(r.shape[1]), -r_all[i]))[:k]
            kept = np.nonzero(r[i] > 0)[0]
            assert set(kept) <= set(top)
            # renormalised over the subset: ratios are those of the exact responsibilities
            assert np.allclose(r[i, top], r_all[i, top] / r_all[i, top].sum(), rtol=1e-10)


def pin_ties_keep_the_lower_index(topk):
    # three identical components: with k = 2 the first two are kept, evenly
    X = np.array([[0.0, 0.0], [0.1, -0.2], [3.0, 1.0]])
    mu = np.array([[0.0, 0.0], [0.0, 0.0], [0.0, 0.0], [5.0, 5.0]])
    var = np.ones((4, 2))
    lw = np.log(np.full(4, 0.25))
    r, _ = topk.responsibilities(X, lw, mu, var, "diag", 2)
    assert np.allclose(r[:, :2], 0.5) and (r[:, 2:] == 0).all()


ALL_PINS = [pin_all_components_is_exact_em, pin_one_component_is_hard_assignment_em,
            pin_subset_properties, pin_ties_keep_the_lower_index]
