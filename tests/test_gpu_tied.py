"""Parity of the tied-covariance EM step and top-m pass (one full D x D
covariance shared by every component) with the float64 oracle.  The GPU runs
the fused kernel on linear logits (the per-point quadratic term cancels in
the responsibilities and returns to the log-likelihood through the data's
Gram matrix) and takes the shared covariance from that Gram matrix and the
components' new means.  Tolerances as for the other covariance types: PRECISE
(float32 data) 1e-4 relative on weights, means and the covariance and 1e-4
per point on the log-likelihood; FAST (bf16 data) 2e-2 and 1e-2."""
import numpy as np
import pytest
import torch

import em_gmm_step_02_b300 as G
import oracle
import workloads as W
from gpu_util import params_to_device, rel_l2_rows

TOL = {"precise": (1e-4, 1e-4), "fast": (2e-2, 1e-2)}


def _case(N, D, K, xd, seed):
    w = W.generic(N, D, K, "tied", xd, seed=seed)
    X = W.make_data(w)
    return w, X, W.make_init(w, X)


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,K,xd,prec", [
    (3000, 16, 8, "f32", "auto"),
    (5000, 48, 40, "f32", "auto"),
    (4000, 32, 16, "bf16", "auto"),
    (4000, 32, 16, "bf16", "precise"),   # bf16 data shifted by the mean of the means
    (20000, 128, 1024, "bf16", "auto"),  # clusters of 8 slices
    (12000, 32, 1100, "bf16", "auto"),   # two passes
    (3000, 128, 16, "f32", "auto"),      # PRECISE, 128 features
])
def test_tied_em_step_against_oracle(N, D, K, xd, prec):
    """Element by element: weights relative; means relative to the larger of
    |mu| and the shared standard deviation of the dimension; the shared
    covariance relative to sqrt(Sigma_dd Sigma_ee) (its natural scale)."""
    w, X, (lw, mu, S) = _case(N, D, K, xd, seed=N + D + K)
    p = params_to_device(lw, mu, S)
    lw2, mu2, S2, ll = G.gmm_em_step(X.cuda(), *p, "tied", precision=prec)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    ref = oracle.tied.em_step(X.float().numpy().astype(np.float64), lw, mu, S)
    path = "precise" if (prec == "precise" or (prec == "auto" and xd == "f32")) else "fast"
    tol, tol_ll = TOL[path]
    lw_g, mu_g, S_g = [t.cpu().numpy().astype(np.float64) for t in (lw2, mu2, S2)]
    w_r = np.exp(ref[0])
    e_w = (np.abs(np.exp(lw_g) - w_r) / np.maximum(w_r, 1e-6 * w_r.max())).max()
    sd = np.sqrt(np.diag(ref[2]))
    e_mu = (np.abs(mu_g - ref[1]) / np.maximum(np.abs(ref[1]), sd[None, :])).max()
    e_S = (np.abs(S_g - ref[2]) / np.sqrt(np.outer(np.diag(ref[2]), np.diag(ref[2])))).max()
    e_ll = abs(float(ll.item()) - ref[3]) / N
    msg = f"w {e_w:.2e} mu {e_mu:.2e} Sigma {e_S:.2e} ll/N {e_ll:.2e}"
    assert e_w <= tol and e_mu <= tol and e_S <= tol and e_ll <= tol_ll, msg
    print(msg)


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,K,xd,m", [(3000, 16, 8, "f32", 3), (4000, 32, 16, "bf16", 4)])
def test_tied_topm_against_oracle(N, D, K, xd, m):
    w, X, (lw, mu, S) = _case(N, D, K, xd, seed=7 * N + K)
    p = params_to_device(lw, mu, S)
    r, idx, ll = G.gmm_predict_topm(X.cuda(), *p, "tied", m)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    r_ref, lse = oracle.tied.responsibilities(X.float().numpy().astype(np.float64), lw, mu, S)
    tol, tol_ll = TOL["fast" if xd == "bf16" else "precise"]
    order = np.lexsort((np.broadcast_to(np.arange(K), r_ref.shape), -r_ref), axis=1)[:, :m + 1]
    r_o = np.take_along_axis(r_ref, order, 1)
    r_g = r.cpu().numpy().astype(np.float64)
    assert np.abs(r_g - r_o[:, :m]).max() <= tol
    nxt = r_o[:, 1:m + 1]
    prv = np.concatenate([np.full((N, 1), np.inf), r_o[:, :m - 1]], 1)
    sure = (r_o[:, :m] - nxt > tol) & (prv - r_o[:, :m] > tol)
    assert not (sure & (idx.cpu().numpy() != order[:, :m])).any()
    assert abs(float(ll.item()) - lse.sum()) / N <= tol_ll
