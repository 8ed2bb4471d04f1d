"""Parity of the CUDA top-m soft assignment (gmm_predict_topm, through the C
ABI) with the float64 oracle.

Every point's m largest responsibilities (normalised over all K components)
and their component indices, best first.  Responsibilities must agree within
the path's tolerance (FAST: 2e-2, PRECISE: 1e-4, absolute); an index must be
identical wherever its responsibility is separated from its neighbours in
the sorted order (including the (m+1)-th) by more than that tolerance, since
closer gaps can legitimately swap under rounding.  The total log-likelihood
is compared per point as in the EM-step tests.

Parameters.  The FAST path (bf16 data, fp16 operands) is checked here at the
workloads' initial parameters, as in the EM-step tests, and at fitted
parameters (oracle EM iterations) in test_gpu_fitted: its logits carry the
fp16 rounding of the expanded quadratic form, an error that grows with the
ratio |x|^2 / sigma^2.  The PRECISE path is
checked at sharpened parameters: a few oracle EM iterations with a variance
floor of 1e-2 times the mean per-dimension data variance; each entry's bound is
the larger of 1e-4 and what PRECISE's logit resolution allows
(gpu_util.precise_resp_tol), which matters at D > 64 and at fitted
parameters.  Without a floor,
components of these small data sets collapse onto single points (variance =
reg_covar = 1e-6 against data of unit scale) and the expanded form's terms
exceed the result by ~1e6, beyond what fp32 accumulation resolves.
"""
import numpy as np
import pytest
import torch

import em_gmm_step_02_b300 as G
import oracle
import workloads as W
from gpu_util import params_to_device, precise_resp_tol

TOL = {"fast": (2e-2, 1e-2), "precise": (1e-4, 1e-4)}


def check_topm(r_g, i_g, ll_g, r_o, i_o, ll_o, N, m, tol, tol_ll):
    """r_o / i_o carry m+1 columns when K > m (the (m+1)-th decides the last gap).
    tol is a scalar or an (N, m) array of per-entry bounds."""
    r_g = np.asarray(r_g, np.float64)
    assert r_g.shape == (N, m) and i_g.shape == (N, m)
    tol = np.broadcast_to(np.asarray(tol, np.float64), (N, m))
    dev = np.abs(r_g - r_o[:, :m])
    err = dev.max()
    worst = np.unravel_index(np.argmax(dev - tol), dev.shape)
    assert (dev <= tol).all(), f"responsibility error {dev[worst]:.3e} > {tol[worst]:.3e} at {worst}"
    # gap to the previous and next entry of the exact sorted list
    pad_hi = np.full((N, 1), np.inf)
    nxt = r_o[:, 1:m + 1] if r_o.shape[1] > m else np.concatenate([r_o[:, 1:m], np.full((N, 1), -np.inf)], 1)
    prv = np.concatenate([pad_hi, r_o[:, :m - 1]], 1)
    sure = (r_o[:, :m] - nxt > tol) & (prv - r_o[:, :m] > tol)
    bad = sure & (i_g != i_o[:, :m])
    assert not bad.any(), f"{bad.sum()} separated indices differ, e.g. row {np.argwhere(bad)[0]}"
    # every row: distinct valid indices, responsibilities non-increasing
    assert (np.diff(r_g, axis=1) <= 1e-6).all()
    srt = np.sort(i_g, axis=1)
    assert (np.diff(srt, axis=1) > 0).all() if m > 1 else True
    if ll_o is not None:
        assert abs(ll_g - ll_o) / N <= tol_ll, (ll_g, ll_o)
    return err, int(sure.sum())


def sharpened(X_cpu, init, cov, iters):
    """Parameters after `iters` oracle EM steps with a variance floor of 1e-2
    times the mean per-dimension data variance (without one, components of
    these small data sets collapse onto single points)."""
    Xf = X_cpu.float().numpy()
    floor = 1e-2 * float(Xf[: 1 << 20].astype(np.float64).var(axis=0).mean())
    lw, mu, var, _ = oracle.em_run(Xf, *init, cov, iters, var_floor=floor)
    return tuple(np.asarray(a, np.float32) for a in (lw, mu, var))


def run_case(X_cpu, lw, mu, var, cov, m, precision="auto", refine="auto"):
    K = len(lw)
    X = X_cpu.cuda()
    p = params_to_device(lw, mu, var)
    r, idx, ll = G.gmm_predict_topm(X, *p, cov, m, precision=precision, topm_refine=refine)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    mo = min(m + 1, K)
    r_o, i_o, ll_o = oracle.topm(X_cpu.float().numpy(), lw, mu, var, cov, mo)
    return r.cpu().numpy(), idx.cpu().numpy(), float(ll.item()), r_o, i_o, ll_o


CASES = [
    # N, D, K, cov, x_dtype, m ; bf16 cases run FAST at the initial parameters,
    # f32 cases run PRECISE at sharpened parameters
    (3001, 96, 200, "diag", "bf16", 4),
    (129, 5, 7, "spherical", "bf16", 7),
    (12000, 32, 1100, "diag", "bf16", 8),
    (6000, 48, 2500, "diag", "bf16", 5),
    (4096, 8, 16, "diag", "f32", 2),
    (5000, 64, 256, "spherical", "f32", 3),
    (1000, 1, 3, "diag", "f32", 3),
    (2000, 16, 20, "diag", "f32", 16),
    (12000, 32, 1100, "diag", "f32", 8),
    (6000, 48, 2500, "spherical", "f32", 5),
    (3000, 128, 300, "diag", "f32", 5),
    (4000, 100, 1100, "diag", "f32", 12),
]


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,K,cov,xd,m", CASES)
def test_topm_small(N, D, K, cov, xd, m):
    w = W.generic(N, D, K, cov, xd, seed=N + 3 * D + K)
    X = W.make_data(w)
    init = W.make_init(w, X)
    path = "fast" if xd == "bf16" else "precise"
    lw, mu, var = init if path == "fast" else sharpened(X, init, cov, 2)
    out = run_case(X, lw, mu, var, cov, m)
    tol, tol_ll = TOL[path]
    if path == "precise":
        tol, tol_ll = precise_resp_tol(X.float().numpy(), mu, var, cov, out[4][:, :m], out[3][:, :m], tol, tol_ll)
    err, n_sure = check_topm(*out[:3], *out[3:], N, m, tol, tol_ll)
    print(f"max |dr| {err:.2e}, {n_sure} separated entries checked")


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,K,cov,xd,m", [CASES[i] for i in (0, 1, 2, 3, 5, 6, 10, 11)])
def test_topm_refinement_switched(N, D, K, cov, xd, m):
    """The other setting of the direct-form refinement than the path's
    default: FAST with it on, PRECISE with it off; each within its path's
    bound (the refinement keeps the pass's candidates and their share)."""
    w = W.generic(N, D, K, cov, xd, seed=N + 3 * D + K)
    X = W.make_data(w)
    init = W.make_init(w, X)
    path = "fast" if xd == "bf16" else "precise"
    lw, mu, var = init if path == "fast" else sharpened(X, init, cov, 2)
    out = run_case(X, lw, mu, var, cov, m, refine="on" if path == "fast" else "off")
    tol, tol_ll = TOL[path]
    if path == "precise":
        tol, tol_ll = precise_resp_tol(X.float().numpy(), mu, var, cov, out[4][:, :m], out[3][:, :m], tol, tol_ll)
    err, n_sure = check_topm(*out[:3], *out[3:], N, m, tol, tol_ll)
    print(f"max |dr| {err:.2e}, {n_sure} separated entries checked")


@pytest.mark.gpu
@pytest.mark.parametrize("name,rows,m", [("tiny_diag", 4096, 2), ("embed_10m", 20000, 4),
                                          ("largek_2m", 30000, 8)])
def test_topm_workload_prefix(name, rows, m):
    w = W.WORKLOADS[name].scaled(rows)
    X = W.make_data(w)
    init = W.make_init(w, X)
    path = "fast" if w.x_dtype == "bf16" else "precise"
    lw, mu, var = init if path == "fast" else sharpened(X, init, w.cov, 3)
    out = run_case(X, lw, mu, var, w.cov, m)
    tol, tol_ll = TOL[path]
    if path == "precise":
        tol, tol_ll = precise_resp_tol(X.float().numpy(), mu, var, w.cov, out[4][:, :m], out[3][:, :m], tol,
                                       tol_ll)
    err, n_sure = check_topm(*out[:3], *out[3:], X.shape[0], m, tol, tol_ll)
    print(f"max |dr| {err:.2e}, {n_sure} separated entries checked")


@pytest.mark.gpu
def test_topm_dead_components_and_m1():
    w = W.generic(3000, 12, 40, "diag", "f32", seed=4)
    X = W.make_data(w)
    lw, mu, var = W.make_init(w, X)
    lw = lw.copy()
    lw[::3] = -np.inf                      # every third component is dead
    out = run_case(X, lw, mu, var, "diag", 1)
    check_topm(*out[:3], *out[3:], X.shape[0], 1, *TOL["precise"])
    assert not np.isin(out[1], np.arange(0, 40, 3)).any()
    # m = 1 is the hard label: the argmax of the oracle's responsibilities
    r_all, _ = oracle.responsibilities(X.numpy(), lw, mu, var, "diag")
    assert (out[1][:, 0] == r_all.argmax(1)).mean() > 0.999


@pytest.mark.gpu
@pytest.mark.parametrize("refine", ["auto", "on"])
def test_topm_full_size_embed_sampled_rows(refine):
    """The full 10M x 128 x 1024 workload in one launch (FAST; with and
    without the refinement); rows are independent, so a sample of rows is
    checked against the oracle run on those rows alone."""
    w = W.WORKLOADS["embed_10m"]
    X = W.make_data(w, device="cuda")
    lw, mu, var = W.make_init(w, X)
    p = params_to_device(lw, mu, var)
    r, idx, ll = G.gmm_predict_topm(X, *p, w.cov, 4, topm_refine=refine)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(X.shape[0], 3000, replace=False))
    rows = np.concatenate([rows, [X.shape[0] - 1]])
    Xs = X[torch.tensor(rows, device="cuda")].cpu()
    r_o, i_o, _ = oracle.topm(Xs.float().numpy(), lw, mu, var, w.cov, 5)
    check_topm(r[rows].cpu().numpy(), idx[rows].cpu().numpy(), None, r_o, i_o, None, len(rows), 4,
               *TOL["fast"])
    rs = r.sum(1)
    assert float(rs.max()) <= 1.0 + 1e-4 and float(r.min()) >= 0.0
    assert np.isfinite(ll.item())
