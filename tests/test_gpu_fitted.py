"""Parity at the workloads' operating point: one EM step and one top-m pass
from FITTED parameters (oracle EM iterations from the workload's starting
point), compared with the float64 oracle element by element.

The workloads run their final top-m pass after their EM iterations, so this is
where the multi-assignment of "Flash-GMM: A Memory-Efficient Kernel for
Scalable Soft Clustering" (conclusion: assignments read off the final
responsibilities) is used; fitted components are sharp, which is where the
expanded-form logits [x, x^2] . [mu/s2, -1/(2 s2)] are hardest.

Bounds (gpu_util.elementwise_errors): per element, weights relative, means
relative to max(|mu|, sigma), variances relative or within four rounding units
of the raw second moment; the per-point mean log-likelihood within the
path's absolute bound; top-m responsibilities within the path's tolerance and
indices identical wherever the responsibility gap to the neighbouring entries
exceeds it.

Log-likelihood where the expanded form cannot resolve it.  The logit of a
component is a difference of terms of size k = max_d x_d^2 / s2_d (in units of
the result); fp32 accumulation resolves it to about k * 2^-24 * sqrt(D), fp16
operands (FAST) to about k * 2^-12.  EM from random-point starts with the
default absolute regulariser (reg_covar = 1e-6) collapses some components
onto single points (s2 = 1e-6 on data of unit scale: k ~ 1e6; 17 of 256
components at 100k rows of the spherical workload, most components of an
8192-point prefix with 8192 components).  The M-step is unaffected (the
collapsed component takes its point with responsibility ~1 either way), so
weights, means and variances are compared there; the log-likelihood is
compared where k is within range: the embedding workload at the default
regulariser, and the spherical workload with the regulariser expressed in
data units (1e-3 times the mean per-dimension data variance).

Top-m responsibilities of the PRECISE path at fitted parameters.  A
responsibility moves by about r (1 - r) times the error of the logit
difference, and PRECISE resolves a logit to about 2^-22 of the size T of its
expanded-form terms (22-bit operand pieces, fp32 accumulation).  At the fitted
spherical parameters (regulariser 1e-3 of the data variance) max_i T_i r_i
(1 - r_i) over the points' best components is about 1.3e3 log2 units, an error
of 2^-22 * 1.3e3 * ln 2 = 2.2e-4 (measured: 3e-4).  Each entry is therefore
held to the larger of 1e-4 and that bound (gpu_util.precise_resp_tol); the
per-point log-likelihood of PRECISE likewise to the larger of 1e-4 and the
mean of the rows' logit resolution (a row's log-sum-exp moves by at most its
largest logit error).  On the float32 descriptor workload (integers up to
255, fitted standard deviations of a few units) the expanded form's terms
reach ~1e4 log2 units per point: its fitted log-likelihood is off by 7.9e-4
per point against a bound of ~8e-3, while weights, means and variances stay
within 1e-4.

Sharp large-K fit (24576 rows, K = 8192, regulariser 1e-3 of the data
variance: about three points per component).  The top-m pass is compared for
PRECISE (refined by default) and for FAST with the refinement switched on:
the candidates' responsibilities and the log-likelihood come from the
direct-form refinement (topm_refine.cu) and agree to ~1e-5.  FAST without it
is off by up to 6e-2 there (fp16 rounding of the expanded form).  The EM step
is not compared there: the M-step of components holding a few points follows
the expanded-form logits, whose resolution (above) moves their weights by
~4e-3 and means by ~4e-2 of sigma on PRECISE (log-likelihood within the
derived bound)."""
import numpy as np
import pytest
import torch

import em_gmm_step_02_b300 as G
import oracle
import workloads as W
from gpu_util import elementwise_errors, params_to_device, precise_resp_tol
from test_gpu_topm import check_topm

TOL = {"fast": (2e-2, 1e-2), "precise": (1e-4, 1e-4)}

_FIT = {}


def fitted(name, rows, iters, rel_reg):
    """(workload, X, fitted parameters, reg_covar): `iters` oracle EM
    iterations from the workload's starting parameters on its first `rows`
    rows; rel_reg > 0 sets reg_covar to rel_reg times the mean per-dimension
    variance of those rows (else the default 1e-6)."""
    key = (name, rows, iters, rel_reg)
    if key not in _FIT:
        w = W.WORKLOADS[name].scaled(rows)
        X = W.make_data(w)
        Xf = X.float().numpy()
        reg = rel_reg * float(Xf.astype(np.float64).var(axis=0).mean()) if rel_reg > 0 else 1e-6
        init = W.make_init(w, X)
        lw, mu, var, _ = oracle.em_run(Xf, *init, w.cov, iters, reg_covar=reg)
        _FIT[key] = (w, X, tuple(np.asarray(a, np.float32) for a in (lw, mu, var)), reg)
    return _FIT[key]


CASES = [
    # workload, rows, oracle iterations, path, m, relative regulariser, log-likelihood and top-m compared
    ("embed_10m", 20000, 10, "fast", 4, 0.0, True),
    ("spherical_1m", 20000, 10, "precise", 3, 0.0, False),
    ("spherical_1m", 20000, 10, "precise", 3, 1e-3, True),
    ("largek_2m", 8192, 4, "fast", 8, 0.0, False),
    ("descriptor_100m", 20000, 5, "precise", 4, 1e-3, True),   # float32, D = 128: streamed parameters
]

# top-m passes compared: the cases above with the log-likelihood compared, the
# collapsed large-K fit, and both paths at a sharp large-K fit (regulariser in
# data units, about three points per component), where the candidates'
# responsibilities and the log-likelihood come from the direct-form refinement
TOPM_CASES = [c + ("auto",) for c in CASES if c[6] or c[0] == "largek_2m"] + [
    ("largek_2m", 24576, 3, "precise", 8, 1e-3, True, "auto"),
    ("largek_2m", 24576, 3, "fast", 8, 1e-3, True, "on"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,rows,iters,path,m,rel_reg,full", CASES)
def test_em_step_at_fitted_parameters(name, rows, iters, path, m, rel_reg, full):
    w, X, (lw, mu, var), reg = fitted(name, rows, iters, rel_reg)
    tol, tol_ll = TOL[path]
    ref = oracle.em_step(X.float().numpy(), lw, mu, var, w.cov, reg_covar=reg)
    p = params_to_device(lw, mu, var)
    out = G.gmm_em_step(X.cuda(), *p, w.cov, precision=path, reg_covar=reg)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    got = [t.cpu().numpy() for t in out[:3]]
    e_w, e_mu, e_v, msg = elementwise_errors(got, ref, X.shape[0], w.cov, path, tol, w.x_dtype, mu)
    e_ll = abs(float(out[3].item()) - ref[3]) / X.shape[0]
    msg += f" ll/N {e_ll:.2e}"
    if full and path == "precise":
        # the log-likelihood's bound from the logit resolution of PRECISE
        # (gpu_util.precise_resp_tol), over each point's best components
        r_o, i_o, _ = oracle.topm(X.float().numpy(), lw, mu, var, w.cov, m)
        tol_ll = precise_resp_tol(X.float().numpy(), mu, var, w.cov, i_o, r_o, tol, tol_ll)[1]
        msg += f" (bound {tol_ll:.2e})"
    print(msg)
    assert e_w <= 1 and e_mu <= 1 and e_v <= 1, msg
    if full:
        assert e_ll <= tol_ll, msg


@pytest.mark.gpu
@pytest.mark.parametrize("name,rows,iters,path,m,rel_reg,full,refine", TOPM_CASES)
def test_topm_at_fitted_parameters(name, rows, iters, path, m, rel_reg, full, refine):
    w, X, (lw, mu, var), reg = fitted(name, rows, iters, rel_reg)
    tol, tol_ll = TOL[path]
    p = params_to_device(lw, mu, var)
    r, idx, ll = G.gmm_predict_topm(X.cuda(), *p, w.cov, m, precision=path, topm_refine=refine)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    r_o, i_o, ll_o = oracle.topm(X.float().numpy(), lw, mu, var, w.cov, min(m + 1, w.K))
    rtol = tol
    if path == "precise":
        rtol, tol_ll = precise_resp_tol(X.float().numpy(), mu, var, w.cov, i_o[:, :m], r_o[:, :m], tol, tol_ll)
    err, n_sure = check_topm(r.cpu().numpy(), idx.cpu().numpy(), float(ll.item()) if full else None, r_o, i_o,
                             ll_o if full else None, X.shape[0], m, rtol, tol_ll)
    print(f"max |dr| {err:.2e}, {n_sure} separated entries checked")
