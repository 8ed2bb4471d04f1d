"""Parity at the workloads' operating point: one EM step and one top-m pass
from FITTED parameters (several oracle EM iterations from the workload's
starting point), compared with the float64 oracle element by element.

The workloads run their final top-m pass after their EM iterations, so this is
where the multi-assignment of "Flash-GMM: A Memory-Efficient Kernel for
Scalable Soft Clustering" (conclusion: assignments read off the final
responsibilities) is used; fitted components are sharp, which is where the
expanded-form logits of the fp16 path are hardest.

Bounds (see gpu_util.elementwise_errors): per element, weights relative,
means relative to max(|mu|, sigma), variances relative or within four
rounding units of the raw second moment; the per-point mean log-likelihood
within the path's absolute bound; top-m responsibilities within the path's
tolerance and indices identical wherever the responsibility gap to the
neighbouring entries exceeds that tolerance."""
import numpy as np
import pytest
import torch

import em_gmm_step_02_b300 as G
import oracle
import workloads as W
from gpu_util import elementwise_errors, params_to_device
from test_gpu_topm import check_topm

TOL = {"fast": (2e-2, 1e-2), "precise": (1e-4, 1e-4)}

_FIT = {}


def fitted(name, rows, iters):
    """(workload, X, fitted parameters): `iters` oracle EM iterations from the
    workload's starting parameters on its first `rows` rows."""
    key = (name, rows, iters)
    if key not in _FIT:
        w = W.WORKLOADS[name].scaled(rows)
        X = W.make_data(w)
        init = W.make_init(w, X)
        lw, mu, var, _ = oracle.em_run(X.float().numpy(), *init, w.cov, iters)
        _FIT[key] = (w, X, tuple(np.asarray(a, np.float32) for a in (lw, mu, var)))
    return _FIT[key]


CASES = [
    # workload, rows, oracle iterations, path, m
    ("embed_10m", 20000, 10, "fast", 4),
    ("spherical_1m", 20000, 10, "precise", 3),
    ("largek_2m", 8192, 4, "fast", 8),
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,rows,iters,path,m", CASES)
def test_em_step_at_fitted_parameters(name, rows, iters, path, m):
    w, X, (lw, mu, var) = fitted(name, rows, iters)
    tol, tol_ll = TOL[path]
    ref = oracle.em_step(X.float().numpy(), lw, mu, var, w.cov)
    p = params_to_device(lw, mu, var)
    out = G.gmm_em_step(X.cuda(), *p, w.cov, precision=path)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    got = [t.cpu().numpy() for t in out[:3]]
    e_w, e_mu, e_v, msg = elementwise_errors(got, ref, w.cov, path, tol)
    e_ll = abs(float(out[3].item()) - ref[3]) / X.shape[0]
    msg += f" ll/N {e_ll:.2e}"
    print(msg)
    assert e_w <= 1 and e_mu <= 1 and e_v <= 1 and e_ll <= tol_ll, msg


@pytest.mark.gpu
@pytest.mark.parametrize("name,rows,iters,path,m", CASES)
def test_topm_at_fitted_parameters(name, rows, iters, path, m):
    w, X, (lw, mu, var) = fitted(name, rows, iters)
    tol, tol_ll = TOL[path]
    p = params_to_device(lw, mu, var)
    r, idx, ll = G.gmm_predict_topm(X.cuda(), *p, w.cov, m, precision=path)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    r_o, i_o, ll_o = oracle.topm(X.float().numpy(), lw, mu, var, w.cov, min(m + 1, w.K))
    err, n_sure = check_topm(r.cpu().numpy(), idx.cpu().numpy(), float(ll.item()), r_o, i_o, ll_o,
                             X.shape[0], m, tol, tol_ll)
    print(f"max |dr| {err:.2e}, {n_sure} separated entries checked")
