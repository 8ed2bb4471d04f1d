"""The bounded device-side waits and their failure report.

Every wait of the kernels polls a bounded number of times.  When one runs
out, the kernel records which barrier and which thread gave up first, every
later wait of the launch returns at once, the launch drains its own in-flight
tensor-core operations and copies (waits that do not give up early), and the
host reports GMM_ERR_TIMEOUT.  Here opts.wait_limit = 1 makes the first wait
that is not already satisfied give up at its first poll: nothing is broken,
a flag that is not yet set is simply not waited for.  The shapes use one CTA
per cluster (K <= 128), so no cross-CTA traffic is in flight when a CTA stops.
The next call with the default limit must be correct (checked against the
float64 oracle)."""
import numpy as np
import pytest
import torch

import em_gmm_step_02_b300 as G
import oracle
import workloads as W
from gpu_util import elementwise_errors, params_to_device
from test_gpu_topm import check_topm

TIMEOUT = -5
TOL = {"fast": (2e-2, 1e-2), "precise": (1e-4, 1e-4)}


def _expect_timeout():
    torch.cuda.synchronize()
    code = G.gmm_stream_status()
    msg = G.gmm_last_error()
    assert code == TIMEOUT, (code, msg)
    assert "thread" in msg and "barrier" in msg, msg
    assert G.gmm_stream_status() == 0          # the status is cleared once read


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,K,cov,xd,path", [
    (4096, 8, 16, "diag", "bf16", "fast"),
    (3000, 12, 40, "diag", "f32", "precise"),
    (2500, 16, 8, "tied", "f32", "precise"),
])
def test_em_step_wait_limit_then_normal_call(N, D, K, cov, xd, path):
    w = W.generic(N, D, K, cov, xd, seed=N + K)
    X = W.make_data(w)
    lw, mu, var = W.make_init(w, X)
    p = params_to_device(lw, mu, var)
    Xd = X.cuda()
    G.gmm_em_step(Xd, *p, cov, precision=path, wait_limit=1)
    _expect_timeout()
    out = G.gmm_em_step(Xd, *p, cov, precision=path)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    tol, tol_ll = TOL[path]
    if cov == "tied":
        ref = oracle.tied.em_step(X.float().numpy().astype(np.float64), lw, mu, var)
        got = [t.cpu().numpy().astype(np.float64) for t in out[:3]]
        assert np.abs(got[1] - ref[1]).max() <= tol * np.abs(ref[1]).max()
        assert np.abs(got[2] - ref[2]).max() <= tol * np.abs(ref[2]).max()
    else:
        ref = oracle.em_step(X.float().numpy(), lw, mu, var, cov)
        e_w, e_mu, e_v, msg = elementwise_errors([t.cpu().numpy() for t in out[:3]], ref, N, cov, path, tol, xd, mu)
        assert e_w <= 1 and e_mu <= 1 and e_v <= 1, msg
    assert abs(float(out[3].item()) - ref[3]) / N <= tol_ll


@pytest.mark.gpu
def test_topm_wait_limit_then_normal_call():
    N, D, K, m = 3000, 32, 100, 4
    w = W.generic(N, D, K, "diag", "bf16", seed=21)
    X = W.make_data(w)
    lw, mu, var = W.make_init(w, X)
    p = params_to_device(lw, mu, var)
    Xd = X.cuda()
    G.gmm_predict_topm(Xd, *p, "diag", m, wait_limit=1)
    _expect_timeout()
    r, idx, ll = G.gmm_predict_topm(Xd, *p, "diag", m)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    r_o, i_o, ll_o = oracle.topm(X.float().numpy(), lw, mu, var, "diag", m + 1)
    check_topm(r.cpu().numpy(), idx.cpu().numpy(), float(ll.item()), r_o, i_o, ll_o, N, m, *TOL["fast"])
