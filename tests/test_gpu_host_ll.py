"""The log-likelihood delivered to a host pointer (gmm_opts.loglik_on_host = 1,
through the C ABI directly): the call waits for the stream, writes the same
double the device-pointer call writes, and reports device-side errors itself.
Covers the exact EM step (one and two passes), approximate top-k EM and the
top-m pass."""
import ctypes

import numpy as np
import pytest
import torch

import em_gmm_step_02_b300 as G
import workloads as W
from gpu_util import params_to_device

vp = ctypes.c_void_p


def _ptr(t):
    return vp(t.data_ptr())


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,K,cov,xd,k", [
    (3000, 32, 100, "diag", "bf16", 0),
    (3000, 32, 100, "diag", "bf16", 4),
    (4000, 16, 1100, "diag", "bf16", 0),      # two passes
    (2500, 24, 50, "spherical", "f32", 3),
])
def test_em_step_loglik_on_host(N, D, K, cov, xd, k):
    w = W.generic(N, D, K, cov, xd, seed=N + K + k)
    X = W.make_data(w).cuda()
    p = params_to_device(*W.make_init(w, X.cpu()))
    dev = G.gmm_em_step(X, *p, cov, approx_top_k=k)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    out = [torch.empty_like(a) for a in p]
    o = G.gmm_default_opts(approx_top_k=k)
    o.loglik_on_host = 1
    ll = ctypes.c_double(0.0)
    rc = G.lib().gmm_em_step(_ptr(X), N, D, K, G.COV[cov], G.F32 if xd == "f32" else G.BF16,
                             _ptr(p[0]), _ptr(p[1]), _ptr(p[2]), _ptr(out[0]), _ptr(out[1]), _ptr(out[2]),
                             ctypes.byref(ll), ctypes.byref(o), vp(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, G.gmm_last_error()
    assert ll.value == float(dev[3].item())
    for a, b in zip(out, dev[:3]):
        assert torch.equal(a, b)


@pytest.mark.gpu
def test_topm_loglik_on_host():
    N, D, K, m = 3000, 32, 100, 4
    w = W.generic(N, D, K, "diag", "bf16", seed=3)
    X = W.make_data(w).cuda()
    p = params_to_device(*W.make_init(w, X.cpu()))
    r, idx, ll_dev = G.gmm_predict_topm(X, *p, "diag", m)
    torch.cuda.synchronize()
    r2 = torch.empty_like(r)
    i2 = torch.empty_like(idx)
    o = G.gmm_default_opts()
    o.loglik_on_host = 1
    ll = ctypes.c_double(0.0)
    rc = G.lib().gmm_predict_topm(_ptr(X), N, D, K, G.DIAG, G.BF16, _ptr(p[0]), _ptr(p[1]), _ptr(p[2]), m,
                                  _ptr(r2), _ptr(i2), ctypes.byref(ll), ctypes.byref(o),
                                  vp(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, G.gmm_last_error()
    assert ll.value == float(ll_dev.item())
    assert torch.equal(r, r2) and torch.equal(idx, i2)


@pytest.mark.gpu
def test_loglik_on_host_reports_device_errors():
    """A non-positive variance is found on the device; with the log-likelihood
    on the host the call itself returns GMM_ERR_NONFINITE."""
    N, D, K = 1000, 8, 8
    w = W.generic(N, D, K, "diag", "f32", seed=2)
    X = W.make_data(w).cuda()
    lw, mu, var = W.make_init(w, X.cpu())
    var = np.array(var, copy=True)
    var[3, 2] = 0.0
    p = params_to_device(lw, mu, var)
    out = [torch.empty_like(a) for a in p]
    o = G.gmm_default_opts()
    o.loglik_on_host = 1
    ll = ctypes.c_double(0.0)
    rc = G.lib().gmm_em_step(_ptr(X), N, D, K, G.DIAG, G.F32, _ptr(p[0]), _ptr(p[1]), _ptr(p[2]),
                             _ptr(out[0]), _ptr(out[1]), _ptr(out[2]), ctypes.byref(ll), ctypes.byref(o),
                             vp(torch.cuda.current_stream().cuda_stream))
    assert rc == -3, (rc, G.gmm_last_error())
    assert G.gmm_stream_status() == 0     # the status was read and cleared by the call
