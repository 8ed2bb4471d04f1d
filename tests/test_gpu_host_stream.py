"""gmm_em_step_host: the EM step over X held in host memory, streamed to the
GPU in chunks whose copies overlap the fused kernel.  The statistics of all
chunks add into one set of partials, so the step must equal gmm_em_step over
the same rows up to the order of floating-point sums (checked tightly), and
must meet the oracle's parity bounds (checked on a small case with a ragged
last chunk).  Cases cover one pass (clusters), the two-pass plan (K > 1024),
the PRECISE path, and a chunk size that is not a multiple of the tile."""
import numpy as np
import pytest
import torch

import em_gmm_step_02_b300 as G
import oracle
import workloads as W
from gpu_util import params_to_device, rel_l2_rows

TOL = {"precise": (1e-4, 1e-4), "fast": (2e-2, 1e-2)}


def _absmax(X):
    return float(X.abs().max().item()) * 1.0001 + 1e-30


def _np(out):
    return [t.cpu().numpy().astype(np.float64) for t in out]


def _rel(a, b, N):
    lw_a, mu_a, var_a, ll_a = a
    lw_b, mu_b, var_b, ll_b = b
    K = len(lw_a)
    return (np.abs(np.exp(lw_a) - np.exp(lw_b)).max(),
            rel_l2_rows(mu_a, mu_b).max(),
            rel_l2_rows(var_a.reshape(K, -1), var_b.reshape(K, -1)).max(),
            abs(ll_a[0] - ll_b[0]) / N)


def _both(w, X, chunk_rows, precision="auto"):
    init = W.make_init(w, X)
    p = params_to_device(*init)
    amax = _absmax(X)
    dev = G.gmm_em_step(X.cuda(), *p, w.cov, precision=precision, x_absmax=amax)
    host = G.gmm_em_step_host(X.pin_memory(), *p, w.cov, chunk_rows=chunk_rows, precision=precision,
                              x_absmax=amax)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    return init, _np(dev), _np(host)


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,K,cov,xd,chunk", [
    (5000, 32, 64, "diag", "bf16", 1024),        # 5 chunks, the last one ragged
    (3001, 48, 40, "diag", "f32", 640),          # PRECISE
    (12000, 32, 1100, "diag", "bf16", 4000),     # two-pass plan per chunk; 4000 -> 3968 rows
    (4096, 64, 256, "spherical", "f32", 128),    # 32 one-tile chunks
    (3000, 128, 100, "diag", "f32", 1024),       # PRECISE with the streamed parameter image
])
def test_host_stream_matches_device_step_and_oracle(N, D, K, cov, xd, chunk):
    w = W.generic(N, D, K, cov, xd, seed=N + K)
    X = W.make_data(w)
    init, dev, host = _both(w, X, chunk)
    e_w, e_mu, e_var, e_ll = _rel(host, dev, N)
    # same arithmetic, other order of the sums (fp32 partials are flushed at
    # every chunk's end): far inside the parity bounds, far outside a lost chunk
    assert e_w <= 1e-5 and e_mu <= 1e-4 and e_var <= 1e-3 and e_ll <= 1e-4, (e_w, e_mu, e_var, e_ll)
    ref = oracle.em_step(X.float().numpy(), *init, w.cov)
    path = "fast" if xd == "bf16" else "precise"
    tol, tol_ll = TOL[path]
    r_w, r_mu, r_var, r_ll = _rel(host, [np.asarray(ref[0]), np.asarray(ref[1]), np.asarray(ref[2]),
                                         np.array([ref[3]])], N)
    assert r_mu <= tol and r_ll <= tol_ll, (r_mu, r_ll)


@pytest.mark.gpu
def test_host_stream_two_million_rows_of_the_embedding_workload():
    w = W.WORKLOADS["embed_10m"].scaled(2_000_000)
    X = W.make_data(w)
    _, dev, host = _both(w, X, 1 << 19)     # 4 chunks of 524,288 rows
    e_w, e_mu, e_var, e_ll = _rel(host, dev, X.shape[0])
    assert e_w <= 1e-5 and e_mu <= 1e-4 and e_var <= 1e-3 and e_ll <= 1e-4, (e_w, e_mu, e_var, e_ll)


@pytest.mark.gpu
def test_host_stream_needs_a_bound_on_x():
    w = W.generic(1000, 8, 4, "diag", "f32", seed=3)
    X = W.make_data(w)
    p = params_to_device(*W.make_init(w, X))
    with pytest.raises(G.GmmError):
        G.gmm_em_step_host(X.pin_memory(), *p, w.cov)
