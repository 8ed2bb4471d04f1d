"""Parity of the CUDA threshold multi-assignment (gmm_assign_threshold,
through the C ABI): the compressed rows of every (point, component) pair with
responsibility >= tau, best first, against the oracle's definition on the
float64 responsibilities.

A pair whose responsibility lies within the path's tolerance of tau may fall
on either side under rounding; every other pair must be kept or dropped
exactly as the oracle does, with its responsibility within the tolerance.
The rows must also be exactly the top-m pass's lists cut at tau (the same
kernels produce both), offsets must survive an overflowing capacity, and the
two-pass plan (K > 1024) must agree too."""
import numpy as np
import pytest
import torch

import em_gmm_step_02_b300 as G
import oracle
import workloads as W
from gpu_util import params_to_device

TOL = {"fast": 2e-2, "precise": 1e-4}


def _check(off, idx, resp, r_ref, tau, m, tol):
    N, K = r_ref.shape
    off = off.astype(np.int64)
    assert off[0] == 0 and (np.diff(off) >= 0).all() and off[-1] == len(idx) == len(resp)
    n_sure = 0
    for i in range(N):
        ks = idx[off[i]:off[i + 1]]
        rs = resp[off[i]:off[i + 1]].astype(np.float64)
        assert len(ks) <= m and len(set(ks.tolist())) == len(ks)
        assert (np.diff(rs) <= 1e-6).all()
        assert (np.abs(rs - r_ref[i, ks]) <= tol).all()
        # kept pairs are not clearly below tau; clearly-above pairs among the
        # point's m largest are kept
        assert (r_ref[i, ks] >= tau - tol).all()
        top = np.lexsort((np.arange(K), -r_ref[i]))[:m]
        must = [k for k in top if r_ref[i, k] >= tau + tol]
        assert set(must) <= set(ks.tolist()), (i, must, ks)
        n_sure += len(must)
    return n_sure


def _run(X_cpu, lw, mu, var, cov, tau, m, **kw):
    p = params_to_device(lw, mu, var)
    off, idx, resp = G.gmm_assign_threshold(X_cpu.cuda(), *p, cov, tau=tau, max_per_point=m, **kw)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    return off.cpu().numpy(), idx.cpu().numpy(), resp.cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,K,cov,xd,tau,m", [
    (3001, 96, 200, "diag", "bf16", 0.1, 9),
    (4096, 8, 16, "diag", "f32", 0.05, 16),
    (12000, 32, 1100, "diag", "bf16", 0.2, 4),      # two-pass plan
    (5000, 64, 256, "spherical", "f32", 0.3, 3),
    (3000, 128, 100, "diag", "f32", 0.2, 4),         # PRECISE, 128 features
])
def test_threshold_against_oracle(N, D, K, cov, xd, tau, m):
    w = W.generic(N, D, K, cov, xd, seed=N + 5 * D + K)
    X = W.make_data(w)
    lw, mu, var = W.make_init(w, X)
    off, idx, resp = _run(X, lw, mu, var, cov, tau, m)
    r_ref, _ = oracle.responsibilities(X.float().numpy(), lw, mu, var, cov)
    path = "fast" if xd == "bf16" else "precise"
    n_sure = _check(off, idx, resp, r_ref, tau, m, TOL[path])
    assert n_sure > 0
    print(f"{off[-1]} entries, {n_sure} clear of the threshold checked")


@pytest.mark.gpu
def test_threshold_rows_are_the_topm_lists_cut_at_tau():
    # 300,000 points: 1,172 blocks of counts, so the scan of block totals
    # carries across two chunks of 1,024
    w = W.WORKLOADS["embed_10m"].scaled(300_000)
    X = W.make_data(w).cuda()
    p = params_to_device(*W.make_init(w, X.cpu()))
    tau, m = 0.05, 8
    r, i, _ = G.gmm_predict_topm(X, *p, w.cov, m)
    off, idx, resp = G.gmm_assign_threshold(X, *p, w.cov, tau=tau, max_per_point=m)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    keep = (r >= tau)
    cnt = keep.sum(1)
    assert torch.equal(off[1:] - off[:-1], cnt.to(torch.int64))
    assert torch.equal(idx, i[keep]) and torch.equal(resp, r[keep])


@pytest.mark.gpu
def test_threshold_capacity_overflow_keeps_offsets():
    w = W.generic(2000, 16, 20, "diag", "f32", seed=5)
    X = W.make_data(w).cuda()
    p = params_to_device(*W.make_init(w, X.cpu()))
    off_full, _, _ = G.gmm_assign_threshold(X, *p, w.cov, tau=0.1, max_per_point=8)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0
    assert int(off_full[-1].item()) > 3
    off_c, _, _ = G.gmm_assign_threshold(X, *p, w.cov, tau=0.1, max_per_point=8, capacity=3)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == -7          # GMM_ERR_CAPACITY, reported by the stream status
    assert torch.equal(off_c, off_full)
