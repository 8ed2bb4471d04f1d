"""Parity of the CUDA EM step (through the C ABI) with the float64 oracle,
element by element (gpu_util.elementwise_errors states the denominators).

Tolerances follow the method's stated accuracy targets:
  PRECISE (float32 data): weights, means and variances within 1e-4
      relative; per-point mean log-likelihood within 1e-4 (absolute).
  FAST (bf16 data): 2e-2 relative and 1e-2 (absolute) per-point mean
      log-likelihood; the log-likelihood after 20 iterations within 1e-3
      relative.
"""
import numpy as np
import pytest
import torch

import em_gmm_step_02_b300 as G
import oracle
import workloads as W
from gpu_util import elementwise_errors, params_to_device, rel_l2_rows

TOL = {"precise": (1e-4, 1e-4), "fast": (2e-2, 1e-2)}


def run_gpu(X_cpu, lw, mu, var, cov, precision="auto", **kw):
    X = X_cpu.cuda()
    lw_d, mu_d, var_d = params_to_device(lw, mu, var)
    out = G.gmm_em_step(X, lw_d, mu_d, var_d, cov, precision=precision, **kw)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0
    return [t.cpu().numpy() for t in out[:3]] + [float(out[3].item())]


def compare(got, ref, N, cov, path, x_dtype, means_in):
    tol, tol_ll = TOL[path]
    e_w, e_mu, e_v, msg = elementwise_errors(got[:3], ref, N, cov, path, tol, x_dtype, means_in)
    e_ll = abs(got[3] - ref[3]) / N
    msg += f" ll/N {e_ll:.2e} (tol {tol}, {tol_ll})"
    assert e_w <= 1 and e_mu <= 1 and e_v <= 1 and e_ll <= tol_ll, msg
    return msg


def one_step_case(w, rows=None, precision="auto", path=None):
    X = W.make_data(w, rows)
    init = W.make_init(w, X)
    ref = oracle.em_step(X.float().numpy(), *init, w.cov)
    got = run_gpu(X, *init, w.cov, precision)
    if path is None:
        path = "fast" if (precision == "fast" or (precision == "auto" and w.x_dtype == "bf16")) else "precise"
    return compare(got, ref, X.shape[0], w.cov, path, w.x_dtype, init[1])


# --------------------------------------------------------------------------- small shapes
CASES = [
    # N, D, K, cov, x_dtype, precision
    (4096, 8, 16, "diag", "f32", "auto"),
    (3001, 63, 40, "diag", "f32", "auto"),
    (1000, 1, 3, "diag", "f32", "auto"),
    (3777, 17, 129, "spherical", "f32", "auto"),
    (5000, 64, 256, "spherical", "f32", "auto"),
    (3001, 96, 200, "diag", "bf16", "auto"),
    (20000, 128, 1024, "diag", "bf16", "auto"),
    (1500, 8, 1, "diag", "bf16", "auto"),
    (2500, 100, 300, "diag", "f32", "fast"),
    (12000, 32, 1100, "diag", "bf16", "auto"),
    (129, 5, 7, "spherical", "bf16", "auto"),
    # float32 data with D > 64: PRECISE with the parameter image streamed per tile
    (3001, 128, 256, "diag", "f32", "auto"),
    (2500, 100, 300, "diag", "f32", "auto"),
    (4000, 96, 129, "spherical", "f32", "auto"),
    (6000, 128, 1100, "diag", "f32", "auto"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,K,cov,xd,prec", CASES)
def test_one_step_small(N, D, K, cov, xd, prec):
    w = W.generic(N, D, K, cov, xd, seed=N + D + K)
    print(one_step_case(w, precision=prec))


SPLIT_CASES = [
    (4096, 8, 16, "diag", "f32", "auto"),
    (3777, 17, 129, "spherical", "f32", "auto"),
    (20000, 128, 1024, "diag", "bf16", "auto"),
    (12000, 32, 1100, "diag", "bf16", "auto"),
    (3001, 96, 200, "diag", "bf16", "auto"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,K,cov,xd,prec", SPLIT_CASES)
def test_one_step_small_split_plan(N, D, K, cov, xd, prec):
    """The two-pass plan (normalisers through memory) against the oracle."""
    w = W.generic(N, D, K, cov, xd, seed=N + D + K)
    X = W.make_data(w)
    init = W.make_init(w, X)
    ref = oracle.em_step(X.float().numpy(), *init, w.cov)
    got = run_gpu(X, *init, w.cov, prec, plan="split")
    path = "fast" if xd == "bf16" else "precise"
    print(compare(got, ref, X.shape[0], w.cov, path, xd, init[1]))


def _moments_ok(X, lw2, mu2, var2, reg=1e-6):
    N = X.shape[0]
    pi = torch.exp(lw2.double())
    assert abs(pi.sum().item() - 1.0) < 1e-5
    Nk = pi * N
    s1 = (Nk[:, None] * mu2.double()).sum(0)
    xs = X.double().sum(0)
    assert ((s1 - xs).abs() / X.double().abs().sum(0)).max().item() < 2e-3
    s2 = (Nk[:, None] * (var2.double() - reg + mu2.double() ** 2)).sum(0)
    x2 = (X.double() ** 2).sum(0)
    assert ((s2 - x2).abs() / x2).max().item() < 2e-2


@pytest.mark.gpu
@pytest.mark.parametrize("K,plan", [(100, "cluster"), (100, "split"), (1000, "split")])
def test_long_run_moments_and_plans_agree(K, plan):
    """Two million points: enough tiles per CTA for every hand-off of the
    pipeline to wrap many times (a single 128-component slice runs without
    the cluster exchange, the fastest schedule).  Moments are conserved and
    the result agrees with the other plan."""
    w = W.generic(2_000_000, 128, K, "diag", "bf16", seed=3)
    X = W.make_data(w, device="cuda")
    init = W.make_init(w, X)
    p = params_to_device(*init)
    a = G.gmm_em_step(X, *p, w.cov, plan=plan)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    _moments_ok(X, *a[:3])
    other = "split" if plan == "cluster" else "cluster"
    b = G.gmm_em_step(X, *p, w.cov, plan=other)
    torch.cuda.synchronize()
    assert G.gmm_stream_status() == 0, G.gmm_last_error()
    assert rel_l2_rows(a[1].cpu().numpy(), b[1].cpu().numpy()).max() < 2e-2
    assert abs(a[3].item() - b[3].item()) / X.shape[0] < 1e-2


@pytest.mark.gpu
def test_tiny_workload_20_iterations():
    w = W.WORKLOADS["tiny_diag"]
    X = W.make_data(w)
    lw, mu, var = W.make_init(w, X)
    Xf = X.numpy()
    ref_lls = []
    ref = (lw.astype(np.float64), mu.astype(np.float64), var.astype(np.float64))
    for _ in range(w.iters):
        *ref, ll = oracle.em_step(Xf, *ref, w.cov)
        ref_lls.append(ll)
    Xd = X.cuda()
    p = params_to_device(lw, mu, var)
    lls = []
    for _ in range(w.iters):
        *p, ll = G.gmm_em_step(Xd, *p, w.cov)
        lls.append(float(ll.item()))
    got = [t.cpu().numpy() for t in p]
    N = X.shape[0]
    assert np.abs(np.asarray(lls) - np.asarray(ref_lls)).max() / N <= 1e-4, (lls, ref_lls)
    assert rel_l2_rows(got[1], ref[1]).max() <= 1e-4


# --------------------------------------------------------------------------- workload prefixes
@pytest.mark.gpu
@pytest.mark.parametrize("name,rows,prec", [
    ("spherical_1m", 20000, "auto"),
    ("embed_10m", 20000, "auto"),
    ("descriptor_100m", 20000, "auto"),    # float32, D = 128: PRECISE
    ("descriptor_100m", 20000, "fast"),
    ("largek_2m", 30000, "auto"),
])
def test_workload_prefix_one_step(name, rows, prec):
    w = W.WORKLOADS[name]
    print(one_step_case(w.scaled(rows), precision=prec))


@pytest.mark.gpu
def test_embed_prefix_20_iterations_ll():
    w = W.WORKLOADS["embed_10m"].scaled(20000)
    X = W.make_data(w)
    lw, mu, var = W.make_init(w, X)
    *_, ref_lls = oracle.em_run(X.float().numpy(), lw, mu, var, w.cov, 20)
    Xd = X.cuda()
    p = params_to_device(lw, mu, var)
    for _ in range(20):
        *p, ll = G.gmm_em_step(Xd, *p, w.cov)
    got = float(ll.item())
    assert abs(got - ref_lls[-1]) / abs(ref_lls[-1]) <= 1e-3, (got, ref_lls[-1])


# --------------------------------------------------------------------------- properties
@pytest.mark.gpu
def test_outputs_may_alias_inputs_and_runs_are_deterministic():
    w = W.generic(3000, 40, 300, "diag", "bf16", seed=5)
    X = W.make_data(w).cuda()
    init = W.make_init(w, X.cpu())
    a = params_to_device(*init)
    b = params_to_device(*init)
    r1 = G.gmm_em_step(X, *a, w.cov)
    G.gmm_em_step(X, *b, w.cov, out=b)        # in place
    torch.cuda.synchronize()
    for x, y in zip(r1[:3], b):
        assert torch.equal(x, y)
    r2 = G.gmm_em_step(X, *a, w.cov)
    for x, y in zip(r1, r2):
        assert torch.equal(x, y)


@pytest.mark.gpu
def test_dead_component_keeps_parameters():
    w = W.generic(2000, 16, 20, "diag", "f32", seed=9)
    X = W.make_data(w)
    lw, mu, var = W.make_init(w, X)
    lw = lw.copy()
    lw[3] = -np.inf
    got = run_gpu(X, lw, mu, var, "diag")
    assert got[0][3] == -np.inf
    np.testing.assert_array_equal(got[1][3], mu[3])
    np.testing.assert_array_equal(got[2][3], var[3])
    ref = oracle.em_step(X.numpy(), lw, mu, var, "diag")
    keep = [k for k in range(20) if k != 3]
    assert rel_l2_rows(got[1][keep], ref[1][keep]).max() < 1e-4


@pytest.mark.gpu
def test_nonpositive_variance_is_reported():
    w = W.generic(500, 4, 3, "diag", "f32", seed=1)
    X = W.make_data(w).cuda()
    lw, mu, var = W.make_init(w, X.cpu())
    var = var.copy()
    var[1, 2] = 0.0
    G.gmm_em_step(X, *params_to_device(lw, mu, var), "diag")
    assert G.gmm_stream_status() == -3
    assert G.gmm_stream_status() == 0     # status is cleared once read


@pytest.mark.gpu
def test_conservation_of_moments_full_size_embed():
    """Full 10M x 128 x 1024 workload in the benchmark's launch configurations
    (both plans): properties that hold at any size (weights sum to 1;
    sum_k N_k mu_k equals the data sum; sum_k N_k (s2_k + mu_k^2) equals the
    sum of squares)."""
    w = W.WORKLOADS["embed_10m"]
    X = W.make_data(w, device="cuda")
    lw, mu, var = W.make_init(w, X)
    p = params_to_device(lw, mu, var)
    for plan in ("cluster", "split"):
        lw2, mu2, var2, ll = G.gmm_em_step(X, *p, w.cov, plan=plan)
        torch.cuda.synchronize()
        assert G.gmm_stream_status() == 0, G.gmm_last_error()
        _moments_ok(X, lw2, mu2, var2)
        assert np.isfinite(ll.item())


# --------------------------------------------------------------------------- flush periods
@pytest.mark.gpu
@pytest.mark.parametrize("N,D,K,cov,xd,path", [
    (800_000, 8, 1024, "diag", "bf16", "fast"),
    (500_000, 64, 256, "diag", "f32", "precise"),
    (500_000, 128, 256, "diag", "f32", "precise"),
])
def test_several_flush_periods_against_oracle(N, D, K, cov, xd, path):
    """Every CTA accumulates at least three flush periods of statistics in
    tensor memory before the fixed-order reduction (the periodic flush, not
    only the one at the end of the CTA's tiles, is compared with the oracle)."""
    info = G.gmm_plan_info(N, D, K, cov, xd, precision=path)
    assert info["tiles"] // info["tile_groups"] >= 3 * info["flush_tiles"], info
    w = W.generic(N, D, K, cov, xd, seed=N % 997 + K)
    X = W.make_data(w)
    init = W.make_init(w, X)
    ref = oracle.em_step(X.float().numpy(), *init, cov)
    got = run_gpu(X, *init, cov, path)
    print(compare(got, ref, N, cov, path, xd, init[1]))
