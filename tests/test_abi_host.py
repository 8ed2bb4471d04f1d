"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/gmm.h declares, rejects bad arguments before touching
the device, and plans a workspace that does not grow with N (the O(K D)
memory claim) while a naive EM's responsibility matrix would."""
import ctypes
import os

import pytest

import em_gmm_step_02_b300 as G

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "naive_footprint.txt")


def test_library_exports_every_declared_symbol():
    lib = G.lib()
    names = G.declared_symbols()
    assert "gmm_em_step" in names and "gmm_predict_topm" in names
    for n in names:
        assert hasattr(lib, n), n


def test_default_opts():
    o = G.gmm_default_opts()
    assert o.precision == 0 and o.loglik_on_host == 0
    assert abs(o.reg_covar - 1e-6) < 1e-12 and o.var_floor == 0.0 and o.x_absmax == 0.0
    assert o.approx_top_k == 0 and o.topm_refine == 0 and o.plan == 0 and o.wait_limit == 0
    # every field is written, whatever the struct held before
    junk = G.gmm_opts(precision=7, approx_top_k=9, topm_refine=5, wait_limit=3, plan=4)
    G.lib().gmm_default_opts(ctypes.byref(junk))
    assert (junk.precision, junk.approx_top_k, junk.topm_refine, junk.wait_limit, junk.plan) == (0, 0, 0, 0, 0)


@pytest.mark.parametrize("v", [-1, 3])
def test_topm_refine_argument_error(v):
    assert _call(opts=G.gmm_default_opts(topm_refine=v)) == -1
    assert "topm_refine" in G.gmm_last_error()
    # a valid setting passes this check (the call may still fail later, e.g.
    # for want of a device)
    _call(opts=G.gmm_default_opts(topm_refine="on"))
    assert "topm_refine" not in G.gmm_last_error()


def _call(N=100, D=8, K=4, cov=1, dt=0, X=0x1000, p=0x2000, ll=0x3000, opts=None):
    o = opts or G.gmm_default_opts()
    vp = ctypes.c_void_p
    return G.lib().gmm_em_step(vp(X), N, D, K, cov, dt, vp(p), vp(p), vp(p), vp(p), vp(p), vp(p),
                               vp(ll), ctypes.byref(o), vp(0))


@pytest.mark.parametrize("kw,code", [
    (dict(N=0), -1), (dict(D=0), -1), (dict(K=0), -1), (dict(cov=3), -1), (dict(dt=3), -1),
    (dict(X=0), -1), (dict(X=0x1004), -1), (dict(p=0x2002), -1), (dict(ll=0), -1),
    (dict(D=129), -2), (dict(K=8193), -2),
])
def test_argument_errors_are_found_on_the_host(kw, code):
    assert _call(**kw) == code
    assert G.gmm_last_error() != ""


def test_approx_top_k_argument_errors_are_found_on_the_host():
    assert _call(K=40, opts=G.gmm_default_opts(approx_top_k=-1)) == -1
    assert _call(K=40, opts=G.gmm_default_opts(approx_top_k=17)) == -2
    assert _call(K=40, cov=2, D=8, opts=G.gmm_default_opts(approx_top_k=4)) == -2
    assert "approx_top_k" in G.gmm_last_error()
    assert _call(N=1 << 31, K=40, opts=G.gmm_default_opts(approx_top_k=4)) == -2
    vp = ctypes.c_void_p
    o = G.gmm_default_opts(approx_top_k=2)
    assert G.lib().gmm_em_step_noalloc(vp(0x1000), 100, 8, 40, 1, 0, vp(0x2000), vp(0x2000), vp(0x2000),
                                       vp(0x2000), vp(0x2000), vp(0x2000), vp(0x3000), ctypes.byref(o),
                                       vp(0)) == -2


def test_host_stream_argument_errors_are_found_on_the_host():
    vp = ctypes.c_void_p
    lib = G.lib()

    def call(X=0x1000, amax=1.0, chunk=0, N=100):
        o = G.gmm_default_opts(x_absmax=amax)
        return lib.gmm_em_step_host(vp(X), N, 8, 4, 1, 0, vp(0x2000), vp(0x2000), vp(0x2000), vp(0x2000),
                                    vp(0x2000), vp(0x2000), vp(0x3000), chunk, ctypes.byref(o), vp(0))
    assert call(X=0) == -1
    assert call(amax=0.0) == -1 and "x_absmax" in G.gmm_last_error()
    assert call(chunk=-5) == -1
    assert call(N=0) == -1


def test_threshold_assignment_argument_errors_are_found_on_the_host():
    vp = ctypes.c_void_p
    lib = G.lib()

    def call(tau=0.3, m=4, off=0x4000, cap=10, K=8):
        o = G.gmm_default_opts()
        return lib.gmm_assign_threshold(vp(0x1000), 100, 8, K, 1, 0, vp(0x2000), vp(0x2000), vp(0x2000),
                                        ctypes.c_float(tau), m, vp(off), vp(0x5000), vp(0x6000), cap,
                                        ctypes.byref(o), vp(0))
    assert call(tau=0.0) == -1 and call(tau=1.5) == -1 and call(tau=float("nan")) == -1
    assert call(m=0) == -2 and call(m=17) == -2 and call(m=9, K=8) == -1
    assert call(off=0) == -1 and call(off=0x4004) == -1 and call(cap=-1) == -1


def test_tied_covariance_is_refused_where_not_supported():
    vp = ctypes.c_void_p
    lib = G.lib()
    o = G.gmm_default_opts(x_absmax=1.0)
    args = (vp(0x1000), 100, 8, 4, 2, 0, vp(0x2000), vp(0x2000), vp(0x2000), vp(0x2000), vp(0x2000),
            vp(0x2000), vp(0x3000))
    assert lib.gmm_em_step_host(*args, 0, ctypes.byref(o), vp(0)) == -2
    assert lib.gmm_em_step_noalloc(*args, ctypes.byref(o), vp(0)) == -2
    assert "spherical and diagonal" in G.gmm_last_error()


def test_bad_options_rejected():
    assert _call(opts=G.gmm_default_opts(precision=7)) == -1
    assert _call(opts=G.gmm_default_opts(reg_covar=-1.0)) == -1
    assert _call(opts=G.gmm_default_opts(var_floor=float("nan"))) == -1


def test_workspace_is_independent_of_N_and_far_below_naive_footprint():
    # page numbers: N = 10M, D = 128, K = 2048 at 4 bytes -> R about 80 GB, X about 5 GB
    N, D, K, bpv, r_gb, x_gb = [float(v) for v in open(GOLDEN).read().split("\n")[-2].split()]
    assert abs(N * K * bpv / 1e9 - r_gb) / r_gb < 0.05
    assert abs(N * D * bpv / 1e9 - x_gb) / x_gb < 0.05
    a = G.gmm_workspace_bytes(1_000_000, 128, 1024, "diag", "bf16")
    b = G.gmm_workspace_bytes(100_000_000, 128, 1024, "diag", "bf16")
    assert a == b > 0
    assert b < 10_000_000 * 1024 * 4 / 100      # < 1% of the N x K matrix at N = 10M


def test_plan_choices_for_large_k():
    """K > 1024 takes two passes; with the AUTO plan the EM step's normaliser
    pass runs without clusters while its N x slices normalisers fit in 4 GiB,
    in clusters of 8 beyond that or when CLUSTER is asked for; the statistics
    pass's tile groups keep the partials within 256 MiB."""
    small = G.gmm_plan_info(2_000_000, 96, 8192, "diag", "bf16")
    assert small["two_pass"] == 1 and small["cluster"] == 1
    big = G.gmm_plan_info(20_000_000, 96, 8192, "diag", "bf16")
    assert big["two_pass"] == 1 and big["cluster"] == 8
    forced = G.gmm_plan_info(2_000_000, 96, 8192, "diag", "bf16", plan="cluster")
    assert forced["cluster"] == 8
    for info, K, F in ((small, 8192, 257), (big, 8192, 257)):
        assert 1 <= info["tile_groups"] and info["tile_groups"] * K * F * 8 <= 256 << 20
    one = G.gmm_plan_info(10_000_000, 128, 1024, "diag", "bf16")
    assert one["two_pass"] == 0 and one["cluster"] == 8
