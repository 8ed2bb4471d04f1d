"""Python binding of the B300 GMM EM-step library (C ABI: include/gmm.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libgmm_b300.so``.  PyTorch supplies device memory and streams.
If the library is missing, every call raises; there is no fallback.

    import em_gmm_step_02_b300 as G
    lw, mu, var, ll = G.gmm_em_step(X, log_weights, means, vars_, "diag")
    r, idx, ll = G.gmm_predict_topm(X, log_weights, means, vars_, "diag", m=4)
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgmm_b300.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "gmm.h")

SPHERICAL, DIAG, TIED = 0, 1, 2
F32, BF16 = 0, 1
PREC = {"auto": 0, "fast": 1, "precise": 2}
PLAN = {"auto": 0, "cluster": 1, "split": 2}
REFINE = {"auto": 0, "on": 1, "off": 2}
COV = {"spherical": SPHERICAL, "diag": DIAG, "tied": TIED}
STATUS = {0: "GMM_OK", -1: "GMM_ERR_INVALID_ARG", -2: "GMM_ERR_UNSUPPORTED",
          -3: "GMM_ERR_NONFINITE", -4: "GMM_ERR_CUDA", -5: "GMM_ERR_TIMEOUT", -6: "GMM_ERR_RANGE",
          -7: "GMM_ERR_CAPACITY"}


class GmmError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS.get(code, code)}: {message}")
        self.code = code


class gmm_opts(ctypes.Structure):
    _fields_ = [("precision", ctypes.c_int32), ("reg_covar", ctypes.c_float),
                ("var_floor", ctypes.c_float), ("x_absmax", ctypes.c_float),
                ("loglik_on_host", ctypes.c_int32), ("plan", ctypes.c_int32),
                ("wait_limit", ctypes.c_int32), ("approx_top_k", ctypes.c_int32),
                ("topm_refine", ctypes.c_int32)]


_lib = None


def lib():
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run `python -m em_gmm_step_02_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        L.gmm_default_opts.argtypes = [ctypes.POINTER(gmm_opts)]
        L.gmm_default_opts.restype = None
        L.gmm_em_step.argtypes = [vp, i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp,
                                  ctypes.POINTER(gmm_opts), vp]
        L.gmm_em_step.restype = ctypes.c_int
        L.gmm_em_step_noalloc.argtypes = L.gmm_em_step.argtypes
        L.gmm_em_step_noalloc.restype = ctypes.c_int
        L.gmm_em_step_host.argtypes = [vp, i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, i64,
                                       ctypes.POINTER(gmm_opts), vp]
        L.gmm_em_step_host.restype = ctypes.c_int
        L.gmm_assign_threshold.argtypes = [vp, i64, i32, i32, i32, i32, vp, vp, vp, ctypes.c_float, i32,
                                           vp, vp, vp, i64, ctypes.POINTER(gmm_opts), vp]
        L.gmm_assign_threshold.restype = ctypes.c_int
        L.gmm_predict_topm.argtypes = [vp, i64, i32, i32, i32, i32, vp, vp, vp, i32, vp, vp, vp,
                                       ctypes.POINTER(gmm_opts), vp]
        L.gmm_predict_topm.restype = ctypes.c_int
        L.gmm_workspace_bytes.argtypes = [i64, i32, i32, i32, i32, ctypes.POINTER(gmm_opts)]
        L.gmm_workspace_bytes.restype = ctypes.c_size_t
        L.gmm_reserve.argtypes = [i64, i32, i32, i32, i32, ctypes.POINTER(gmm_opts)]
        L.gmm_reserve.restype = ctypes.c_int
        L.gmm_stream_status.argtypes = [vp]
        L.gmm_stream_status.restype = ctypes.c_int
        L.gmm_last_error.argtypes = []
        L.gmm_last_error.restype = ctypes.c_char_p
        L.gmm_release.argtypes = []
        L.gmm_release.restype = None
        L.gmm_plan_info.argtypes = [i64, i32, i32, i32, i32, ctypes.POINTER(gmm_opts), ctypes.POINTER(ctypes.c_int32)]
        L.gmm_plan_info.restype = ctypes.c_int
        L.gmm_last_launch_count.argtypes = []
        L.gmm_last_launch_count.restype = ctypes.c_int32
        L.gmm_profile_begin.argtypes = []
        L.gmm_profile_begin.restype = None
        L.gmm_profile_end.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int32)]
        L.gmm_profile_end.restype = ctypes.c_int
        L.gmm_selftest_mma.argtypes = [ctypes.c_int, vp, vp, vp, vp, vp]
        L.gmm_selftest_mma.restype = ctypes.c_int
        _lib = L
    return _lib


def declared_symbols() -> list[str]:
    """Function names declared in include/gmm.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(gmm_[a-z_]+)\s*\(", text)))


def gmm_last_error() -> str:
    return lib().gmm_last_error().decode()


def gmm_last_launch_count() -> int:
    return int(lib().gmm_last_launch_count())


def gmm_default_opts(**kw) -> gmm_opts:
    o = gmm_opts()
    lib().gmm_default_opts(ctypes.byref(o))
    for k, v in kw.items():
        if k == "precision" and isinstance(v, str):
            v = PREC[v]
        if k == "plan" and isinstance(v, str):
            v = PLAN[v]
        if k == "topm_refine" and isinstance(v, str):
            v = REFINE[v]
        setattr(o, k, v)
    return o


def _check(rc: int):
    if rc != 0:
        raise GmmError(rc, gmm_last_error())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _shape(X, means, cov):
    if X.dim() != 2:
        raise ValueError("X must be (N, D)")
    if X.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("X must be float32 or bfloat16")
    N, D = X.shape
    K = means.shape[0]
    cov_i = COV[cov] if isinstance(cov, str) else int(cov)
    return N, D, K, cov_i, (BF16 if X.dtype == torch.bfloat16 else F32)


def gmm_em_step(X, log_weights, means, vars_, cov="diag", *, out=None, opts: gmm_opts | None = None,
                stream=None, **opt_kw):
    """One EM step.  Returns (new_log_weights, new_means, new_vars, total_loglik);
    total_loglik is a 1-element float64 CUDA tensor (evaluated at the input
    parameters).  ``out`` may name the three output tensors (they may be the
    inputs themselves)."""
    N, D, K, cov_i, dt = _shape(X, means, cov)
    if opts is None:
        opts = gmm_default_opts(**opt_kw)
    if out is None:
        out = (torch.empty_like(log_weights), torch.empty_like(means), torch.empty_like(vars_))
    ll = torch.empty(1, dtype=torch.float64, device=X.device)
    opts.loglik_on_host = 0
    rc = lib().gmm_em_step(_dev(X, "X"), N, D, K, cov_i, dt,
                           _dev(log_weights, "log_weights", torch.float32),
                           _dev(means, "means", torch.float32), _dev(vars_, "vars", torch.float32),
                           _dev(out[0], "new_log_weights", torch.float32),
                           _dev(out[1], "new_means", torch.float32),
                           _dev(out[2], "new_vars", torch.float32),
                           _dev(ll, "total_loglik", torch.float64), ctypes.byref(opts), _stream(stream))
    _check(rc)
    return out[0], out[1], out[2], ll


def gmm_assign_threshold(X, log_weights, means, vars_, cov="diag", *, tau, max_per_point=16,
                         capacity=None, opts: gmm_opts | None = None, stream=None, **opt_kw):
    """Threshold multi-assignment as compressed rows (see include/gmm.h):
    returns (offsets (N+1) int64, idx int32, resp float32), CUDA tensors;
    point i's entries are idx/resp[offsets[i]:offsets[i+1]].  With
    ``capacity`` None the output is sized for the worst case
    (N * max_per_point entries) and trimmed to the total."""
    N, D, K, cov_i, dt = _shape(X, means, cov)
    if opts is None:
        opts = gmm_default_opts(**opt_kw)
    cap = N * max_per_point if capacity is None else int(capacity)
    offsets = torch.empty(N + 1, dtype=torch.int64, device=X.device)
    idx = torch.empty(max(cap, 1), dtype=torch.int32, device=X.device)
    resp = torch.empty(max(cap, 1), dtype=torch.float32, device=X.device)
    opts.loglik_on_host = 0
    rc = lib().gmm_assign_threshold(_dev(X, "X"), N, D, K, cov_i, dt,
                                    _dev(log_weights, "log_weights", torch.float32),
                                    _dev(means, "means", torch.float32), _dev(vars_, "vars", torch.float32),
                                    ctypes.c_float(tau), int(max_per_point), _dev(offsets, "offsets"),
                                    _dev(idx, "idx_out"), _dev(resp, "resp_out"), cap, ctypes.byref(opts),
                                    _stream(stream))
    _check(rc)
    if capacity is None:
        total = int(offsets[N].item())
        return offsets, idx[:total], resp[:total]
    return offsets, idx, resp


def gmm_em_step_host(X_host, log_weights, means, vars_, cov="diag", *, chunk_rows=0, out=None,
                     opts: gmm_opts | None = None, stream=None, **opt_kw):
    """One EM step over X held in host memory (see gmm_em_step_host in
    include/gmm.h): the library copies X to the GPU in chunks of
    ``chunk_rows`` rows (0: its default) while the previous chunk is being
    processed.  X_host is a contiguous CPU tensor, best page-locked
    (``pin_memory()``) so that the copies overlap the kernels; ``x_absmax``
    (a bound on max |X|) must be given.  Parameters and outputs are CUDA
    tensors, as for gmm_em_step."""
    if not isinstance(X_host, torch.Tensor) or X_host.is_cuda:
        raise TypeError("X_host must be a CPU tensor")
    if not X_host.is_contiguous():
        raise ValueError("X_host must be contiguous")
    N, D, K, cov_i, dt = _shape(X_host, means, cov)
    if opts is None:
        opts = gmm_default_opts(**opt_kw)
    if out is None:
        out = (torch.empty_like(log_weights), torch.empty_like(means), torch.empty_like(vars_))
    ll = torch.empty(1, dtype=torch.float64, device=means.device)
    opts.loglik_on_host = 0
    rc = lib().gmm_em_step_host(ctypes.c_void_p(X_host.data_ptr()), N, D, K, cov_i, dt,
                                _dev(log_weights, "log_weights", torch.float32),
                                _dev(means, "means", torch.float32), _dev(vars_, "vars", torch.float32),
                                _dev(out[0], "new_log_weights", torch.float32),
                                _dev(out[1], "new_means", torch.float32),
                                _dev(out[2], "new_vars", torch.float32),
                                _dev(ll, "total_loglik", torch.float64), int(chunk_rows), ctypes.byref(opts),
                                _stream(stream))
    _check(rc)
    return out[0], out[1], out[2], ll


def gmm_em_step_noalloc(X, log_weights, means, vars_, cov="diag", *, out, opts: gmm_opts | None = None,
                        stream=None, **opt_kw):
    """The EM step without any device allocation inside the library (see
    gmm_em_step_noalloc in include/gmm.h).  ``out`` = (new_log_weights,
    new_means, new_vars, total_loglik) must be given: the caller provides all
    memory.  Returns ``out``."""
    N, D, K, cov_i, dt = _shape(X, means, cov)
    if opts is None:
        opts = gmm_default_opts(**opt_kw)
    opts.loglik_on_host = 0
    rc = lib().gmm_em_step_noalloc(_dev(X, "X"), N, D, K, cov_i, dt,
                                   _dev(log_weights, "log_weights", torch.float32),
                                   _dev(means, "means", torch.float32), _dev(vars_, "vars", torch.float32),
                                   _dev(out[0], "new_log_weights", torch.float32),
                                   _dev(out[1], "new_means", torch.float32),
                                   _dev(out[2], "new_vars", torch.float32),
                                   _dev(out[3], "total_loglik", torch.float64), ctypes.byref(opts),
                                   _stream(stream))
    _check(rc)
    return out


def gmm_predict_topm(X, log_weights, means, vars_, cov="diag", m=1, *, opts: gmm_opts | None = None,
                     stream=None, **opt_kw):
    """Top-m responsibilities (N, m) float32 and indices (N, m) int32, plus the
    total log-likelihood (1-element float64 CUDA tensor).  Keywords set
    gmm_opts fields by name, e.g. precision="fast" | "precise",
    topm_refine="auto" | "on" | "off" (the direct-form refinement of the
    candidates; AUTO refines PRECISE only)."""
    N, D, K, cov_i, dt = _shape(X, means, cov)
    if opts is None:
        opts = gmm_default_opts(**opt_kw)
    r = torch.empty((N, m), dtype=torch.float32, device=X.device)
    idx = torch.empty((N, m), dtype=torch.int32, device=X.device)
    ll = torch.empty(1, dtype=torch.float64, device=X.device)
    opts.loglik_on_host = 0
    rc = lib().gmm_predict_topm(_dev(X, "X"), N, D, K, cov_i, dt,
                                _dev(log_weights, "log_weights", torch.float32),
                                _dev(means, "means", torch.float32), _dev(vars_, "vars", torch.float32),
                                int(m), _dev(r, "resp_out"), _dev(idx, "idx_out"), _dev(ll, "total_loglik"),
                                ctypes.byref(opts), _stream(stream))
    _check(rc)
    return r, idx, ll


def gmm_workspace_bytes(N, D, K, cov="diag", x_dtype="bf16", **opt_kw) -> int:
    cov_i = COV[cov] if isinstance(cov, str) else int(cov)
    dt = BF16 if x_dtype in ("bf16", BF16) else F32
    o = gmm_default_opts(**opt_kw)
    return int(lib().gmm_workspace_bytes(int(N), int(D), int(K), cov_i, dt, ctypes.byref(o)))


def gmm_reserve(N, D, K, cov="diag", x_dtype="bf16", **opt_kw):
    cov_i = COV[cov] if isinstance(cov, str) else int(cov)
    dt = BF16 if x_dtype in ("bf16", BF16) else F32
    o = gmm_default_opts(**opt_kw)
    _check(lib().gmm_reserve(int(N), int(D), int(K), cov_i, dt, ctypes.byref(o)))


def gmm_plan_info(N, D, K, cov="diag", x_dtype="bf16", **opt_kw) -> dict:
    """The launch plan of an EM step with these arguments on the current device
    (see gmm_plan_info in include/gmm.h)."""
    cov_i = COV[cov] if isinstance(cov, str) else int(cov)
    dt = BF16 if x_dtype in ("bf16", BF16) else F32
    o = gmm_default_opts(**opt_kw)
    info = (ctypes.c_int32 * 8)()
    _check(lib().gmm_plan_info(int(N), int(D), int(K), cov_i, dt, ctypes.byref(o), info))
    keys = ("cluster", "tile_groups", "two_pass", "tile_groups_pass1", "flush_tiles", "threads",
            "noalloc_tile_groups", "tiles")
    return dict(zip(keys, [int(v) for v in info]))


def gmm_stream_status(stream=None) -> int:
    return int(lib().gmm_stream_status(_stream(stream)))


def gmm_profile_begin():
    lib().gmm_profile_begin()


def gmm_profile_end():
    """(summed device milliseconds of the main kernel launches, their count)."""
    ms = ctypes.c_double(0.0)
    n = ctypes.c_int32(0)
    _check(lib().gmm_profile_end(ctypes.byref(ms), ctypes.byref(n)))
    return float(ms.value), int(n.value)


def gmm_release():
    lib().gmm_release()


def gmm_selftest_mma(variant: int, a_img: torch.Tensor, b_img: torch.Tensor, d_out: torch.Tensor,
                     status: torch.Tensor, stream=None):
    """Diagnostic: one tensor-core contraction on ready-made operand images."""
    _check(lib().gmm_selftest_mma(int(variant), _dev(a_img, "a_img"), _dev(b_img, "b_img"),
                                  _dev(d_out, "d_out"), _dev(status, "status"), _stream(stream)))
