"""Helpers shared by the GPU tests: operand images, error metrics, runners."""
from __future__ import annotations

import numpy as np
import torch


def sw128_off(r: np.ndarray, c16: np.ndarray) -> np.ndarray:
    """Byte offset of 16-byte chunk c16 of row r inside one 128-byte-swizzled atom column."""
    return (r // 8) * 1024 + (r % 8) * 128 + ((c16 ^ (r % 8)) << 4)


def kmajor_image(M: np.ndarray) -> np.ndarray:
    """Rows x 64 matrix (16-bit values as uint16) -> K-major swizzled image bytes."""
    rows, cols = M.shape
    assert cols == 64
    img = np.zeros(rows * 128, np.uint8)
    r, c = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    off = sw128_off(r, c // 8) + (c % 8) * 2
    v = M.astype(np.uint16)
    img[off] = (v & 0xFF).astype(np.uint8)
    img[off + 1] = (v >> 8).astype(np.uint8)
    return img


def mnmajor_image(M: np.ndarray) -> np.ndarray:
    """K x MN matrix (uint16) -> MN-major swizzled image: MN split in 64-wide atom
    columns of K*128 bytes each."""
    k, mn = M.shape
    img = np.zeros(k * mn * 2, np.uint8)
    r, c = np.meshgrid(np.arange(k), np.arange(mn), indexing="ij")
    off = (c // 64) * (k * 128) + sw128_off(r, (c % 64) // 8) + (c % 8) * 2
    v = M.astype(np.uint16)
    img[off] = (v & 0xFF).astype(np.uint8)
    img[off + 1] = (v >> 8).astype(np.uint8)
    return img


def rel_l2_rows(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per-row relative L2 error ||got - ref|| / ||ref|| (rows = components)."""
    got = np.atleast_2d(np.asarray(got, np.float64).T).T
    ref = np.atleast_2d(np.asarray(ref, np.float64).T).T
    if got.ndim == 1:
        got, ref = got[:, None], ref[:, None]
    num = np.linalg.norm(got - ref, axis=1)
    den = np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    return num / den


def params_to_device(lw, mu, var, device="cuda"):
    return (torch.tensor(np.asarray(lw, np.float32), device=device),
            torch.tensor(np.asarray(mu, np.float32), device=device),
            torch.tensor(np.asarray(var, np.float32), device=device))


# ------------------------------------------------------------------ element-wise parity
# Relative error is taken element by element.  Each quantity gets the floor of
# its denominator from the scale on which the arithmetic resolves it:
#   weights    relative to pi_k (a dead component, pi = 0, must stay 0);
#   means      relative to max(|mu_kd|, sigma_kd): a coordinate is compared on
#              the larger of its own size and the component's spread in that
#              dimension (a mean coordinate near zero has no relative digits,
#              and EM moves means in units of sigma);
#   variances  relative to s2_kd, or within four units of EPS[arithmetic] of
#              the second moment in the arithmetic's own frame,
#              m2_kd = s2_kd + (mu_kd - shift_d)^2, because the one-pass
#              M-step forms s2 = m2 - (mu - shift)^2 from sums of
#              ((x - shift) scale)^2 that carry EPS relative precision (FAST:
#              fp16 products, one rounding for bf16 data, two for float32 data
#              whose x' is rounded too; PRECISE: fp32 accumulation of a flush
#              period, 2048 points per CTA: about 2^-24 sqrt(2048)).  The shift
#              is the mean of the input component means (float32 data, or
#              PRECISE), else zero.
# Components with fewer than MIN_NK effective points: a variance estimated
# from so few points is fixed by a handful of responsibilities, each of which
# carries the E-step's logit rounding (FAST: about 2^-12 times the size of the
# expanded form's terms) to first order, and it has a sampling error of
# sqrt(2 / N_k) > 35%: no stable relative digits.  For these, PRECISE compares
# m2 within 3 tol m2 (what the mean and variance bounds imply for
# m2 = s2 + (mu - shift)^2: |d s2| + 2 |mu - shift| |d mu| <= 3 tol m2);
# FAST compares their weights and means only (the E-step itself is compared
# directly, point by point, by the top-m tests).
EPS = {"fast_bf16": 2.0 ** -12, "fast_f32": 2.0 ** -11, "precise": 2.0 ** -18}
MIN_NK = 16.0


def elementwise_errors(got, ref, N, cov, path, tol, x_dtype="bf16", means_in=None):
    """(weights, means, variances) error maxima of one EM step on N points,
    each already divided by its allowed bound (pass: <= 1), plus a
    description.  x_dtype is the data's storage type ("bf16" or "f32");
    means_in are the step's input means (for the arithmetic's shift)."""
    lw_g, mu_g, var_g = [np.asarray(a, np.float64) for a in got[:3]]
    lw_r, mu_r, var_r = [np.asarray(a, np.float64) for a in ref[:3]]
    K, D = mu_r.shape
    fast_bf16 = path == "fast" and x_dtype == "bf16"
    eps = EPS["precise"] if path == "precise" else EPS["fast_bf16" if fast_bf16 else "fast_f32"]
    shift = np.zeros(D) if (fast_bf16 or means_in is None) else np.asarray(means_in, np.float64).mean(0)
    w_g, w_r = np.exp(lw_g), np.exp(lw_r)
    e_w = np.abs(w_g - w_r) / np.maximum(w_r, 1e-6 * w_r.max()) / tol
    v_r = var_r.reshape(K, -1)
    v_g = var_g.reshape(K, -1)
    sig = np.sqrt(np.broadcast_to(v_r, (K, D)))
    e_mu = np.abs(mu_g - mu_r) / np.maximum(np.abs(mu_r), sig) / tol
    sq = (lambda m: m ** 2) if v_r.shape[1] == D else (lambda m: (m ** 2).mean(1, keepdims=True))
    m2_r = v_r + sq(mu_r - shift)
    nk = w_r * N                       # effective points of each component
    big = np.broadcast_to((nk >= MIN_NK)[:, None], v_r.shape)
    bound = np.maximum(tol * v_r, 4.0 * eps * m2_r)
    e_v = np.where(big, np.abs(v_g - v_r) / bound, 0.0)
    if path == "precise":
        e_small = np.where(big, 0.0, np.abs(v_g - v_r) / (3.0 * tol * m2_r))
    else:
        e_small = np.zeros_like(e_v)
    worst = np.unravel_index(np.argmax(e_v), e_v.shape)
    msg = (f"w {e_w.max() * tol:.2e} mu {e_mu.max() * tol:.2e} "
           f"var {e_v.max():.2e}x bound over {int(big[:, 0].sum())}/{K} comps with N_k >= {MIN_NK:g} "
           f"(worst k={worst[0]}: ref {v_r[worst]:.3e} got {v_g[worst]:.3e} m2 {m2_r[worst]:.3e}); "
           f"small comps var {e_small.max():.2e}x bound")
    return e_w.max(), e_mu.max(), max(e_v.max(), e_small.max()), msg


# ------------------------------------------------------------------ top-m bounds of PRECISE
def precise_resp_tol(X, means, vars_, cov, idx, r, tol, tol_ll):
    """Per-entry bound (N x m) on a PRECISE responsibility, the larger of tol
    and 2 eps T min(r, 1 - r), and the bound on the per-point mean
    log-likelihood, the larger of tol_ll and the mean of eps T (a row's
    log-sum-exp moves by at most its largest logit error).  PRECISE resolves a
    logit to about eps (natural-log units) of the size T of its expanded-form
    terms: eps = (2^-22 + 2^-24 sqrt(n)) ln 2, the 22-bit operand pieces plus
    the fp32 accumulation over the n = 3 * 2 D_pad / 16 MMA K steps of the
    three products (rounding errors of a random walk),
        T = sum_d ((x - s)^2 + 2 |x - s| |mu - s| + (mu - s)^2) / (2 s2)  (log2 units),
    s the mean of the component means; T is taken as the largest over the
    point's listed components.  A responsibility moves by
    r_k (dl_k - sum_j r_j dl_j), at most 2 eps T r_k, and the largest one
    by at most 2 eps T (1 - r_k) since the responsibilities sum to one."""
    X = np.asarray(X, np.float64)
    mu = np.asarray(means, np.float64)
    K, D = mu.shape
    v = np.asarray(vars_, np.float64)
    v = np.repeat(v.reshape(K, 1), D, 1) if cov == "spherical" else v.reshape(K, D)
    s = mu.mean(0)
    y = X - s
    ay = np.abs(y)
    T = np.zeros(X.shape[0])
    for j in range(idx.shape[1]):
        k = np.asarray(idx[:, j])
        nu = mu[k] - s
        t = ((y * y + 2 * ay * np.abs(nu) + nu * nu) / (2 * v[k])).sum(1) * np.log2(np.e)
        T = np.maximum(T, t)
    d_pad = 64 * ((D + 63) // 64)
    eps = (2.0 ** -22 + 2.0 ** -24 * np.sqrt(3 * 2 * d_pad / 16)) * np.log(2.0)
    r = np.asarray(r, np.float64)
    return np.maximum(tol, 2 * eps * T[:, None] * np.minimum(r, 1 - r)), max(tol_ll, float((eps * T).mean()))
