"""Seeded synthetic inputs for the GMM EM step (data X and starting parameters).

This module is shared by the CUDA path's tests and benchmark and by the
oracle's tests.  It draws random numbers and shapes them into the workloads
below; it contains none of the EM arithmetic.

Workloads (shapes and distributions after the method's own benchmark
descriptions; where a distribution was left open the choice is stated):

=====================  ===========  ====  =====  ==========  =====  ==========
name                   N            D     K      covariance  X      run
=====================  ===========  ====  =====  ==========  =====  ==========
tiny_diag              4,096        8     16     diag        f32    20 it + top-2
spherical_1m           1,000,000    64    256    spherical   f32    20 it
embed_10m              10,000,000   128   1024   diag        bf16   10 it + top-4
descriptor_100m        100,000,000  128   1024   diag        f32    5 it
largek_2m              2,000,000    96    8192   diag        bf16   10 it + top-8
=====================  ===========  ====  =====  ==========  =====  ==========

Data are generated in chunks of 2**20 rows; chunk ``c`` uses a generator
seeded ``seed * 1000003 + c + 1`` on the requested device, so any prefix of a
data set can be regenerated on its own.  The mixture that generates the data
(centres, spreads, weights) comes from ``numpy.random.default_rng(seed)``.
Starting parameters use a separate CPU generator seeded ``seed + 100``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

CHUNK = 1 << 20


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int
    D: int
    K: int
    cov: str          # "diag" | "spherical" | "tied"
    x_dtype: str      # "f32" | "bf16"
    iters: int
    topm: int         # 0: no top-m pass
    seed: int
    kind: str         # generator recipe, see _mixture / _post

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.x_dtype == "bf16" else torch.float32

    def scaled(self, N: int) -> "Workload":
        """The same recipe with fewer rows (a prefix of the full data set)."""
        return dataclasses.replace(self, N=int(N))


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_diag", 4096, 8, 16, "diag", "f32", 20, 2, 0, "tiny"),
        Workload("spherical_1m", 1_000_000, 64, 256, "spherical", "f32", 20, 0, 1,
                 "spherical"),
        Workload("embed_10m", 10_000_000, 128, 1024, "diag", "bf16", 10, 4, 2, "embed"),
        Workload("descriptor_100m", 100_000_000, 128, 1024, "diag", "f32", 5, 0, 3,
                 "descriptor"),
        Workload("largek_2m", 2_000_000, 96, 8192, "diag", "bf16", 10, 8, 4, "largek"),
    ]
}


def _mixture(w: Workload):
    """(centres C x D, spreads C x D, weights C) of the generating mixture."""
    rng = np.random.default_rng(w.seed)
    D = w.D
    if w.kind == "tiny":
        C = 16
        centres = rng.uniform(-10.0, 10.0, size=(C, D))
        spread = rng.uniform(0.5, 2.0, size=(C, D))
        weights = rng.dirichlet(np.ones(C))
    elif w.kind == "spherical":
        C = 256
        centres = rng.normal(0.0, 2.0, size=(C, D))            # N(0, 4 I)
        spread = np.repeat(rng.uniform(0.3, 1.5, size=(C, 1)), D, axis=1)
        weights = np.full(C, 1.0 / C)
    elif w.kind == "embed":
        C = 4096
        centres = rng.normal(0.0, 1.0, size=(C, D))
        spread = rng.uniform(0.05, 0.3, size=(C, D))
        weights = np.full(C, 1.0 / C)
    elif w.kind == "descriptor":
        C = 2048
        centres = rng.uniform(32.0, 224.0, size=(C, D))
        spread = rng.uniform(5.0, 30.0, size=(C, D))
        weights = np.full(C, 1.0 / C)
    elif w.kind == "largek":
        C = 8192
        centres = rng.normal(0.0, 1.0, size=(C, D))
        spread = rng.uniform(0.05, 0.3, size=(C, D))
        weights = rng.dirichlet(np.full(C, 0.5))
    elif w.kind == "generic":
        # Small parity cases: a well-mixed mixture with as many centres as
        # components, unit-scale spreads.
        C = max(w.K, 1)
        centres = rng.normal(0.0, 2.0, size=(C, D))
        spread = rng.uniform(0.5, 1.5, size=(C, D))
        weights = rng.dirichlet(np.ones(C))
    else:
        raise ValueError(w.kind)
    return centres, spread, weights


def _post(w: Workload, x: torch.Tensor) -> torch.Tensor:
    if w.kind == "embed":
        x = x / x.norm(dim=1, keepdim=True)
    elif w.kind == "descriptor":
        x = x.round().clamp_(0.0, 255.0)
    return x.to(w.torch_dtype)


def make_data(w: Workload, n_rows: int | None = None, device="cpu") -> torch.Tensor:
    """The first ``n_rows`` (default: all N) rows of workload ``w``'s data,
    as an (n_rows, D) tensor of ``w.torch_dtype`` on ``device``."""
    n = w.N if n_rows is None else int(n_rows)
    device = torch.device(device)
    centres, spread, weights = _mixture(w)
    c_t = torch.tensor(centres, dtype=torch.float32, device=device)
    s_t = torch.tensor(spread, dtype=torch.float32, device=device)
    p_t = torch.tensor(weights, dtype=torch.float64, device=device)
    out = torch.empty((n, w.D), dtype=w.torch_dtype, device=device)
    for c in range(math.ceil(n / CHUNK)):
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        rows = hi - lo
        g = torch.Generator(device=device)
        g.manual_seed(w.seed * 1000003 + c + 1)
        # Always draw a whole chunk so that a prefix equals the full data set's rows.
        lab = torch.multinomial(p_t, CHUNK, replacement=True, generator=g)[:rows]
        eps = torch.randn((CHUNK, w.D), generator=g, device=device,
                          dtype=torch.float32)[:rows]
        out[lo:hi] = _post(w, c_t[lab] + s_t[lab] * eps)
    return out


def _distinct_indices(N: int, K: int, g: torch.Generator) -> torch.Tensor:
    if N <= 4_000_000:
        return torch.randperm(N, generator=g)[:K]
    picked: list[int] = []
    seen: set[int] = set()
    while len(picked) < K:
        for v in torch.randint(0, N, (2 * K,), generator=g).tolist():
            if v not in seen:
                seen.add(v)
                picked.append(v)
                if len(picked) == K:
                    break
    return torch.tensor(picked, dtype=torch.int64)


def make_init(w: Workload, X: torch.Tensor):
    """Starting parameters (log_weights[K], means[K,D], vars[K], [K,D] or, for
    a tied model, the shared [D,D] covariance) as float32 numpy arrays: means
    are K distinct random data points; variances are 1 for the tiny workload,
    else the per-dimension variance of the data (over the first 2**20 rows;
    averaged over dimensions for a spherical model; the data's covariance
    matrix for a tied one); weights are uniform."""
    N, D, K = X.shape[0], w.D, w.K
    if N < K:
        raise ValueError(f"need at least K={K} rows to pick starting means, got {N}")
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed + 100)
    idx = _distinct_indices(N, K, g)
    means = X[idx.to(X.device)].float().cpu().numpy().astype(np.float32)
    if w.kind == "tiny":
        v = np.ones(D, np.float64)
        cm = np.eye(D)
    else:
        sample = X[: min(N, CHUNK)].double().cpu().numpy()
        v = sample.var(axis=0)
        cm = np.cov(sample.T, bias=True).reshape(D, D) if w.cov == "tied" else None
    if w.cov == "tied":
        vars_ = cm.astype(np.float32)
    elif w.cov == "spherical":
        vars_ = np.full(K, v.mean(), np.float32)
    else:
        vars_ = np.tile(v.astype(np.float32), (K, 1))
    log_weights = np.full(K, -math.log(K), np.float32)
    return log_weights, means, vars_.astype(np.float32)


def generic(N: int, D: int, K: int, cov: str = "diag", x_dtype: str = "f32",
            seed: int = 0) -> Workload:
    """A small parity-test workload of arbitrary shape (edge cases)."""
    return Workload(f"generic_{N}x{D}x{K}_{cov}_{x_dtype}", N, D, K, cov, x_dtype,
                    1, 0, seed, "generic")
