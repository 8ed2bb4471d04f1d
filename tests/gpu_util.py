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
