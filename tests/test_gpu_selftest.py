"""Tensor-core building blocks: one tcgen05 contraction on operand images laid
out exactly as the EM kernels lay out theirs (128-byte swizzle, K-major and
MN-major), read back through tensor memory.  Inputs are small integers so
the fp32 result is exact and the comparison is bit-exact."""
import numpy as np
import pytest
import torch

import em_gmm_step_02_b300 as G
from gpu_util import kmajor_image, mnmajor_image


def _as_u16(x: np.ndarray, bf16: bool) -> np.ndarray:
    t = torch.tensor(x, dtype=torch.float32)
    t = t.to(torch.bfloat16 if bf16 else torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.gpu
@pytest.mark.parametrize("variant", [0, 1, 2, 3])
def test_mma_layouts(variant):
    rng = np.random.default_rng(variant)
    mn = variant & 1
    bf16 = bool(variant & 2)
    if not mn:
        A = rng.integers(-4, 5, size=(128, 64)).astype(np.float32) / 4
        B = rng.integers(-4, 5, size=(128, 64)).astype(np.float32) / 4
        ref = A @ B.T
        a_img, b_img = kmajor_image(_as_u16(A, bf16)), kmajor_image(_as_u16(B, bf16))
        N = 128
    else:
        A = rng.integers(-4, 5, size=(64, 128)).astype(np.float32) / 4   # K x M
        B = rng.integers(-4, 5, size=(64, 256)).astype(np.float32) / 4   # K x N
        ref = A.T @ B
        a_img, b_img = mnmajor_image(_as_u16(A, bf16)), mnmajor_image(_as_u16(B, bf16))
        N = 256
    a = torch.tensor(a_img, device="cuda")
    b = torch.tensor(b_img, device="cuda")
    d = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.gmm_selftest_mma(variant, a, b, d, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(d.cpu().numpy(), ref.astype(np.float32))


def const_image(M: np.ndarray) -> np.ndarray:
    """128 x 16 matrix (uint16) -> the unswizzled K-major image of the logit
    constant step: 8-row x 16-byte core matrices, K neighbours 128 bytes
    apart, row groups 256 bytes apart."""
    rows, cols = M.shape
    assert rows == 128 and cols == 16
    img = np.zeros(rows * cols * 2, np.uint8)
    r, k = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    off = (r // 8) * 256 + (k // 8) * 128 + (r % 8) * 16 + (k % 8) * 2
    v = M.astype(np.uint16)
    img[off] = (v & 0xFF).astype(np.uint8)
    img[off + 1] = (v >> 8).astype(np.uint8)
    return img


@pytest.mark.gpu
def test_constant_step_layout_and_minus_inf():
    """The unswizzled operand layout of the logit constant step, and a -inf
    parameter entry giving a -inf logit (padded and dead components)."""
    rng = np.random.default_rng(4)
    A = rng.integers(-4, 5, size=(128, 16)).astype(np.float32) / 4
    A[:, 0] = 2.0 ** 15                   # the constant step's data side is nonzero in column 0
    B = rng.integers(-4, 5, size=(128, 16)).astype(np.float32) / 4
    B[5, 0] = -np.inf
    B[77, 0] = -np.inf
    with np.errstate(invalid="ignore"):
        ref = A @ B.T
    a = torch.tensor(const_image(_as_u16(A, False)), device="cuda")
    b = torch.tensor(const_image(_as_u16(B, False)), device="cuda")
    d = torch.full((128, 128), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.gmm_selftest_mma(4, a, b, d, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = d.cpu().numpy()
    assert np.isneginf(got[:, 5]).all() and np.isneginf(got[:, 77]).all()
    np.testing.assert_array_equal(got, ref.astype(np.float32))
