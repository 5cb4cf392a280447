"""The 3-D linear C = A.B (+ b) (GELU), forward and backward (oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

MP3D Algorithm 1 (all-gather A_il in y, all-gather B_lj in x, multiply,
reduce-scatter in z) reaches exactly the dense product C = A.B: device
(i, j, l) ends with rows l*m .. l*m+m-1 of C_ij = sum_l A_il B_lj, which is a
block of the dense product (MP3D §2.3 worked 2x2x2 formula and §3.1.1).  The
oracle is therefore that definition: gather every shard through the layout
maps, one float64 matrix product (a library primitive), bias, GELU, scatter.

Bias (MP3D Algorithm 7, C + b): the output block with column block j adds
b_j, the slice of the diagonally stored vector gathered over x; in global
terms every column c adds b[c].

Backward (MP3D §3.1.2 differentiation formulas, Algorithm 2): dA = dC B^T,
dB = A^T dC.  Bias gradient (Algorithm 8): the printed algorithm sums the
local rows and keeps the result only where j = l; read plainly the gradient
of b[c] is the sum of dC[:, c] over all M rows (the definition), which is
what the oracle returns.

Parity status: pinned.  ``tests/test_oracle_linear.py`` checks, on integer
data (exact in float64), that a literal device-by-device emulation of
Algorithm 1 and of the unbalanced 2-D broadcast form of MP3D §2.3 equal this
oracle bit for bit, that the forward product equals a textbook triple loop
on tiny inputs, and the backward against central finite differences.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

from .layouts import CUBE_A, CUBE_B, CUBE_C, CUBE_B_SWAP, Cube, from_sharded, to_sharded


def gelu(x: np.ndarray) -> np.ndarray:
    """Exact GELU, x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)).  The pages name
    GELU only (TT11 "Tensor parallelism"); erf is its definition."""
    return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))


def gelu_grad(x: np.ndarray) -> np.ndarray:
    """d/dx [x Phi(x)] = Phi(x) + x phi(x)."""
    cdf = 0.5 * (1.0 + erf(x / math.sqrt(2.0)))
    pdf = np.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)
    return cdf + x * pdf


def linear_layouts(p: int, y: int):
    """(A, B, C) layouts for input group index y (MP3D §3.2): y = 0 is the
    first linear of a block (A in direction y, C in z); y = 1 has y and z
    exchanged, so the output comes back in the input direction."""
    if y == 0:
        return CUBE_A(p), CUBE_B(p), CUBE_C(p)
    return Cube("A", p, swap=True), CUBE_B_SWAP(p), Cube("C", p, swap=True)


def linear3d_dense(A: np.ndarray, B: np.ndarray, bias=None, act: str | None = None):
    """C = A.B (+ b) (GELU) on global float64 matrices."""
    C = np.asarray(A, dtype=np.float64) @ np.asarray(B, dtype=np.float64)
    if bias is not None:
        C = C + np.asarray(bias, dtype=np.float64)[None, :]
    if act == "gelu":
        C = gelu(C)
    return C


def linear3d(A_buf, B_buf, p, M, N, K, bias=None, act=None, y=0):
    """MP3D Algorithm 1 (+ Algorithm 7): sharded A (M x N), B (N x K) in, the
    sharded output C (M x K) out, all float64."""
    la, lb, lc = linear_layouts(p, y)
    A = from_sharded(np.asarray(A_buf, dtype=np.float64), la, M, N)
    B = from_sharded(np.asarray(B_buf, dtype=np.float64), lb, N, K)
    return to_sharded(linear3d_dense(A, B, bias, act), lc)


def linear3d_backward_dense(dC, A, B):
    """MP3D §3.1.2 for C = A.B + b: dA = dC B^T, dB = A^T dC, db = column
    sums of dC over all rows."""
    dC = np.asarray(dC, dtype=np.float64)
    return dC @ np.asarray(B, np.float64).T, np.asarray(A, np.float64).T @ dC, dC.sum(axis=0)


def linear3d_backward(dC_buf, A_buf, B_buf, p, M, N, K, y=0):
    """MP3D Algorithm 2 (and Algorithm 8 for the bias): dA in A's layout, dB
    in B's layout, db as a plain vector."""
    la, lb, lc = linear_layouts(p, y)
    A = from_sharded(np.asarray(A_buf, np.float64), la, M, N)
    B = from_sharded(np.asarray(B_buf, np.float64), lb, N, K)
    dC = from_sharded(np.asarray(dC_buf, np.float64), lc, M, K)
    dA, dB, db = linear3d_backward_dense(dC, A, B)
    return to_sharded(dA, la), to_sharded(dB, lb), db
