"""The MLP block on the cube: Y = GELU(X W1 + b1) W2 + b2 (oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

TT11 "Tensor parallelism": the first FFN matrix is split by columns, each
part applies GELU locally, the second matrix is split by rows and the
partial outputs are summed.  MP3D §3.2: the MLP block is two 3-D linears;
the first takes input group y = 0 (X in CUBE_A, W1 in CUBE_B, Y1 out in
CUBE_C), the second runs with y and z exchanged (Y1 as input, W2 in the
swapped weight layout, Y back in CUBE_A).  All of it reaches exactly the
unsplit MLP, which is what the oracle computes, in float64, with no rounding
of the hidden activation.

Parity status: pinned up to the definition of GELU.  The tests check the
Megatron identity (sum over t column/row splits equals the unsplit MLP), the
cube identity (two sharded ``linear3d`` calls equal it), GELU(0) = 0 and
GELU(x) -> x for large x.
"""
from __future__ import annotations

import numpy as np

from .layouts import CUBE_A, CUBE_B, CUBE_B_SWAP, CUBE_C, from_sharded, to_sharded
from .linear import gelu


def mlp_dense(X, W1, b1, W2, b2):
    """Returns (Y, Z1, Y1) as float64 global matrices."""
    Z1 = np.asarray(X, np.float64) @ np.asarray(W1, np.float64) + np.asarray(b1, np.float64)[None, :]
    Y1 = gelu(Z1)
    Y = Y1 @ np.asarray(W2, np.float64) + np.asarray(b2, np.float64)[None, :]
    return Y, Z1, Y1


def mlp3d(X_buf, W1_buf, b1, W2_buf, b2, p, M, h, f):
    """Sharded MLP: X (M x h) CUBE_A, W1 (h x f) CUBE_B, W2 (f x h)
    CUBE_B_SWAP.  Returns (Y in CUBE_A, Y1 in CUBE_C), float64."""
    X = from_sharded(np.asarray(X_buf, np.float64), CUBE_A(p), M, h)
    W1 = from_sharded(np.asarray(W1_buf, np.float64), CUBE_B(p), h, f)
    W2 = from_sharded(np.asarray(W2_buf, np.float64), CUBE_B_SWAP(p), f, h)
    Y, _, Y1 = mlp_dense(X, W1, b1, W2, b2)
    return to_sharded(Y, CUBE_A(p)), to_sharded(Y1, CUBE_C(p))


def mlp_rows_dense(X_rows, W1, b1, W2, b2):
    """The MLP on a subset of rows (it is row-separable); used for sampled
    parity at sizes where the full oracle is too slow."""
    return mlp_dense(X_rows, W1, b1, W2, b2)[0]
