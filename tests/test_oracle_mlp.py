"""Pins of the oracle's MLP, CPU only.

"Transformer Training 11: Model Parallelism", section "Tensor parallelism":
the first FFN matrix split by columns with GELU applied per part, the second
split by rows, and the partial outputs summed, equals the unsplit MLP.
"Maximizing Parallelism ..." §3.2: the MLP block is two 3-D linears, the
second with directions exchanged; composed, they equal the same MLP.
"""
import numpy as np
import pytest

from oracle import layouts as L
from oracle import linear as OL
from oracle import mlp as OM


def _inputs(rng, M, h, f):
    return (rng.standard_normal((M, h)), 0.3 * rng.standard_normal((h, f)), 0.1 * rng.standard_normal(f),
            0.3 * rng.standard_normal((f, h)), 0.1 * rng.standard_normal(h))


@pytest.mark.parametrize("t", [2, 4])
def test_megatron_split_identity(t):
    rng = np.random.default_rng(t)
    M, h, f = 16, 8, 32
    X, W1, b1, W2, b2 = _inputs(rng, M, h, f)
    w = f // t
    Y = sum(OL.gelu(X @ W1[:, s * w:(s + 1) * w] + b1[s * w:(s + 1) * w]) @ W2[s * w:(s + 1) * w, :]
            for s in range(t)) + b2
    want = OM.mlp_dense(X, W1, b1, W2, b2)[0]
    assert np.max(np.abs(Y - want)) <= 1e-12 * np.max(np.abs(want))


@pytest.mark.parametrize("p,M,h,f", [(2, 16, 8, 32), (3, 18, 9, 27)])
def test_cube_mlp_equals_two_cube_linears(p, M, h, f):
    rng = np.random.default_rng(p)
    X, W1, b1, W2, b2 = _inputs(rng, M, h, f)
    Xb = L.to_sharded(X, L.CUBE_A(p))
    W1b = L.to_sharded(W1, L.CUBE_B(p))
    W2b = L.to_sharded(W2, L.CUBE_B_SWAP(p))
    Y1b = OL.linear3d(Xb, W1b, p, M, h, f, bias=b1, act="gelu", y=0)
    Yb = OL.linear3d(Y1b, W2b, p, M, f, h, bias=b2, y=1)
    Ym, Y1m = OM.mlp3d(Xb, W1b, b1, W2b, b2, p, M, h, f)
    assert np.max(np.abs(Yb - Ym)) <= 1e-12 * np.max(np.abs(Ym))
    assert np.max(np.abs(Y1b - Y1m)) <= 1e-12 * np.max(np.abs(Y1m))
    # the output is back in the input's direction (CUBE_A) and equals the dense MLP
    want = OM.mlp_dense(X, W1, b1, W2, b2)[0]
    assert np.allclose(L.from_sharded(Ym, L.CUBE_A(p), M, h), want, rtol=1e-12, atol=1e-12)


def test_mlp_is_row_separable():
    # the sampled-row parity of large MLPs relies on it: any subset of rows
    # through the MLP equals the same rows of the full output (up to the
    # summation order a matrix library picks for a different height)
    rng = np.random.default_rng(11)
    X, W1, b1, W2, b2 = _inputs(rng, 24, 8, 32)
    rows = np.array([0, 5, 6, 17, 23])
    full = OM.mlp_dense(X, W1, b1, W2, b2)[0]
    got = OM.mlp_rows_dense(X[rows], W1, b1, W2, b2)
    assert np.max(np.abs(got - full[rows])) <= 1e-13 * np.max(np.abs(full))


def test_mlp_bias_paths():
    # W2 = 0: every output row is b2; W1 = 0 and b1 = 0: the hidden
    # activation is GELU(0) = 0, so again every row is b2; b1 alone reaches
    # the output as GELU(b1) W2 + b2 in every row
    rng = np.random.default_rng(12)
    X, W1, b1, W2, b2 = _inputs(rng, 6, 8, 16)
    Y = OM.mlp_dense(X, W1, b1, np.zeros_like(W2), b2)[0]
    assert np.array_equal(Y, np.broadcast_to(b2, Y.shape))
    Y, Z1, Y1 = OM.mlp_dense(X, np.zeros_like(W1), np.zeros_like(b1), W2, b2)
    assert not Y1.any() and np.array_equal(Y, np.broadcast_to(b2, Y.shape))
    Y = OM.mlp_dense(X, np.zeros_like(W1), b1, W2, b2)[0]
    want = OL.gelu(b1) @ W2 + b2
    assert np.allclose(Y, np.broadcast_to(want, Y.shape), rtol=0, atol=1e-15)
