"""Pins of the oracle's 3-D linear, CPU only.

"Maximizing Parallelism in Distributed Training for Huge Neural Networks":
* §2.3: the unbalanced 2x2x2 algorithm and its printed block formula;
* §3.1.1 / Algorithm 1: all-gather in y and x, block products, reduce-scatter
  in z, emulated device by device below;
* Algorithm 7: C + b with b_j gathered from the diagonal layout;
* §3.1.2 differentiation formulas: pinned by central finite differences.
Integer inputs in [-8, 8] make every product and sum exact in float64, so the
emulations must equal the oracle bit for bit.
"""
import numpy as np
import pytest

from oracle import layouts as L
from oracle import linear as O


def _ints(rng, shape):
    return rng.integers(-8, 9, size=shape).astype(np.float64)


def _alg1_emulation(A, B, p, swap=False):
    """Device-by-device Algorithm 1 on shards, returns the flat output buffer."""
    M, N = A.shape
    K = B.shape[1]
    la, lb, lc = O.linear_layouts(p, 1 if swap else 0)
    a_sl, b_sl = la.slices(M, N), lb.slices(N, K)
    dev = lambda i, j, l: L.device_index(i, *((l, j) if swap else (j, l)), p)
    Ash = {d: A[a_sl[d]] for d in range(p ** 3)}
    Bsh = {d: B[b_sl[d]] for d in range(p ** 3)}
    Cpart = {}
    for i, j, l in L.cube_devices(p):
        # all-gather A_il in y: the p shards A_{i j' l}, stacked by rows
        A_il = np.vstack([Ash[dev(i, jj, l)] for jj in range(p)])
        # all-gather B_lj in x: the p shards B_{l j i'}, side by side
        B_lj = np.hstack([Bsh[dev(ii, j, l)] for ii in range(p)])
        Cpart[(i, j, l)] = A_il @ B_lj
    out = {}
    m = M // (p * p)
    for i, j, l in L.cube_devices(p):
        # reduce-scatter in z: sum over l in ascending order, keep rows l*m..
        C_ij = Cpart[(i, j, 0)].copy()
        for ll in range(1, p):
            C_ij = C_ij + Cpart[(i, j, ll)]
        out[dev(i, j, l)] = C_ij[l * m:(l + 1) * m]
    return np.concatenate([out[d].ravel() for d in range(p ** 3)])


@pytest.mark.parametrize("p,M,N,K", [(1, 4, 4, 4), (2, 8, 8, 8), (2, 16, 6, 12), (3, 18, 9, 27), (4, 32, 8, 32)])
@pytest.mark.parametrize("swap", [False, True])
def test_algorithm1_emulation_is_bit_exact(p, M, N, K, swap):
    rng = np.random.default_rng(p * 100 + M)
    A, B = _ints(rng, (M, N)), _ints(rng, (N, K))
    la, lb, _ = O.linear_layouts(p, 1 if swap else 0)
    got = O.linear3d(L.to_sharded(A, la), L.to_sharded(B, lb), p, M, N, K, y=1 if swap else 0)
    assert np.array_equal(got, _alg1_emulation(A, B, p, swap))


def test_unbalanced_2x2x2_block_formula():
    rng = np.random.default_rng(7)
    A, B = _ints(rng, (6, 4)), _ints(rng, (4, 10))
    A00, A01, A10, A11 = A[:3, :2], A[:3, 2:], A[3:, :2], A[3:, 2:]
    B00, B01, B10, B11 = B[:2, :5], B[:2, 5:], B[2:, :5], B[2:, 5:]
    C = np.block([[A00 @ B00 + A01 @ B10, A00 @ B01 + A01 @ B11],
                  [A10 @ B00 + A11 @ B10, A10 @ B01 + A11 @ B11]])
    assert np.array_equal(O.linear3d_dense(A, B), C)


def test_dense_product_against_triple_loop():
    rng = np.random.default_rng(3)
    A, B = rng.standard_normal((5, 7)), rng.standard_normal((7, 3))
    C = np.zeros((5, 3))
    for r in range(5):
        for c in range(3):
            acc = 0.0
            for t in range(7):
                acc += A[r, t] * B[t, c]
            C[r, c] = acc
    assert np.allclose(O.linear3d_dense(A, B), C, rtol=1e-13, atol=1e-13)


def test_bias_algorithm7_per_device():
    p, M, N, K = 2, 8, 8, 8
    rng = np.random.default_rng(11)
    A, B, b = _ints(rng, (M, N)), _ints(rng, (N, K)), _ints(rng, (K,))
    got = O.linear3d(L.to_sharded(A, L.CUBE_A(p)), L.to_sharded(B, L.CUBE_B(p)), p, M, N, K, bias=b)
    want = _alg1_emulation(A, B, p).copy()
    m, kp = M // (p * p), K // p
    for i, j, l in L.cube_devices(p):
        d = L.device_index(i, j, l, p)
        blk = want[d * m * kp:(d + 1) * m * kp].reshape(m, kp)
        blk += L.vec_diag_gather_b(b, p, j)[None, :]
    assert np.array_equal(got, want)


def test_gelu_special_values():
    assert O.gelu(np.array([0.0]))[0] == 0.0
    assert abs(O.gelu(np.array([10.0]))[0] - 10.0) < 1e-12
    assert abs(O.gelu(np.array([-10.0]))[0]) < 1e-12
    # GELU(1) = Phi(1) = 0.841344746068542949 (standard normal table)
    assert abs(O.gelu(np.array([1.0]))[0] - 0.841344746068542949) < 1e-15
    x = np.linspace(-4, 4, 17)
    h = 1e-6
    fd = (O.gelu(x + h) - O.gelu(x - h)) / (2 * h)
    assert np.allclose(O.gelu_grad(x), fd, rtol=1e-8, atol=1e-9)


def test_backward_finite_differences():
    rng = np.random.default_rng(5)
    M, N, K = 6, 5, 4
    A, B, b = rng.standard_normal((M, N)), rng.standard_normal((N, K)), rng.standard_normal(K)
    G = rng.standard_normal((M, K))
    loss = lambda A_, B_, b_: float(np.sum(O.linear3d_dense(A_, B_, b_) * G))
    dA, dB, db = O.linear3d_backward_dense(G, A, B)
    h = 1e-6
    for X, dX, name in ((A, dA, "A"), (B, dB, "B"), (b, db, "b")):
        fd = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"A": (Xp, B, b), "B": (A, Xp, b), "b": (A, B, Xp)}[name]
            args_m = {"A": (Xm, B, b), "B": (A, Xm, b), "b": (A, B, Xm)}[name]
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.allclose(dX, fd, rtol=1e-6, atol=1e-7), name


def test_sharded_backward_layouts():
    p, M, N, K = 2, 8, 8, 8
    rng = np.random.default_rng(9)
    A, B, G = _ints(rng, (M, N)), _ints(rng, (N, K)), _ints(rng, (M, K))
    for y in (0, 1):
        la, lb, lc = O.linear_layouts(p, y)
        dA, dB, db = O.linear3d_backward(L.to_sharded(G, lc), L.to_sharded(A, la), L.to_sharded(B, lb), p, M, N, K, y=y)
        assert np.array_equal(L.from_sharded(dA, la, M, N), G @ B.T)
        assert np.array_equal(L.from_sharded(dB, lb, N, K), A.T @ G)
        # bias gradient: all M rows contribute (Algorithm 8 read by its definition)
        assert np.array_equal(db, G.sum(axis=0))
