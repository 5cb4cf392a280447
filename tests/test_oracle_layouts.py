"""Pins of the oracle's layout maps and resharding, CPU only.

What pins them (none of it re-types the oracle's formulas):
* hand-worked shard ranges from the index formulas of "Maximizing
  Parallelism in Distributed Training for Huge Neural Networks" §3.1.1;
* bijection (every global element exactly once in a non-replicated layout);
* round trips and composition of resharding;
* the per-device memory formula of the same section;
* the y <-> z exchange of the same section (last paragraph);
* the worked example of "On Optimizing the Communication of Model
  Parallelism" §2 / Figure 2 (tests/golden/cmr_figure2_unit_tasks.json).
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import layouts as L

HERE = os.path.dirname(os.path.abspath(__file__))


def _layouts_for(p):
    return [L.CUBE_A(p), L.CUBE_B(p), L.CUBE_C(p), L.CUBE_B_SWAP(p)]


SHAPES = {1: [(16, 16), (48, 32)], 2: [(16, 16), (48, 32)], 3: [(36, 36), (72, 18)]}
MESH = [L.ROW(4), L.COL(4), L.BLOCK(2, 2), L.ROW(2), L.COL(8), L.BLOCK(4, 2), L.ROW(1)]


def test_hand_worked_cube_a_ranges():
    # p = 2, M = N = 8: m = n = 2.  Device (1, 0, 1) holds
    # A[imp+jm : +m, lnp : +np] = rows 4..5, columns 4..7.
    sl = L.CUBE_A(2).slices(8, 8)
    rs, cs = sl[L.device_index(1, 0, 1, 2)]
    assert (rs.start, rs.stop, cs.start, cs.stop) == (4, 6, 4, 8)
    # device (0, 1, 0): rows 2..3, columns 0..3
    rs, cs = sl[L.device_index(0, 1, 0, 2)]
    assert (rs.start, rs.stop, cs.start, cs.stop) == (2, 4, 0, 4)


def test_hand_worked_cube_b_and_c_ranges():
    # p = 2, N = K = 8 (n = k = 2).  Device (1, 0, 1) holds
    # B_lji = B[lnp : +np, jkp+ik : +k] = rows 4..7, columns 2..3.
    rs, cs = L.CUBE_B(2).slices(8, 8)[L.device_index(1, 0, 1, 2)]
    assert (rs.start, rs.stop, cs.start, cs.stop) == (4, 8, 2, 4)
    # and C_ilj = C[imp+lm : +m, jkp : +kp] = rows 6..7, columns 0..3.
    rs, cs = L.CUBE_C(2).slices(8, 8)[L.device_index(1, 0, 1, 2)]
    assert (rs.start, rs.stop, cs.start, cs.stop) == (6, 8, 0, 4)


@pytest.mark.parametrize("p", [1, 2, 3])
def test_cube_bijection_and_round_trip(p):
    for (R, C) in SHAPES[p]:
        G = np.arange(R * C).reshape(R, C)
        for lay in _layouts_for(p):
            buf = L.to_sharded(G, lay)
            assert buf.size == R * C
            assert np.array_equal(np.sort(buf), np.arange(R * C)), lay
            assert np.array_equal(L.from_sharded(buf, lay, R, C), G)


def test_mesh_bijection_and_replicas():
    R, C = 16, 16
    G = np.arange(R * C).reshape(R, C)
    for lay in MESH:
        buf = L.to_sharded(G, lay)
        assert np.array_equal(np.sort(buf), np.arange(R * C)), lay
        assert np.array_equal(L.from_sharded(buf, lay, R, C), G)
    rep = L.to_sharded(G, L.REP(4))
    assert rep.size == 4 * R * C
    for k in range(4):
        assert np.array_equal(rep[k * R * C:(k + 1) * R * C].reshape(R, C), G)


def test_replica_read_is_replica_zero():
    R, C = 4, 4
    G = np.arange(16).reshape(R, C)
    buf = L.to_sharded(G, L.REP(3)).copy()
    buf[16:] = -1  # corrupt replicas 1 and 2: replica 0 must still be read
    assert np.array_equal(L.from_sharded(buf, L.REP(3), R, C), G)


def _all_layouts_16():
    return [L.ROW(4), L.COL(4), L.BLOCK(2, 2), L.CUBE_A(2), L.CUBE_B(2), L.CUBE_C(2),
            L.CUBE_B_SWAP(2), L.REP(4)]


def test_reshard_round_trip_and_composition():
    R, C = 16, 16
    rng = np.random.default_rng(0)
    G = rng.integers(0, 65536, size=(R, C)).astype(np.uint16)
    lays = _all_layouts_16()
    for a, b in itertools.product(lays, lays):
        x = L.to_sharded(G, a)
        y = L.reshard(x, a, b, R, C)
        assert y.dtype == np.uint16
        assert np.array_equal(L.reshard(y, b, a, R, C), x)
    for a, b, c in itertools.product(lays[:5], lays[:5], lays[:5]):
        x = L.to_sharded(G, a)
        assert np.array_equal(L.reshard(L.reshard(x, a, b, R, C), b, c, R, C), L.reshard(x, a, c, R, C))


@pytest.mark.parametrize("p,M,N,K", [(2, 16, 8, 32), (3, 18, 9, 27), (4, 32, 16, 64)])
def test_memory_per_device_formula(p, M, N, K):
    a = L.CUBE_A(p).slices(M, N)
    b = L.CUBE_B(p).slices(N, K)
    c = L.CUBE_C(p).slices(M, K)
    for d in range(p ** 3):
        size = sum((rs.stop - rs.start) * (cs.stop - cs.start) for rs, cs in (a[d], b[d], c[d]))
        assert size == L.cube_memory_per_device(M, N, K, p)


def test_direction_exchange():
    # y <-> z exchange: the A layout read in exchanged directions is where the
    # C layout left the output, and vice versa; weights keep x.
    for p in (2, 3):
        R, C = (18, 9) if p == 3 else (16, 8)
        assert L.Cube("A", p, swap=True).slices(R, C) == L.CUBE_C(p).slices(R, C)
        assert L.Cube("C", p, swap=True).slices(R, C) == L.CUBE_A(p).slices(R, C)
        assert L.CUBE_B_SWAP(p).slices(C * p, C * p) != L.CUBE_B(p).slices(C * p, C * p)


def test_vector_diagonal_layout():
    p, V = 2, 16
    b = np.arange(V)
    sl = L.vec_diag_slices(V, p)
    assert set(k for k in sl) == {(i, j, j) for i in range(p) for j in range(p)}
    # concatenated in (j, i) order the pieces are the plain vector
    cat = np.concatenate([b[sl[(i, j, j)]] for j in range(p) for i in range(p)])
    assert np.array_equal(cat, b)
    # C + b on output column block j uses b[j*V/p : (j+1)*V/p]
    for j in range(p):
        assert np.array_equal(L.vec_diag_gather_b(b, p, j), b[j * V // p:(j + 1) * V // p])


def test_rejects_non_divisible():
    with pytest.raises(ValueError):
        L.CUBE_A(2).slices(6, 8)
    with pytest.raises(ValueError):
        L.CUBE_B(2).slices(8, 6)
    with pytest.raises(ValueError):
        L.to_sharded(np.zeros((6, 6)), L.ROW(4))


def test_cmr_figure2_worked_example():
    gold = json.load(open(os.path.join(HERE, "golden", "cmr_figure2_unit_tasks.json")))
    D = np.arange(16).reshape(4, 4)
    row4 = L.ROW(4)
    s0r = L.MeshSpec(2, 2, ("S0", "R"))
    t1 = L.unit_tasks(row4, s0r, 4, 4, src_offset=0, dst_offset=4)
    assert len(t1) == gold["task1"]["n_unit_tasks"]
    rs, cs, srcs, dsts = t1[0]
    assert D[rs, cs].ravel().tolist() == gold["task1"]["first_unit_task"]["slice_elements"]
    assert dsts == gold["task1"]["first_unit_task"]["dst_devices"]
    t2 = L.unit_tasks(s0r, row4, 4, 4, src_offset=4, dst_offset=0)
    assert len(t2) == gold["task2"]["n_unit_tasks"]
    rs, cs, srcs, dsts = t2[0]
    assert D[rs, cs].ravel().tolist() == gold["task2"]["first_unit_task"]["slice_elements"]
    assert srcs == gold["task2"]["first_unit_task"]["src_devices"]
    assert dsts == gold["task2"]["first_unit_task"]["dst_devices"]
    # devices 4 and 5 hold a replica of the top slice (elements 0..7)
    buf = L.to_sharded(D, s0r)
    for dev in gold["replica_statement"]["dst_devices_holding_elements_0_to_7"]:
        assert buf[(dev - 4) * 8:(dev - 4) * 8 + 8].tolist() == list(range(8))
    # the column-slice reading contradicts the page: slice [0, 4, 8, 12]
    # would have to go to all of devices 4..7
    col = L.unit_tasks(L.COL(4), s0r, 4, 4, dst_offset=4)
    assert col[0][3] == [4, 5, 6, 7]
