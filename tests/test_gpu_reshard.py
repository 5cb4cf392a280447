"""GPU parity of tp3d_reshard against the oracle: bit-exact.

Resharding is the layout conversion of "On Optimizing the Communication of
Model Parallelism" §2 among row-split, column-split, 2-D block, cube and
replicated layouts; every destination word must equal the oracle's bit for
bit, for every ordered pair of layouts.  Every destination buffer sits between
two 64 KiB guard bands that must come back unchanged (a store outside the
output would show there).  The cases cover the three kernels: cells whose
rows are whole 16-byte vectors, cells of 64 bytes and more whose rows are not
16-byte aligned (staged through shared memory and realigned), and narrow
cells.
"""
import itertools

import numpy as np
import pytest
import torch

import synth_inputs as S
import tensor_transformer_layer_cube_gb300 as t
from oracle import layouts as L
from tests.gpu_util import assert_guards_intact, bits_u16, device, guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = t.tp3d_create(0)
    yield c
    t.tp3d_destroy(c)


def _pairs(q=2, s=4):
    lays = [
        ("ROW4", L.ROW(s), t.layout(t.ROW, 0, s)),
        ("COL4", L.COL(s), t.layout(t.COL, 0, s)),
        ("BLK2x2", L.BLOCK(2, 2), t.layout(t.BLOCK2D, 0, 2, 2)),
        ("CUBE_A", L.CUBE_A(q), t.layout(t.CUBE_A, q)),
        ("REP4", L.REP(s), t.layout(t.REPLICATED, 0, s)),
    ]
    return [(a, b) for a, b in itertools.product(lays, lays) if a[0] != b[0]]


def _run(ctx, R, C, G_bits, src, dst, esz=2):
    dt = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}[esz]
    npdt = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}[esz]
    sbuf = L.to_sharded(G_bits, src[1])
    want = L.reshard(sbuf, src[1], dst[1], R, C)
    sview = {1: np.uint8, 2: np.int16, 4: np.int32, 8: np.int64}[esz]
    d_src = torch.from_numpy(np.ascontiguousarray(sbuf.astype(npdt)).view(sview)).to(device())
    whole, d_dst = guarded(want.size, dt)
    assert t.tp3d_reshard(ctx, R, C, esz, src[2], d_src, dst[2], d_dst) == 0
    assert t.tp3d_sync_status(ctx) == 0
    got = d_dst.cpu().numpy().view(npdt)
    assert np.array_equal(got, want.astype(npdt)), (src[0], dst[0])
    assert_guards_intact(whole, f"{src[0]} -> {dst[0]}")


@pytest.mark.parametrize("R,C", [(64, 64), (256, 512), (1024, 96)])
def test_all_pairs_small_bits(ctx, R, C):
    G = S.bf16_bits(S.random_bits16((R, C), 7).view(torch.bfloat16)).reshape(R, C)
    for src, dst in _pairs():
        _run(ctx, R, C, G, src, dst)


def test_cube_layouts_all_kinds(ctx):
    R, C = 288, 144  # q = 3: block sizes 32 / 48 / 16 rows and cols
    G = S.bf16_bits(S.random_bits16((R, C), 8).view(torch.bfloat16)).reshape(R, C)
    lays = [(n, f(3), t.layout(k, 3)) for n, f, k in
            (("A", L.CUBE_A, t.CUBE_A), ("B", L.CUBE_B, t.CUBE_B), ("C", L.CUBE_C, t.CUBE_C),
             ("BS", L.CUBE_B_SWAP, t.CUBE_B_SWAP))]
    lays.append(("ROW1", L.ROW(1), t.layout(t.ROW, 0, 1)))
    for a, b in itertools.permutations(lays, 2):
        _run(ctx, R, C, G, a, b)


def _q3_lays(q=3, rep=3):
    return [("CUBE_A", L.CUBE_A(q), t.layout(t.CUBE_A, q)), ("CUBE_B", L.CUBE_B(q), t.layout(t.CUBE_B, q)),
            ("CUBE_C", L.CUBE_C(q), t.layout(t.CUBE_C, q)), ("COL3", L.COL(3), t.layout(t.COL, 0, 3)),
            ("ROW3", L.ROW(3), t.layout(t.ROW, 0, 3)), ("REP3", L.REP(rep), t.layout(t.REPLICATED, 0, rep))]


@pytest.mark.parametrize("esz,R,C", [(2, 1170, 1170), (1, 630, 630), (4, 450, 450), (8, 99, 99)])
def test_unaligned_rows_staged_path(ctx, esz, R, C):
    # q = 3 cube layouts whose block widths are not whole 16-byte vectors
    # (bf16 1170: 390 / 130 columns = 780 / 260 bytes), cells of 64 bytes and
    # more: the shared-memory staged kernel (rows of 2340 bytes take two jobs);
    # a replicated destination whose copies
    # start at other alignments (R C esz not a multiple of 16)
    rng = np.random.default_rng(esz + 100)
    npdt = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}[esz]
    G = rng.integers(0, np.iinfo(npdt).max, size=(R, C), dtype=npdt)
    for a, b in itertools.permutations(_q3_lays(), 2):
        _run(ctx, R, C, G, a, b, esz=esz)


def test_full_size_unaligned_8190(ctx):
    # 8190 x 8190 bf16 (128 MiB) on the q = 3 cube: 2730- and 910-column
    # blocks (5460 and 1820 bytes, not 16-byte multiples)
    R = C = 8190
    G = S.bf16_bits(S.random_bits16((R, C), S.SEED_BASE + 51).view(torch.bfloat16)).reshape(R, C)
    lays = _q3_lays()
    for a, b in [(lays[0], lays[1]), (lays[1], lays[3]), (lays[4], lays[2]), (lays[0], lays[5])]:
        _run(ctx, R, C, G, a, b)


def test_unaligned_cells_take_the_element_path(ctx):
    R, C = 36, 36  # q = 3 cube: 4-row blocks and 12-column blocks; ROW(3): 12 rows (8-byte cells)
    G = S.bf16_bits(S.random_bits16((R, C), 9).view(torch.bfloat16)).reshape(R, C)
    a = ("CUBE_B", L.CUBE_B(3), t.layout(t.CUBE_B, 3))
    b = ("COL3", L.COL(3), t.layout(t.COL, 0, 3))
    c = ("ROW3", L.ROW(3), t.layout(t.ROW, 0, 3))
    for x, y in itertools.permutations([a, b, c], 2):
        _run(ctx, R, C, G, x, y)


@pytest.mark.parametrize("esz", [1, 4, 8])
def test_other_word_sizes(ctx, esz):
    R, C = 64, 128
    rng = np.random.default_rng(esz)
    npdt = {1: np.uint8, 4: np.uint32, 8: np.uint64}[esz]
    G = rng.integers(0, np.iinfo(npdt).max, size=(R, C), dtype=npdt)
    for src, dst in _pairs()[:8]:
        _run(ctx, R, C, G, src, dst, esz=esz)


@pytest.mark.parametrize("values", ["ints", "bits"])
def test_full_size_8192_all_20_pairs(ctx, values):
    R = C = 8192
    if values == "ints":
        G = S.bf16_bits(S.uniform_ints((R, C), -256, 256, S.SEED_BASE + 5)).reshape(R, C)
    else:
        G = S.bf16_bits(S.random_bits16((R, C), S.SEED_BASE + 50).view(torch.bfloat16)).reshape(R, C)
    pairs = _pairs()
    assert len(pairs) == 20
    for src, dst in pairs:
        _run(ctx, R, C, G, src, dst)


def test_errors_are_returned_before_launch(ctx):
    x = torch.zeros(64 * 64, dtype=torch.int16, device=device())
    y = torch.zeros(64 * 64, dtype=torch.int16, device=device())
    ok = t.layout(t.ROW, 0, 4)
    assert t.tp3d_reshard(ctx, 64, 64, 2, ok, x, ok, x) == 8          # overlap
    assert t.tp3d_reshard(ctx, 64, 64, 2, t.layout(t.ROW, 0, 3), x, ok, y) == 2  # 64 % 3
    assert t.tp3d_reshard(ctx, 64, 64, 3, ok, x, ok, y) == 1          # word size
    assert t.tp3d_reshard(ctx, 64, 64, 2, t.layout(99), x, ok, y) == 1  # kind
    assert t.tp3d_reshard(ctx, 64, 64, 2, ok, None, ok, y) == 1
    assert t.tp3d_reshard(ctx, 64, 64, 2, t.layout(t.CUBE_A, 0), x, ok, y) == 1  # q = 0
    assert t.tp3d_sync_status(ctx) == 0
