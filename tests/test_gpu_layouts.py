"""GPU parity of tp3d_mlp_layout: the MLP block in the 1-D (Megatron) and 2-D
(SUMMA) layouts that "Maximizing Parallelism in Distributed Training for Huge
Neural Networks" compares the 3-D cube with (§2, §4), against the oracle.

The oracle shards the seeded inputs by its own layout maps (ROW / COL /
BLOCK / REP) and computes the unpartitioned MLP in float64; the outputs come
back through the same maps.  Bar: element-wise relative error with an RMS
floor <= 1e-2 (bf16 in, fp32 accumulate)."""
import numpy as np
import pytest
import torch

import synth_inputs as S
import tensor_transformer_layer_cube_gb300 as t
from oracle import layouts as L
from oracle import mlp as OM
from oracle.metrics import BF16_TOL, rel_err
from tests.gpu_util import as_np64, device, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = t.tp3d_create(0)
    yield c
    t.tp3d_destroy(c)


def _layouts(scheme, p):
    if scheme == t.TP3D_SCHEME_1D:
        return L.REP(1), L.COL(p), L.COL(p), L.ROW(p), L.REP(1)
    if scheme == t.TP3D_SCHEME_2D:
        b = L.BLOCK(p, p)
        return b, b, b, b, b
    return L.CUBE_A(p), L.CUBE_B(p), L.CUBE_C(p), L.CUBE_B_SWAP(p), L.CUBE_A(p)


def _case(ctx, scheme, p, M, h, f, seed, bias_std=0.05):
    I = S.mlp_inputs(M, h, f, seed, bias_std=bias_std)
    lx, lw1, ly1, lw2, ly = _layouts(scheme, p)
    dX, dW1, dW2 = to_dev_bf16(I["X"], lx), to_dev_bf16(I["W1"], lw1), to_dev_bf16(I["W2"], lw2)
    dY1 = torch.full((M * f,), float("nan"), dtype=torch.bfloat16, device=device())
    dY = torch.full((M * h,), float("nan"), dtype=torch.bfloat16, device=device())
    st = t.tp3d_mlp_layout(ctx, scheme, p, M, h, f, t.TP3D_BF16, dX, dW1, I["b1"].to(device()), dW2,
                           I["b2"].to(device()), dY1, dY)
    assert st == 0, t.STATUS[st]
    assert t.tp3d_sync_status(ctx) == 0
    Y, _, Y1 = OM.mlp_dense(S.as_f64(I["X"]), S.as_f64(I["W1"]), S.as_f64(I["b1"]), S.as_f64(I["W2"]),
                            S.as_f64(I["b2"]))
    got_Y = L.from_sharded(as_np64(dY), ly, M, h)
    got_Y1 = L.from_sharded(as_np64(dY1), ly1, M, f)
    return rel_err(got_Y, Y), rel_err(got_Y1, Y1)


@pytest.mark.parametrize("t_ways", [2, 4, 8])
def test_megatron_1d(ctx, t_ways):
    e, e1 = _case(ctx, t.TP3D_SCHEME_1D, t_ways, 1024, 512, 2048, 500 + t_ways)
    assert e <= BF16_TOL and e1 <= BF16_TOL


@pytest.mark.parametrize("q,M,h,f", [(2, 1024, 512, 2048), (3, 1152, 384, 1536), (4, 2048, 512, 2048)])
def test_summa_2d(ctx, q, M, h, f):
    e, e1 = _case(ctx, t.TP3D_SCHEME_2D, q, M, h, f, 600 + q)
    assert e <= BF16_TOL and e1 <= BF16_TOL


def test_cube_3d_is_tp3d_mlp(ctx):
    e, e1 = _case(ctx, t.TP3D_SCHEME_3D, 2, 1024, 512, 2048, 700)
    assert e <= BF16_TOL and e1 <= BF16_TOL


def test_layouts_agree_with_each_other(ctx):
    # the three layouts compute the same MLP from the same values: their
    # outputs differ only by fp32 summation order and bf16 rounding
    M, h, f = 512, 256, 1024
    outs = []
    for scheme, p in ((t.TP3D_SCHEME_1D, 4), (t.TP3D_SCHEME_2D, 2), (t.TP3D_SCHEME_3D, 2)):
        I = S.mlp_inputs(M, h, f, 800, bias_std=0.05)
        lx, lw1, ly1, lw2, ly = _layouts(scheme, p)
        dY1 = torch.empty(M * f, dtype=torch.bfloat16, device=device())
        dY = torch.empty(M * h, dtype=torch.bfloat16, device=device())
        assert t.tp3d_mlp_layout(ctx, scheme, p, M, h, f, t.TP3D_BF16, to_dev_bf16(I["X"], lx),
                                 to_dev_bf16(I["W1"], lw1), I["b1"].to(device()), to_dev_bf16(I["W2"], lw2),
                                 I["b2"].to(device()), dY1, dY) == 0
        assert t.tp3d_sync_status(ctx) == 0
        outs.append(L.from_sharded(as_np64(dY), ly, M, h))
    scale = np.max(np.abs(outs[2]))
    for o in outs[:2]:
        assert np.max(np.abs(o - outs[2])) <= 2.0 ** -7 * scale


def test_layout_errors(ctx):
    x = torch.zeros(1 << 16, dtype=torch.bfloat16, device=device())
    y = torch.zeros(1 << 16, dtype=torch.bfloat16, device=device())
    z = torch.zeros(1 << 16, dtype=torch.bfloat16, device=device())
    assert t.tp3d_mlp_layout(ctx, 7, 2, 64, 64, 64, t.TP3D_BF16, x, x, None, x, None, y, z) == 1   # scheme
    assert t.tp3d_mlp_layout(ctx, 1, 3, 64, 64, 64, t.TP3D_BF16, x, x, None, x, None, y, z) == 2   # f % t
    assert t.tp3d_mlp_layout(ctx, 2, 3, 64, 64, 64, t.TP3D_BF16, x, x, None, x, None, y, z) == 2   # M % q
    assert t.tp3d_mlp_layout(ctx, 1, 2, 64, 64, 64, t.TP3D_F32, x, x, None, x, None, y, z) == 4
    assert t.tp3d_mlp_layout(ctx, 2, 2, 64, 64, 64, t.TP3D_BF16, x, x, None, x, None, y, x) == 8  # Y overlaps X
    assert t.tp3d_sync_status(ctx) == 0
