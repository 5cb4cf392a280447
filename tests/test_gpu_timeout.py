"""The bounded waits' timeout path, made to run out on purpose, on the GPU.

Every wait inside the kernels gives up after the context's wait limit; the
kernel then lets what it issued land, frees its tensor memory, returns, and
the host reads TP3D_ETIMEOUT.  Here the limit is set to 20 ms and the GEMM
producers are told to stop loading after a given number of contraction
stages (tp3d_inject_load_stall), so the tensor-core issuer's next wait can
only run out: nothing faults and nothing hangs.  The stall points leave work
in flight: loads and products of a half-accumulated tile, and, past the
first tile, a finished tile's epilogue stores.  Both GEMM kernels are driven
(one CTA per tile, and CTA pairs, whose odd CTA learns of the abort only from
its own limit).  After each run-out the hook is cleared and the limit reset;
the same call then returns TP3D_OK and matches the oracle, so the drain left
the device and the context usable.
"""
import numpy as np
import pytest
import torch

import synth_inputs as S
import tensor_transformer_layer_cube_gb300 as t
from oracle import linear as OL
from oracle.metrics import BF16_TOL, rel_err
from tests.gpu_util import as_np64, device, sharded_f64, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = t.tp3d_create(0)
    yield c
    t.tp3d_inject_load_stall(c, -1)
    t.tp3d_set_wait_limit_ns(c, 0)
    t.tp3d_destroy(c)


def _linear(ctx, q, M, N, K, seed):
    A = S.normal((M, N), 1.0, seed)
    B = S.normal((N, K), 0.05, seed + 1)
    la, lb, _ = OL.linear_layouts(q, 0)
    dA, dB = to_dev_bf16(A, la), to_dev_bf16(B, lb)
    C = torch.full((M * K,), float("nan"), dtype=torch.bfloat16, device=device())

    def call():
        return t.tp3d_linear(ctx, q, 0, M, N, K, t.TP3D_BF16, dA, dB, None, 0, C)
    want = OL.linear3d(sharded_f64(A, la), sharded_f64(B, lb), q, M, N, K)
    return call, C, want


# (q, M, N, K): a CTA-pair shape (256 x 256 tiles, 8 contraction stages of
# 128 per tile, one or two tiles per pair) and a one-CTA shape (128 rows:
# 128 x 256 tiles of 4 stages of 64, three tiles per CTA on 152 SMs).  A stall
# after 0 or 2 stages stops the first tile; after 10, later tiles, with
# finished tiles' epilogues behind them
SHAPES = {"cta_pairs": (2, 2048, 1024, 4096), "one_cta": (1, 128, 256, 256 * 152 * 3)}


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("stall", [0, 2, 10])
def test_wait_runs_out_then_context_recovers(ctx, shape, stall):
    q, M, N, K = SHAPES[shape]
    call, C, want = _linear(ctx, q, M, N, K, 900 + stall)
    assert t.tp3d_sync_status(ctx) == 0
    assert t.tp3d_set_wait_limit_ns(ctx, 20_000_000) == 0
    assert t.tp3d_inject_load_stall(ctx, stall) == 0
    assert call() == 0
    assert t.STATUS[t.tp3d_sync_status(ctx)] == "TP3D_ETIMEOUT"
    # the context and the device are still usable: the same call runs clean
    assert t.tp3d_inject_load_stall(ctx, -1) == 0
    assert t.tp3d_set_wait_limit_ns(ctx, 0) == 0
    C.fill_(float("nan"))
    assert call() == 0
    assert t.tp3d_sync_status(ctx) == 0
    got = as_np64(C)
    assert not np.isnan(got).any()
    assert rel_err(got, want) <= BF16_TOL


def test_hook_arguments(ctx):
    assert t.tp3d_inject_load_stall(ctx, -2) == 1
    assert t.tp3d_inject_load_stall(None, 3) == 1
    assert t.tp3d_set_wait_limit_ns(None, 5) == 1
    assert t.tp3d_inject_load_stall(ctx, -1) == 0
