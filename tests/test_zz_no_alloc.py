"""tp3d_mlp_noalloc: the MLP entry point for callers that cannot allocate.

Some callers cannot hand the library a hidden-activation buffer: they run
where cudaMalloc is not allowed (it would synchronise the device, or all
device memory belongs to another pool) or they only own the tensors they
read and write.  tp3d_mlp_noalloc keeps the hidden activation in the
library's own fixed device array instead.  This test calls it through the C
ABI twice in a row at the array's full size, with different inputs, then
once with a much smaller hidden activation (which must not pick up what the
larger call left in the array), and checks each output against tp3d_mlp's
on the same inputs: bit for bit (both run the same deterministic kernels in
the same order; only the hidden buffer's address differs), and within the
bf16 tolerance of the other GPU tests.  It lives in its own file, collected
last, and sets up everything it uses itself, so it passes alone in a fresh
process or after the other tests.
"""
import numpy as np
import pytest
import torch

import synth_inputs as S
import tensor_transformer_layer_cube_gb300 as t
from oracle import layouts as L
from oracle.metrics import BF16_TOL, rel_err
from tests.gpu_util import as_np64, device, to_dev_bf16

pytestmark = pytest.mark.gpu


def test_mlp_noalloc_matches_tp3d_mlp_on_two_calls():
    ctx = t.tp3d_create(0)
    try:
        # M * f = 8 Mi (the whole static array) twice, then 512 x 1024 = 0.5 Mi
        for call, (q, M, h, f, seed) in enumerate(((2, 2048, 1024, 4096, 611), (2, 2048, 1024, 4096, 733),
                                                   (2, 512, 256, 1024, 857))):
            I = S.mlp_inputs(M, h, f, seed, bias_std=0.05)
            X = to_dev_bf16(I["X"], L.CUBE_A(q))
            W1 = to_dev_bf16(I["W1"], L.CUBE_B(q))
            W2 = to_dev_bf16(I["W2"], L.CUBE_B_SWAP(q))
            b1, b2 = I["b1"].to(device()), I["b2"].to(device())
            Y1 = torch.empty(M * f, dtype=torch.bfloat16, device=device())
            Y_ref = torch.empty(M * h, dtype=torch.bfloat16, device=device())
            assert t.tp3d_mlp(ctx, q, M, h, f, t.TP3D_BF16, X, W1, b1, W2, b2, Y1, Y_ref) == 0
            Y = torch.full((M * h,), float("nan"), dtype=torch.bfloat16, device=device())
            assert t.tp3d_mlp_noalloc(ctx, q, M, h, f, t.TP3D_BF16, X, W1, b1, W2, b2, Y) == 0, call
            assert t.tp3d_sync_status(ctx) == 0
            got, want = as_np64(Y), as_np64(Y_ref)
            assert not np.isnan(got).any()
            assert torch.equal(Y.view(torch.int16), Y_ref.view(torch.int16)), call
            assert rel_err(got, want) <= BF16_TOL, call
    finally:
        t.tp3d_destroy(ctx)


def test_mlp_noalloc_rejects_sizes_beyond_its_array():
    ctx = t.tp3d_create(0)
    try:
        x = torch.zeros(1 << 12, dtype=torch.bfloat16, device=device())
        y = torch.zeros(1 << 12, dtype=torch.bfloat16, device=device())
        # 4096 x 4096 hidden elements > 8 Mi: refused before anything is launched
        assert t.tp3d_mlp_noalloc(ctx, 2, 4096, 1024, 4096, t.TP3D_BF16, x, x, None, x, None, y) == 7
        assert t.tp3d_sync_status(ctx) == 0
    finally:
        t.tp3d_destroy(ctx)
