"""GPU parity of tp3d_linear and tp3d_mlp against the oracle.

The 3-D linear is Algorithm 1 (+ Algorithm 7) of "Maximizing Parallelism in
Distributed Training for Huge Neural Networks": shards in, shards out; the
oracle computes the same sharded output through its own layout maps and a
float64 product.  Bars: max element-wise relative error with an RMS floor
<= 1e-2 for bf16 (tensor cores, fp32 accumulate), <= 1e-4 for fp32 (FFMA).
Sizes span several tiles, ragged tails (shard sizes that are not multiples
of the 128 x 256 x 64 tile), q = 1..4 and both directions (y = 0, 1).
"""
import numpy as np
import pytest
import torch

import synth_inputs as S
import tensor_transformer_layer_cube_gb300 as t
from oracle import layouts as L
from oracle import linear as OL
from oracle import mlp as OM
from oracle.metrics import BF16_TOL, F32_TOL, MLP_ELEM_TOL, fro_err, max_rel_err, rel_err
from tests.gpu_util import as_np64, assert_guards_intact, device, guarded, sharded_f64, to_dev_bf16, to_dev_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = t.tp3d_create(0)
    yield c
    t.tp3d_destroy(c)


def _linear_case(ctx, q, y, M, N, K, bias, act, seed, wstd=0.05):
    A = S.normal((M, N), 1.0, seed)
    B = S.normal((N, K), wstd, seed + 1)
    b = S.normal((K,), 0.1, seed + 2) if bias else None
    la, lb, lc = OL.linear_layouts(q, y)
    whole, dC = guarded(M * K, torch.bfloat16)  # NaN-filled, between 64 KiB guard bands
    st = t.tp3d_linear(ctx, q, y, M, N, K, t.TP3D_BF16, to_dev_bf16(A, la), to_dev_bf16(B, lb),
                       b.to(device()) if bias else None, 1 if act else 0, dC)
    assert st == 0, t.STATUS[st]
    assert t.tp3d_sync_status(ctx) == 0
    assert_guards_intact(whole, f"linear q={q} y={y} {M}x{N}x{K}")
    want = OL.linear3d(sharded_f64(A, la), sharded_f64(B, lb), q, M, N, K,
                       bias=S.as_f64(b) if bias else None, act="gelu" if act else None, y=y)
    got = as_np64(dC)
    assert not np.isnan(got).any(), "output element not written"
    return rel_err(got, want)


@pytest.mark.parametrize("q,M,N,K", [
    (1, 256, 128, 256),
    (2, 512, 256, 1024),     # several tiles per shard
    (2, 1024, 512, 2048),
    (3, 1152, 384, 576),     # q = 3: 128-row, 128-col, 64-col shards
    (4, 2048, 256, 4096),
])
@pytest.mark.parametrize("y", [0, 1])
def test_linear_bf16_parity(ctx, q, M, N, K, y):
    assert _linear_case(ctx, q, y, M, N, K, bias=False, act=False, seed=100 + q) <= BF16_TOL


@pytest.mark.parametrize("q,M,N,K", [
    (2, 4000, 1040, 4192),   # large enough for CTA pairs: 1000-row shards, 520 / 1048-wide blocks
    (2, 800, 192, 416),      # m = 200 rows, contraction block 96, weight block 104: ragged everywhere
    (2, 4 * 136, 2 * 72, 4 * 264),
    (3, 9 * 72, 3 * 80, 9 * 40),
    (1, 2048, 1024, 1280),   # an odd number of 256-column tiles: clusters of two CTA pairs end half-used
    (1, 2304, 512, 768),
])
def test_linear_bf16_ragged_tiles(ctx, q, M, N, K):
    for y in (0, 1):
        assert _linear_case(ctx, q, y, M, N, K, bias=True, act=True, seed=200 + q) <= BF16_TOL


def test_linear_bf16_bias_gelu(ctx):
    assert _linear_case(ctx, 2, 0, 2048, 1024, 4096, bias=True, act=True, seed=S.SEED_BASE + 2) <= BF16_TOL


@pytest.mark.parametrize("y,bias,act", [(0, False, False), (1, False, False), (0, True, True), (1, True, False)])
def test_linear_f32_config_q2_64(ctx, y, bias, act):
    q, M, N, K = 2, 64, 64, 64
    seed = S.SEED_BASE + 1
    A = S.normal((M, N), 1.0, seed, dtype=torch.float32)
    B = S.normal((N, K), 1.0, seed + 1, dtype=torch.float32)
    b = S.normal((K,), 1.0, seed + 2, dtype=torch.float32) if bias else None
    la, lb, lc = OL.linear_layouts(q, y)
    dC = torch.full((M * K,), float("nan"), dtype=torch.float32, device=device())
    st = t.tp3d_linear(ctx, q, y, M, N, K, t.TP3D_F32, to_dev_f32(A, la), to_dev_f32(B, lb),
                       b.to(device()) if bias else None, 1 if act else 0, dC)
    assert st == 0
    assert t.tp3d_sync_status(ctx) == 0
    want = OL.linear3d(sharded_f64(A, la), sharded_f64(B, lb), q, M, N, K,
                       bias=S.as_f64(b) if bias else None, act="gelu" if act else None, y=y)
    assert rel_err(dC.cpu().numpy(), want) <= F32_TOL


def _mlp_case(ctx, q, M, h, f, seed, bias_std, sample_rows=None):
    I = S.mlp_inputs(M, h, f, seed, bias_std=bias_std)
    dX = to_dev_bf16(I["X"], L.CUBE_A(q))
    dW1 = to_dev_bf16(I["W1"], L.CUBE_B(q))
    dW2 = to_dev_bf16(I["W2"], L.CUBE_B_SWAP(q))
    whole1, dY1 = guarded(M * f, torch.bfloat16)
    whole, dY = guarded(M * h, torch.bfloat16)
    st = t.tp3d_mlp(ctx, q, M, h, f, t.TP3D_BF16, dX, dW1, I["b1"].to(device()), dW2, I["b2"].to(device()), dY1, dY)
    assert st == 0, t.STATUS[st]
    assert t.tp3d_sync_status(ctx) == 0
    assert_guards_intact(whole1, "MLP Y1")
    assert_guards_intact(whole, "MLP Y")
    Yg = L.from_sharded(as_np64(dY), L.CUBE_A(q), M, h)
    X, W1, W2 = S.as_f64(I["X"]), S.as_f64(I["W1"]), S.as_f64(I["W2"])
    b1, b2 = S.as_f64(I["b1"]), S.as_f64(I["b2"])
    if sample_rows is None:
        Ym, Y1m = OM.mlp3d(L.to_sharded(X, L.CUBE_A(q)), L.to_sharded(W1, L.CUBE_B(q)), b1,
                           L.to_sharded(W2, L.CUBE_B_SWAP(q)), b2, q, M, h, f)
        got, want = as_np64(dY), Ym
        e1 = rel_err(as_np64(dY1), Y1m)
    else:
        got, want = Yg[sample_rows], OM.mlp_rows_dense(X[sample_rows], W1, b1, W2, b2)
        e1 = 0.0
    # Y passes through the bf16 hidden activation: the 1e-2 bar on the
    # max-normalised and Frobenius errors, the element-wise one at MLP_ELEM_TOL
    em, ef = max_rel_err(got, want), fro_err(got, want)
    print(f"MLP q={q} M={M} h={h} f={f}: Y max-normalised {em:.5f} Frobenius {ef:.5f}; Y1 element-wise {e1:.5f}")
    assert em <= BF16_TOL and ef <= BF16_TOL, (em, ef)
    return rel_err(got, want), e1


def test_mlp_q2_tokens2048_hidden1024_ffn4096(ctx):
    e, e1 = _mlp_case(ctx, 2, 2048, 1024, 4096, S.SEED_BASE + 2, 0.0)
    assert e <= MLP_ELEM_TOL and e1 <= BF16_TOL


def test_mlp_q2_with_biases(ctx):
    e, e1 = _mlp_case(ctx, 2, 1024, 512, 2048, 300, 0.05)
    assert e <= MLP_ELEM_TOL and e1 <= BF16_TOL


def test_mlp_plan_chains_small_blocks(ctx):
    # config 2 (36 MiB of operands, 32 tiles in the second GEMM): one launch,
    # the second GEMM's contraction in two halves
    assert t.tp3d_mlp_plan(ctx, 2, 2048, 1024, 4096) == (0, 1, 2)
    # 4096 tokens, ffn 2048 (32 MiB): one launch; 64 second-GEMM tiles, whole contractions
    assert t.tp3d_mlp_plan(ctx, 2, 4096, 1024, 2048) == (0, 1, 1)
    # config 4 (far beyond 64 MiB): two GEMM launches
    assert t.tp3d_mlp_plan(ctx, 4, 8192, 4096, 16384) == (0, 2, 0)
    # tiles that would be partial: two launches
    assert t.tp3d_mlp_plan(ctx, 1, 200, 64, 128) == (0, 2, 0)


def test_mlp_chain_whole_contractions(ctx):
    # the chained launch without contraction halves, against the oracle in full
    assert t.tp3d_mlp_plan(ctx, 2, 4096, 1024, 2048)[1:] == (1, 1)
    e, e1 = _mlp_case(ctx, 2, 4096, 1024, 2048, 310, 0.05)
    assert e <= MLP_ELEM_TOL and e1 <= BF16_TOL


def _bf16_ulp(x: np.ndarray) -> np.ndarray:
    """The spacing of bf16 numbers at |x| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def _chain_vs_separate(ctx, q, M, h, f, seed, splits):
    """tp3d_mlp (one chained launch) and the same block as two tp3d_linear
    launches on the same inputs.  Y1 agrees bit for bit (the same products in
    the same order).  So does Y when the chain contracts whole rows of Y1
    (splits 1); with the contraction in two halves (splits 2) Y's fp32 sums
    are the two halves' sums added, so Y agrees to one bf16 unit (and the
    accumulation noise where a sum cancels)."""
    assert t.tp3d_mlp_plan(ctx, q, M, h, f) == (0, 1, splits)
    I = S.mlp_inputs(M, h, f, seed, bias_std=0.05)
    dX = to_dev_bf16(I["X"], L.CUBE_A(q))
    dW1 = to_dev_bf16(I["W1"], L.CUBE_B(q))
    dW2 = to_dev_bf16(I["W2"], L.CUBE_B_SWAP(q))
    b1, b2 = I["b1"].to(device()), I["b2"].to(device())
    outs = []
    for chained in (True, False):
        Y1 = torch.full((M * f,), float("nan"), dtype=torch.bfloat16, device=device())
        Y = torch.full((M * h,), float("nan"), dtype=torch.bfloat16, device=device())
        if chained:
            assert t.tp3d_mlp(ctx, q, M, h, f, t.TP3D_BF16, dX, dW1, b1, dW2, b2, Y1, Y) == 0
        else:
            assert t.tp3d_linear(ctx, q, 0, M, h, f, t.TP3D_BF16, dX, dW1, b1, 1, Y1) == 0
            assert t.tp3d_linear(ctx, q, 1, M, f, h, t.TP3D_BF16, Y1, dW2, b2, 0, Y) == 0
        assert t.tp3d_sync_status(ctx) == 0
        outs.append((Y1, Y))
    (c1, c), (s1, sy) = outs
    assert torch.equal(c1.view(torch.int16), s1.view(torch.int16))
    if splits == 1:
        assert torch.equal(c.view(torch.int16), sy.view(torch.int16))
    else:
        # one bf16 unit, plus the fp32 accumulation's own noise where the sum
        # cancels (1e-4 of the output's scale: a 4096-term sum of products of
        # magnitude 1e-2 carries about 1e-5 absolute)
        a, b = as_np64(c), as_np64(sy)
        assert not np.isnan(a).any()
        diff = np.abs(a - b)
        tol = _bf16_ulp(np.maximum(np.abs(a), np.abs(b))) + 1e-4 * np.abs(b).max()
        assert (diff <= tol).all(), float((diff / tol).max())
        print(f"chain (two halves) vs two launches: {np.count_nonzero(diff)} of {a.size} Y elements differ")


def test_mlp_chain_matches_two_launches(ctx):
    _chain_vs_separate(ctx, 2, 4096, 1024, 2048, 330, 1)
    _chain_vs_separate(ctx, 2, 2048, 1024, 4096, 331, 2)


def test_mlp_chain_calls_in_a_row(ctx):
    # chained calls back to back on one context, different sizes, inputs and
    # contraction splits: each launch leaves its counters zero for the next
    e, e1 = _mlp_case(ctx, 2, 2048, 1024, 4096, 320, 0.05)  # two contraction halves
    assert e <= MLP_ELEM_TOL and e1 <= BF16_TOL
    _chain_vs_separate(ctx, 2, 4096, 1024, 2048, 321, 1)  # whole contractions
    _chain_vs_separate(ctx, 2, 2048, 1024, 4096, 322, 2)
    e, e1 = _mlp_case(ctx, 2, 2048, 1024, 4096, 323, 0.05)
    assert e <= MLP_ELEM_TOL and e1 <= BF16_TOL


def test_mlp_q4_tokens8192_hidden4096_ffn16384_sampled_rows(ctx):
    # row-separable: a seeded sample of rows covering every virtual shard of the output
    q, M = 4, 8192
    rng = np.random.default_rng(4)
    m = M // (q * q)
    rows = np.concatenate([blk * m + rng.choice(m, 16, replace=False) for blk in range(q * q)])
    e, _ = _mlp_case(ctx, q, M, 4096, 16384, S.SEED_BASE + 4, 0.0, sample_rows=np.sort(rows))
    assert e <= BF16_TOL


def test_linear_gelu_activation_values(ctx):
    # A = 0: every output is GELU(bias) of its column, for bf16 biases densely
    # covering [-8, 8] (the epilogue's erf is a rational approximation,
    # |error| <= 1.5e-7): within one bf16 unit of the exact value, plus 1e-6
    # absolute where GELU's lower tail is far below fp32's resolution of 1 + erf
    q, M, N, K = 1, 256, 64, 4096
    b = torch.linspace(-8.0, 8.0, K, dtype=torch.float64).to(torch.bfloat16)
    A = torch.zeros(M * N, dtype=torch.bfloat16, device=device())
    B = torch.zeros(N * K, dtype=torch.bfloat16, device=device())
    C = torch.full((M * K,), float("nan"), dtype=torch.bfloat16, device=device())
    assert t.tp3d_linear(ctx, q, 0, M, N, K, t.TP3D_BF16, A, B, b.to(device()), 1, C) == 0
    assert t.tp3d_sync_status(ctx) == 0
    x = b.double()
    want = (x * 0.5 * (1.0 + torch.erf(x / np.sqrt(2.0)))).numpy()
    got = C.view(M, K).double().cpu().numpy()
    ulp = np.maximum(np.abs(want), 2.0 ** -126) * 2.0 ** -7
    assert np.all(np.abs(got - want[None, :]) <= ulp[None, :] + 1e-6)


def test_linear_errors_before_launch(ctx):
    x = torch.zeros(1 << 16, dtype=torch.bfloat16, device=device())
    w = torch.zeros(1 << 16, dtype=torch.bfloat16, device=device())
    o = torch.zeros(1 << 16, dtype=torch.bfloat16, device=device())
    assert t.tp3d_linear(ctx, 2, 0, 6, 8, 8, t.TP3D_BF16, x, w, None, 0, o) == 2    # M % q^2
    assert t.tp3d_linear(ctx, 2, 0, 8, 8, 6, t.TP3D_BF16, x, w, None, 0, o) == 2    # K % q^2
    assert t.tp3d_linear(ctx, 0, 0, 8, 8, 8, t.TP3D_BF16, x, w, None, 0, o) == 1    # q
    assert t.tp3d_linear(ctx, 2, 2, 8, 8, 8, t.TP3D_BF16, x, w, None, 0, o) == 1    # y
    assert t.tp3d_linear(ctx, 2, 0, 8, 8, 8, 7, x, w, None, 0, o) == 4              # dtype
    assert t.tp3d_linear(ctx, 2, 0, 64, 64, 64, t.TP3D_BF16, x.data_ptr() + 2, w, None, 0, o) == 3  # align
    assert t.tp3d_linear(ctx, 2, 0, 64, 64, 64, t.TP3D_BF16, x, w, None, 0, x) == 8  # overlap
    assert t.tp3d_linear(ctx, 2, 0, 64, 64, 64, t.TP3D_BF16, None, w, None, 0, o) == 1
    assert t.tp3d_mlp(ctx, 2, 64, 64, 64, t.TP3D_F32, x, w, None, w, None, o, o) == 4
    assert t.tp3d_sync_status(ctx) == 0
