"""GPU parity of tp3d_layer_fwd / tp3d_layer_bwd against the oracle.

The layer is the pre-LN GPT decoder layer of "Maximizing Parallelism in
Distributed Training for Huge Neural Networks" §3.2 on the cube (readings
in oracle/layer.py).  The oracle keeps every intermediate in float64; the GPU
keeps bf16 intermediates with fp32 accumulation and fp32 LN / softmax
statistics, and the inputs of the attention scores (LN1 output, W_qkv, Q,
K, score gradients) in fp16.  Bars, for the output, dX and every parameter
gradient: max relative error max|g - o| / max|o| <= 1e-2 and Frobenius
relative error <= 1e-2; the element-wise error with an RMS floor, which
bf16 rounding of the stored activations alone pushes past 1e-2 on tensors
of 1e5..1e7 elements, <= LAYER_ELEM_TOL (LAYER_ELEM_TOL_PEAKED for sharply
peaked attention), the measured maxima plus a margin (oracle/metrics.py): a
localised error would not stay under them.  Every case prints its triples.
"""
import numpy as np
import pytest
import torch

import synth_inputs as S
import tensor_transformer_layer_cube_gb300 as t
from oracle import layer as OY
from oracle import layouts as L
from oracle.metrics import BF16_TOL, LAYER_ELEM_TOL, LAYER_ELEM_TOL_PEAKED, fro_err, max_rel_err, rel_err
from tests.gpu_util import as_np64, assert_guards_intact, device, guarded, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = t.tp3d_create(0)
    yield c
    t.tp3d_destroy(c)


def _run(ctx, cfg: OY.LayerConfig, seed, perturb, wqkv_mult=1, forward_only=False):
    I = S.layer_inputs(cfg.batch, cfg.seq, cfg.hidden, cfg.heads, cfg.ffn, seed, perturb=perturb)
    if wqkv_mult != 1:  # a power of two: exact in bf16
        I["w_qkv"] = (I["w_qkv"].float() * wqkv_mult).to(torch.bfloat16)
    q, M, h = cfg.p, cfg.M, cfg.hidden
    params = {}
    for k, lay in OY.WEIGHT_LAYOUTS.items():
        params[k] = to_dev_bf16(I[k], lay(q))
    for k in OY.VECTORS:
        params[k] = I[k].to(device())
    X = to_dev_bf16(I["X"], L.CUBE_A(q))
    dY = to_dev_bf16(I["dY"], L.CUBE_A(q))
    c = t.tp3d_layer_cfg(q, cfg.batch, cfg.seq, h, cfg.heads, cfg.ffn, t.TP3D_BF16, cfg.eps)
    wsb = t.tp3d_layer_workspace_bytes(c)
    assert wsb > 0
    ws = torch.empty(wsb, dtype=torch.uint8, device=device())
    # outputs NaN-filled between 64 KiB guard bands (checked after each call)
    wY, Y = guarded(M * h, torch.bfloat16)
    st = t.tp3d_layer_fwd(ctx, c, params, X, Y, ws)
    assert st == 0, t.STATUS[st]
    assert t.tp3d_sync_status(ctx) == 0
    assert_guards_intact(wY, "layer Y")
    gw = {k: guarded(v.numel(), torch.bfloat16) for k, v in params.items()}
    grads = {k: g[1] for k, g in gw.items()}
    wdX, dX = guarded(M * h, torch.bfloat16)
    if not forward_only:
        st = t.tp3d_layer_bwd(ctx, c, params, X, ws, dY, dX, grads)
        assert st == 0, t.STATUS[st]
        assert t.tp3d_sync_status(ctx) == 0
        assert_guards_intact(wdX, "layer dX")
        for k, g in gw.items():
            assert_guards_intact(g[0], f"layer d{k}")
    # oracle on the same bf16 values, sharded by its own layout maps
    P64 = {k: S.as_f64(v) for k, v in I.items() if k not in ("X", "dY")}
    Ps = OY.shard_params(P64, cfg)
    Xb = L.to_sharded(S.as_f64(I["X"]), L.CUBE_A(q))
    dYb = L.to_sharded(S.as_f64(I["dY"]), L.CUBE_A(q))
    return Y, dX, grads, Xb, dYb, Ps


def _check(ctx, cfg, seed, perturb, tol=BF16_TOL, wqkv_mult=1, forward_only=False, elem_tol=LAYER_ELEM_TOL):
    Y, dX, grads, Xb, dYb, Ps = _run(ctx, cfg, seed, perturb, wqkv_mult, forward_only)
    want_Y = OY.layer_forward(Xb, Ps, cfg)
    pairs = {"Y": (as_np64(Y), want_Y)}
    if not forward_only:
        want_dX, want_g = OY.layer_backward(dYb, Xb, Ps, cfg)
        pairs["dX"] = (as_np64(dX), want_dX)
        for k in want_g:
            pairs[k] = (as_np64(grads[k]), want_g[k])
    report, bad = {}, {}
    for k, (got, want) in pairs.items():
        assert not np.isnan(got).any(), k
        e = (max_rel_err(got, want), fro_err(got, want), rel_err(got, want))
        report[k] = tuple(round(x, 5) for x in e)
        if not (e[0] <= tol and e[1] <= tol and e[2] <= elem_tol):
            bad[k] = report[k]
    # the (max-normalised, Frobenius, element-wise) triple of every tensor, shown on pass too (-rP)
    print(f"layer p={cfg.p} b={cfg.batch} s={cfg.seq} h={cfg.hidden} heads={cfg.heads} f={cfg.ffn} "
          f"seed={seed} wqkv_mult={wqkv_mult}")
    for k, e in report.items():
        print(f"  {k:7s} max {e[0]:.5f}  fro {e[1]:.5f}  elem {e[2]:.5f}")
    assert not bad, (bad, report)
    return report


def test_layer_small_perturbed(ctx):
    cfg = OY.LayerConfig(p=2, batch=2, seq=256, hidden=256, heads=2, ffn=1024)
    _check(ctx, cfg, 500, perturb=True)


def test_layer_small_zero_bias(ctx):
    cfg = OY.LayerConfig(p=2, batch=2, seq=256, hidden=512, heads=4, ffn=2048)
    _check(ctx, cfg, 510, perturb=False)


def test_layer_q1(ctx):
    cfg = OY.LayerConfig(p=1, batch=1, seq=384, hidden=256, heads=4, ffn=768)
    _check(ctx, cfg, 520, perturb=True)


def test_layer_peaked_attention(ctx):
    # QKV weights x 8 (scores x 64, |scores| about 6.6 rms): sharply peaked
    # softmax rows whose maximum keeps growing along the keys, so the
    # forward's online softmax rescales its running output many times; 3
    # query tiles per sequence (odd).  Forward and backward at the same bars:
    # the backward's sensitivity to the scores' inputs is what the fp16 score
    # path (LN1 output, W_qkv, Q, K, dS) is there for.
    cfg = OY.LayerConfig(p=1, batch=2, seq=384, hidden=256, heads=2, ffn=512)
    _check(ctx, cfg, 77, True, wqkv_mult=8, elem_tol=LAYER_ELEM_TOL_PEAKED)


def test_layer_peaked_attention_q2_d128_s1024(ctx):
    # the same regime on the q = 2 cube: head size 128, 1024 tokens per sequence
    cfg = OY.LayerConfig(p=2, batch=1, seq=1024, hidden=256, heads=2, ffn=1024)
    _check(ctx, cfg, 78, True, wqkv_mult=8, elem_tol=LAYER_ELEM_TOL_PEAKED)


def test_layer_small_qkv_weights(ctx):
    # QKV weights x 2^-10 (about 2e-5, inside fp16's subnormal range): the fp16
    # copy of W_qkv is scaled by a power of two, so the QKV product keeps its
    # precision; the scores are near zero (nearly uniform attention)
    cfg = OY.LayerConfig(p=2, batch=2, seq=256, hidden=256, heads=2, ffn=1024)
    _check(ctx, cfg, 79, True, wqkv_mult=2.0 ** -10)


def test_layer_fp16_range_error(ctx):
    # LN1 gamma = 2^15: the LN1 output (held in fp16 for the score products)
    # leaves fp16's range; the forward raises TP3D_ERANGE in the device error
    # word, and the next call with ordinary parameters runs clean
    cfg = OY.LayerConfig(p=1, batch=1, seq=128, hidden=256, heads=2, ffn=512)
    I = S.layer_inputs(cfg.batch, cfg.seq, cfg.hidden, cfg.heads, cfg.ffn, 80, perturb=False)
    q, M, h = cfg.p, cfg.M, cfg.hidden
    params = {k: to_dev_bf16(I[k], lay(q)) for k, lay in OY.WEIGHT_LAYOUTS.items()}
    params.update({k: I[k].to(device()) for k in OY.VECTORS})
    X = to_dev_bf16(I["X"], L.CUBE_A(q))
    c = t.tp3d_layer_cfg(q, cfg.batch, cfg.seq, h, cfg.heads, cfg.ffn, t.TP3D_BF16, cfg.eps)
    ws = torch.empty(t.tp3d_layer_workspace_bytes(c), dtype=torch.uint8, device=device())
    Y = torch.empty(M * h, dtype=torch.bfloat16, device=device())
    assert t.tp3d_sync_status(ctx) == 0
    big = dict(params)
    big["ln1_g"] = torch.full_like(params["ln1_g"], 2.0 ** 15)
    assert t.tp3d_layer_fwd(ctx, c, big, X, Y, ws) == 0
    assert t.STATUS[t.tp3d_sync_status(ctx)] == "TP3D_ERANGE"
    assert t.tp3d_layer_fwd(ctx, c, params, X, Y, ws) == 0
    assert t.tp3d_sync_status(ctx) == 0
    assert torch.isfinite(Y.float()).all()


def test_layer_q4_head64(ctx):
    cfg = OY.LayerConfig(p=4, batch=2, seq=1024, hidden=512, heads=8, ffn=2048)
    _check(ctx, cfg, 530, perturb=True)


def test_layer_gpt_b4_s1024_h2048_16heads(ctx):
    cfg = OY.LayerConfig(p=2, batch=4, seq=1024, hidden=2048, heads=16, ffn=8192)
    _check(ctx, cfg, S.SEED_BASE + 3, perturb=False)


def test_layer_errors_before_launch(ctx):
    x = torch.zeros(1 << 16, dtype=torch.bfloat16, device=device())
    params = {k: x for k in t.PARAM_NAMES}
    bad_seq = t.tp3d_layer_cfg(2, 2, 100, 256, 2, 1024, t.TP3D_BF16, 1e-5)
    assert t.tp3d_layer_workspace_bytes(bad_seq) == 0
    assert t.tp3d_layer_fwd(ctx, bad_seq, params, x, x, x) == 7       # seq % 128
    bad_heads = t.tp3d_layer_cfg(2, 2, 256, 256, 3, 1024, t.TP3D_BF16, 1e-5)
    assert t.tp3d_layer_fwd(ctx, bad_heads, params, x, x, x) == 2     # hidden % heads
    bad_dt = t.tp3d_layer_cfg(2, 2, 256, 256, 2, 1024, t.TP3D_F32, 1e-5)
    assert t.tp3d_layer_fwd(ctx, bad_dt, params, x, x, x) == 4
    ok = t.tp3d_layer_cfg(2, 2, 256, 256, 2, 1024, t.TP3D_BF16, 1e-5)
    p2 = dict(params)
    p2["w_o"] = None
    assert t.tp3d_layer_fwd(ctx, ok, p2, x, x, x) == 1
    assert t.tp3d_sync_status(ctx) == 0


def test_layer_step_in_a_cuda_graph(ctx):
    # The forward and the backward (whose independent launches fork onto the
    # context's side streams and join back) can be captured in one CUDA graph;
    # replaying it gives the bits of direct calls.
    cfg = OY.LayerConfig(p=2, batch=2, seq=256, hidden=512, heads=4, ffn=2048)
    I = S.layer_inputs(cfg.batch, cfg.seq, cfg.hidden, cfg.heads, cfg.ffn, 4242, perturb=True)
    q, M, h = cfg.p, cfg.M, cfg.hidden
    params = {k: to_dev_bf16(I[k], lay(q)) for k, lay in OY.WEIGHT_LAYOUTS.items()}
    params.update({k: I[k].to(device()) for k in OY.VECTORS})
    X = to_dev_bf16(I["X"], L.CUBE_A(q))
    dY = to_dev_bf16(I["dY"], L.CUBE_A(q))
    c = t.tp3d_layer_cfg(q, cfg.batch, cfg.seq, h, cfg.heads, cfg.ffn, t.TP3D_BF16, cfg.eps)
    ws = torch.empty(t.tp3d_layer_workspace_bytes(c), dtype=torch.uint8, device=device())
    Y = torch.empty(M * h, dtype=torch.bfloat16, device=device())
    dX = torch.empty(M * h, dtype=torch.bfloat16, device=device())
    grads = {k: torch.empty_like(v) for k, v in params.items()}

    def step():
        assert t.tp3d_layer_fwd(ctx, c, params, X, Y, ws) == 0
        assert t.tp3d_layer_bwd(ctx, c, params, X, ws, dY, dX, grads) == 0

    step()
    torch.cuda.synchronize()
    assert t.tp3d_sync_status(ctx) == 0
    direct = [Y.clone(), dX.clone()] + [v.clone() for v in grads.values()]
    for v in [Y, dX] + list(grads.values()):
        v.fill_(float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for v in [Y, dX] + list(grads.values()):
        v.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert t.tp3d_sync_status(ctx) == 0
    replayed = [Y, dX] + list(grads.values())
    for a, b in zip(direct, replayed):
        assert torch.equal(a, b)


def _device_case(cfg, seed):
    """Device buffers (params, X, dY) of one seeded case, and its oracle inputs."""
    I = S.layer_inputs(cfg.batch, cfg.seq, cfg.hidden, cfg.heads, cfg.ffn, seed, perturb=True)
    q = cfg.p
    params = {k: to_dev_bf16(I[k], lay(q)) for k, lay in OY.WEIGHT_LAYOUTS.items()}
    params.update({k: I[k].to(device()) for k in OY.VECTORS})
    X = to_dev_bf16(I["X"], L.CUBE_A(q))
    dY = to_dev_bf16(I["dY"], L.CUBE_A(q))
    P64 = {k: S.as_f64(v) for k, v in I.items() if k not in ("X", "dY")}
    ref = (L.to_sharded(S.as_f64(I["X"]), L.CUBE_A(q)), L.to_sharded(S.as_f64(I["dY"]), L.CUBE_A(q)),
           OY.shard_params(P64, cfg))
    return params, X, dY, ref


def _layer_outputs_vs_oracle(cfg, Y, dX, grads, ref):
    Xb, dYb, Ps = ref
    want_dX, want_g = OY.layer_backward(dYb, Xb, Ps, cfg)
    pairs = {"Y": (as_np64(Y), OY.layer_forward(Xb, Ps, cfg)), "dX": (as_np64(dX), want_dX)}
    pairs.update({k: (as_np64(grads[k]), want_g[k]) for k in want_g})
    for k, (got, want) in pairs.items():
        e = (max_rel_err(got, want), fro_err(got, want), rel_err(got, want))
        assert e[0] <= BF16_TOL and e[1] <= BF16_TOL and e[2] <= LAYER_ELEM_TOL, (k, e)


def test_layer_calls_again_with_new_contents(ctx):
    # The context keeps a CUDA graph of each call, keyed by its arguments: the
    # second forward + backward on the same buffers replays those graphs, and
    # must read the buffers' new contents (a second seed copied in place).
    cfg = OY.LayerConfig(p=2, batch=2, seq=256, hidden=256, heads=2, ffn=1024)
    q, M, h = cfg.p, cfg.M, cfg.hidden
    c = t.tp3d_layer_cfg(q, cfg.batch, cfg.seq, h, cfg.heads, cfg.ffn, t.TP3D_BF16, cfg.eps)
    ws = torch.empty(t.tp3d_layer_workspace_bytes(c), dtype=torch.uint8, device=device())
    params, X, dY, ref = _device_case(cfg, 530)
    Y = torch.empty(M * h, dtype=torch.bfloat16, device=device())
    dX = torch.empty(M * h, dtype=torch.bfloat16, device=device())
    grads = {k: torch.empty_like(v) for k, v in params.items()}
    for seed in (None, 531, 532):
        if seed is not None:
            p2, X2, dY2, ref = _device_case(cfg, seed)
            for k in params:
                params[k].copy_(p2[k])
            X.copy_(X2)
            dY.copy_(dY2)
        Y.fill_(float("nan"))
        dX.fill_(float("nan"))
        assert t.tp3d_layer_fwd(ctx, c, params, X, Y, ws) == 0
        assert t.tp3d_layer_bwd(ctx, c, params, X, ws, dY, dX, grads) == 0
        assert t.tp3d_sync_status(ctx) == 0
        _layer_outputs_vs_oracle(cfg, Y, dX, grads, ref)


def test_layer_inside_a_captured_graph(ctx):
    # Called while the caller's stream is being captured, the layer enqueues
    # its launches into that capture; replaying it gives the same bits as the
    # direct call.
    cfg = OY.LayerConfig(p=2, batch=2, seq=256, hidden=256, heads=2, ffn=1024)
    q, M, h = cfg.p, cfg.M, cfg.hidden
    c = t.tp3d_layer_cfg(q, cfg.batch, cfg.seq, h, cfg.heads, cfg.ffn, t.TP3D_BF16, cfg.eps)
    ws = torch.empty(t.tp3d_layer_workspace_bytes(c), dtype=torch.uint8, device=device())
    params, X, dY, _ = _device_case(cfg, 540)
    outs = []
    for captured in (False, True):
        Y = torch.full((M * h,), float("nan"), dtype=torch.bfloat16, device=device())
        dX = torch.full((M * h,), float("nan"), dtype=torch.bfloat16, device=device())
        grads = {k: torch.empty_like(v) for k, v in params.items()}

        def step():
            assert t.tp3d_layer_fwd(ctx, c, params, X, Y, ws) == 0
            assert t.tp3d_layer_bwd(ctx, c, params, X, ws, dY, dX, grads) == 0
        if captured:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                step()
            g.replay()
        else:
            step()
        torch.cuda.synchronize()
        assert t.tp3d_sync_status(ctx) == 0
        outs.append([Y, dX] + [grads[k] for k in sorted(grads)])
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
