"""Pins of the oracle's GPT layer (forward and backward), CPU only.

The page ("Maximizing Parallelism ..." §3.2) fixes the structure (two 3-D
linears per block, LayerNorm as matrix-vector ops, direction restored per
block); the attention core and LayerNorm statistics are readings.  Pins:
special cases with closed forms, torch float64 functional ops (an
independent library) on a tiny layer, and central finite differences plus
torch autograd for the backward.
"""
import math

import numpy as np
import pytest
import torch

from oracle import layer as OY
from oracle import layouts as L

TINY = OY.LayerConfig(p=2, batch=2, seq=8, hidden=16, heads=2, ffn=64)
FD = OY.LayerConfig(p=2, batch=1, seq=4, hidden=8, heads=2, ffn=32)


def _params(cfg, rng, scale=0.3):
    h, f = cfg.hidden, cfg.ffn
    P = {k: scale * rng.standard_normal(s) for k, s in OY.weight_shapes(cfg).items()}
    for k, n in (("b_qkv", 3 * h), ("b_o", h), ("b_1", f), ("b_2", h), ("ln1_b", h), ("ln2_b", h)):
        P[k] = 0.1 * rng.standard_normal(n)
    P["ln1_g"] = 1 + 0.1 * rng.standard_normal(h)
    P["ln2_g"] = 1 + 0.1 * rng.standard_normal(h)
    return P


def test_layer_norm_of_constant_row_is_beta():
    x = np.full((3, 8), 2.5)
    g, b = np.arange(8.0), np.linspace(-1, 1, 8)
    y, _, _ = OY.layer_norm(x, g, b, 1e-5)
    assert np.allclose(y, np.broadcast_to(b, y.shape), atol=0, rtol=0)


def test_layer_norm_zero_mean_unit_variance():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 64)) * 3 + 1
    y, _, _ = OY.layer_norm(x, np.ones(64), np.zeros(64), 0.0)
    assert np.allclose(y.mean(axis=1), 0, atol=1e-14)
    assert np.allclose((y ** 2).mean(axis=1), 1, atol=1e-12)


def test_single_token_attention_is_value_projection():
    cfg = OY.LayerConfig(p=2, batch=4, seq=1, hidden=16, heads=2, ffn=64)
    rng = np.random.default_rng(1)
    P = _params(cfg, rng)
    X = rng.standard_normal((cfg.M, cfg.hidden))
    Xn1, _, _ = OY.layer_norm(X, P["ln1_g"], P["ln1_b"], cfg.eps)
    QKV = Xn1 @ P["w_qkv"] + P["b_qkv"]
    h = cfg.hidden
    assert np.allclose(OY.attention(QKV, cfg), QKV[:, 2 * h:], rtol=0, atol=1e-15)


def test_zero_queries_give_prefix_mean_and_first_token_attends_to_itself():
    cfg = OY.LayerConfig(p=2, batch=2, seq=6, hidden=8, heads=2, ffn=32)
    rng = np.random.default_rng(2)
    QKV = rng.standard_normal((cfg.M, 3 * cfg.hidden))
    QKV[:, :cfg.hidden] = 0.0
    O = OY.attention(QKV, cfg)
    V = QKV[:, 2 * cfg.hidden:]
    for bb in range(cfg.batch):
        rows = slice(bb * cfg.seq, (bb + 1) * cfg.seq)
        Vb = V[rows]
        want = np.cumsum(Vb, axis=0) / np.arange(1, cfg.seq + 1)[:, None]
        assert np.allclose(O[rows], want, rtol=1e-13, atol=1e-13)
    # with arbitrary queries the first token of each sequence sees only itself
    QKV2 = rng.standard_normal((cfg.M, 3 * cfg.hidden))
    O2 = OY.attention(QKV2, cfg)
    for bb in range(cfg.batch):
        r = bb * cfg.seq
        assert np.allclose(O2[r], QKV2[r, 2 * cfg.hidden:], rtol=0, atol=1e-15)


def _torch_layer(X, P, cfg):
    F = torch.nn.functional
    M, h, H, d = cfg.M, cfg.hidden, cfg.heads, cfg.d
    x1 = F.layer_norm(X, (h,), P["ln1_g"], P["ln1_b"], cfg.eps)
    qkv = x1 @ P["w_qkv"] + P["b_qkv"]
    q, k, v = qkv.split(h, dim=1)
    sh = lambda t: t.reshape(cfg.batch, cfg.seq, H, d).transpose(1, 2)
    o = F.scaled_dot_product_attention(sh(q), sh(k), sh(v), is_causal=True)
    o = o.transpose(1, 2).reshape(M, h)
    Hh = X + o @ P["w_o"] + P["b_o"]
    x2 = F.layer_norm(Hh, (h,), P["ln2_g"], P["ln2_b"], cfg.eps)
    return Hh + F.gelu(x2 @ P["w_1"] + P["b_1"], approximate="none") @ P["w_2"] + P["b_2"]


def test_forward_matches_torch_float64_functional():
    rng = np.random.default_rng(3)
    P = _params(TINY, rng)
    X = rng.standard_normal((TINY.M, TINY.hidden))
    want = _torch_layer(torch.tensor(X), {k: torch.tensor(v) for k, v in P.items()}, TINY).numpy()
    got = OY.layer_forward_dense(X, P, TINY)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_backward_matches_torch_autograd():
    rng = np.random.default_rng(4)
    P = _params(TINY, rng)
    X = rng.standard_normal((TINY.M, TINY.hidden))
    dY = rng.standard_normal((TINY.M, TINY.hidden))
    Pt = {k: torch.tensor(v, requires_grad=True) for k, v in P.items()}
    Xt = torch.tensor(X, requires_grad=True)
    _torch_layer(Xt, Pt, TINY).backward(torch.tensor(dY))
    dX, g = OY.layer_backward_dense(dY, X, P, TINY)
    assert np.allclose(dX, Xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    for k in P:
        assert np.allclose(g[k], Pt[k].grad.numpy(), rtol=1e-10, atol=1e-12), k


def test_backward_central_finite_differences():
    rng = np.random.default_rng(5)
    P = _params(FD, rng)
    X = rng.standard_normal((FD.M, FD.hidden))
    G = rng.standard_normal((FD.M, FD.hidden))
    loss = lambda X_, P_: float(np.sum(OY.layer_forward_dense(X_, P_, FD) * G))
    dX, g = OY.layer_backward_dense(G, X, P, FD)
    h = 1e-6

    def fd_of(get, setv, shape):
        out = np.zeros(shape)
        for idx in np.ndindex(shape):
            base = get()[idx]
            setv(idx, base + h)
            lp = loss(X, P)
            setv(idx, base - h)
            lm = loss(X, P)
            setv(idx, base)
            out[idx] = (lp - lm) / (2 * h)
        return out

    def set_x(idx, v):
        X[idx] = v
    fdx = fd_of(lambda: X, set_x, X.shape)
    assert np.max(np.abs(fdx - dX)) <= 1e-6 * max(1.0, np.max(np.abs(dX)))
    for k in P:
        def set_p(idx, v, k=k):
            P[k][idx] = v
        fdp = fd_of(lambda k=k: P[k], set_p, P[k].shape)
        assert np.max(np.abs(fdp - g[k])) <= 1e-6 * max(1.0, np.max(np.abs(g[k]))), k


def test_sharded_wrappers_round_trip():
    rng = np.random.default_rng(6)
    P = _params(TINY, rng)
    X = rng.standard_normal((TINY.M, TINY.hidden))
    dY = rng.standard_normal((TINY.M, TINY.hidden))
    Ps = OY.shard_params(P, TINY)
    Xb = L.to_sharded(X, L.CUBE_A(2))
    Yb = OY.layer_forward(Xb, Ps, TINY)
    assert np.allclose(L.from_sharded(Yb, L.CUBE_A(2), TINY.M, TINY.hidden), OY.layer_forward_dense(X, P, TINY))
    dXb, gs = OY.layer_backward(L.to_sharded(dY, L.CUBE_A(2)), Xb, Ps, TINY)
    dX, g = OY.layer_backward_dense(dY, X, P, TINY)
    assert np.allclose(L.from_sharded(dXb, L.CUBE_A(2), TINY.M, TINY.hidden), dX)
    for k, lay in OY.WEIGHT_LAYOUTS.items():
        shp = OY.weight_shapes(TINY)[k]
        assert np.allclose(L.from_sharded(gs[k], lay(2), *shp), g[k]), k


def test_flop_count_of_the_gpt_workload():
    cfg = OY.LayerConfig(p=2, batch=4, seq=1024, hidden=2048, heads=16, ffn=8192)
    fl = OY.layer_flops(cfg)
    assert abs(fl["fwd"] - (412.3e9 + 17.2e9)) < 0.1e9
    assert abs(fl["total"] / 1e9 - 1288.5) < 0.5
