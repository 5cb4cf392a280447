"""The pre-LN GPT decoder layer on the cube, forward and backward
(oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

MP3D §3.2: a Transformer layer is a Self-Attention block and an MLP block;
each block is two 3-D linears (the first with input group y = 0, the second
with y and z exchanged) so that the layer's input and output share one
direction; 3-D LayerNorm applies the matrix-vector operations of MP3D §3.1.3
(C = A * gamma, C = A + beta) and changes no direction; the 3-D linear
flattens [b/p, s/p, h/p] into [b*s/p^2, h/p], i.e. token row = batch * s +
position.  The attention core and the statistics of LayerNorm are not
described on the page (its figures are lost); every partition of them
reaches the unpartitioned layer, which is what the oracle computes.

Readings where the pages are silent: pre-LN (as GPT-2), biased variance with
eps = 1e-5, exact-erf GELU, QKV columns packed [Q | K | V] with head t using
columns t*d .. t*d+d-1 of each, causal mask (key position > query position
excluded), no dropout, softmax over keys in float64.

Layouts: X, H, Y in CUBE_A (M x h); QKV in CUBE_C (M x 3h) and the attention
output O in CUBE_C (M x h), i.e. the output direction of the first linear
and the input direction of the second; W_qkv, W_1 in CUBE_B; W_o, W_2 in
CUBE_B_SWAP; every vector (biases, gamma, beta) as a plain contiguous vector
(the diagonal layout of MP3D §3.1.1 concatenated in (j, i) order).

Backward: the vector-Jacobian product for a given upstream gradient dY,
written out from MP3D §3.1.2 (dA = dC B^T, dB = A^T dC), MP3D §3.1.3 (bias
gradient = column sums; gamma gradient = sum of dC * A-hat over rows) and the
textbook derivatives of LayerNorm, softmax and GELU.

Parity status: forward partly pinned (LN of a constant row, s = 1
attention, Q = 0 prefix mean, first token attends to itself, agreement with
torch float64 functional ops on a tiny layer); the readings above are not
pinned by the pages.  Backward pinned by central finite differences and by
torch float64 autograd on a tiny layer.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from .layouts import CUBE_A, CUBE_B, CUBE_B_SWAP, CUBE_C, from_sharded, to_sharded
from .linear import gelu, gelu_grad


@dataclass(frozen=True)
class LayerConfig:
    p: int
    batch: int
    seq: int
    hidden: int
    heads: int
    ffn: int
    eps: float = 1e-5

    @property
    def M(self):
        return self.batch * self.seq

    @property
    def d(self):
        return self.hidden // self.heads


WEIGHT_LAYOUTS = {"w_qkv": CUBE_B, "w_o": CUBE_B_SWAP, "w_1": CUBE_B, "w_2": CUBE_B_SWAP}
VECTORS = ("ln1_g", "ln1_b", "b_qkv", "b_o", "ln2_g", "ln2_b", "b_1", "b_2")


def weight_shapes(cfg: LayerConfig):
    h, f = cfg.hidden, cfg.ffn
    return {"w_qkv": (h, 3 * h), "w_o": (h, h), "w_1": (h, f), "w_2": (f, h)}


def layer_norm(x, g, b, eps):
    mu = x.mean(axis=1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mu) * rstd
    return xhat * g[None, :] + b[None, :], xhat, rstd


def layer_norm_backward(dy, xhat, rstd, g):
    dxhat = dy * g[None, :]
    return rstd * (dxhat - dxhat.mean(axis=1, keepdims=True)
                   - xhat * (dxhat * xhat).mean(axis=1, keepdims=True))


def _head_cols(cfg, t):
    h, d = cfg.hidden, cfg.d
    return slice(t * d, t * d + d), slice(h + t * d, h + t * d + d), slice(2 * h + t * d, 2 * h + t * d + d)


def _softmax_causal(Q, K, scale):
    S = (Q @ K.T) * scale
    n = S.shape[0]
    S[np.triu(np.ones((n, n), dtype=bool), 1)] = -np.inf
    S = S - S.max(axis=1, keepdims=True)
    E = np.exp(S)
    return E / E.sum(axis=1, keepdims=True)


def attention(QKV, cfg):
    """Causal multi-head attention per (batch, head): O = softmax(Q K^T/sqrt d) V."""
    O = np.zeros((cfg.M, cfg.hidden))
    scale = 1.0 / math.sqrt(cfg.d)
    for bb in range(cfg.batch):
        rows = slice(bb * cfg.seq, (bb + 1) * cfg.seq)
        for t in range(cfg.heads):
            qc, kc, vc = _head_cols(cfg, t)
            P = _softmax_causal(QKV[rows, qc], QKV[rows, kc], scale)
            O[rows, qc] = P @ QKV[rows, vc]
    return O


def attention_backward(dO, QKV, cfg):
    dQKV = np.zeros_like(QKV)
    scale = 1.0 / math.sqrt(cfg.d)
    for bb in range(cfg.batch):
        rows = slice(bb * cfg.seq, (bb + 1) * cfg.seq)
        for t in range(cfg.heads):
            qc, kc, vc = _head_cols(cfg, t)
            Q, K, V = QKV[rows, qc], QKV[rows, kc], QKV[rows, vc]
            P = _softmax_causal(Q, K, scale)
            g = dO[rows, qc]
            dV = P.T @ g
            dP = g @ V.T
            dS = P * (dP - (dP * P).sum(axis=1, keepdims=True))
            dQKV[rows, qc] = scale * (dS @ K)
            dQKV[rows, kc] = scale * (dS.T @ Q)
            dQKV[rows, vc] = dV
    return dQKV


def layer_forward_dense(X, P, cfg: LayerConfig, keep=False):
    """Y = H + MLP(LN2(H)), H = X + Attn(LN1(X)), on global float64 matrices.
    ``P`` maps parameter names to global float64 arrays."""
    X = np.asarray(X, np.float64)
    Xn1, xhat1, rstd1 = layer_norm(X, P["ln1_g"], P["ln1_b"], cfg.eps)
    QKV = Xn1 @ P["w_qkv"] + P["b_qkv"][None, :]
    O = attention(QKV, cfg)
    H = X + O @ P["w_o"] + P["b_o"][None, :]
    Xn2, xhat2, rstd2 = layer_norm(H, P["ln2_g"], P["ln2_b"], cfg.eps)
    Z1 = Xn2 @ P["w_1"] + P["b_1"][None, :]
    Y1 = gelu(Z1)
    Y = H + Y1 @ P["w_2"] + P["b_2"][None, :]
    if not keep:
        return Y
    cache = dict(X=X, Xn1=Xn1, xhat1=xhat1, rstd1=rstd1, QKV=QKV, O=O, H=H, Xn2=Xn2,
                 xhat2=xhat2, rstd2=rstd2, Z1=Z1, Y1=Y1)
    return Y, cache


def layer_backward_dense(dY, X, P, cfg: LayerConfig):
    """Returns (dX, grads) with grads keyed like the parameters."""
    _, c = layer_forward_dense(X, P, cfg, keep=True)
    dY = np.asarray(dY, np.float64)
    g = {}
    g["b_2"] = dY.sum(axis=0)
    g["w_2"] = c["Y1"].T @ dY
    dZ1 = (dY @ P["w_2"].T) * gelu_grad(c["Z1"])
    g["b_1"] = dZ1.sum(axis=0)
    g["w_1"] = c["Xn2"].T @ dZ1
    dXn2 = dZ1 @ P["w_1"].T
    g["ln2_g"] = (dXn2 * c["xhat2"]).sum(axis=0)
    g["ln2_b"] = dXn2.sum(axis=0)
    dH = dY + layer_norm_backward(dXn2, c["xhat2"], c["rstd2"], P["ln2_g"])
    g["b_o"] = dH.sum(axis=0)
    g["w_o"] = c["O"].T @ dH
    dO = dH @ P["w_o"].T
    dQKV = attention_backward(dO, c["QKV"], cfg)
    g["b_qkv"] = dQKV.sum(axis=0)
    g["w_qkv"] = c["Xn1"].T @ dQKV
    dXn1 = dQKV @ P["w_qkv"].T
    g["ln1_g"] = (dXn1 * c["xhat1"]).sum(axis=0)
    g["ln1_b"] = dXn1.sum(axis=0)
    dX = dH + layer_norm_backward(dXn1, c["xhat1"], c["rstd1"], P["ln1_g"])
    return dX, g


# ---------------------------------------------------------------- sharded

def gather_params(params, cfg: LayerConfig):
    """Sharded parameter buffers -> global float64 arrays."""
    shapes = weight_shapes(cfg)
    P = {}
    for k, lay in WEIGHT_LAYOUTS.items():
        P[k] = from_sharded(np.asarray(params[k], np.float64), lay(cfg.p), *shapes[k])
    for k in VECTORS:
        P[k] = np.asarray(params[k], np.float64)
    return P


def shard_params(P, cfg: LayerConfig):
    """Global parameter arrays -> sharded buffers (weights) / plain vectors."""
    out = {}
    for k, lay in WEIGHT_LAYOUTS.items():
        out[k] = to_sharded(np.asarray(P[k]), lay(cfg.p))
    for k in VECTORS:
        out[k] = np.asarray(P[k])
    return out


def layer_forward(X_buf, params, cfg: LayerConfig):
    """Sharded forward: X, Y in CUBE_A."""
    X = from_sharded(np.asarray(X_buf, np.float64), CUBE_A(cfg.p), cfg.M, cfg.hidden)
    Y = layer_forward_dense(X, gather_params(params, cfg), cfg)
    return to_sharded(Y, CUBE_A(cfg.p))


def layer_backward(dY_buf, X_buf, params, cfg: LayerConfig):
    """Sharded backward: dX in CUBE_A; weight gradients in their weights'
    layouts; vector gradients plain."""
    lay = CUBE_A(cfg.p)
    X = from_sharded(np.asarray(X_buf, np.float64), lay, cfg.M, cfg.hidden)
    dY = from_sharded(np.asarray(dY_buf, np.float64), lay, cfg.M, cfg.hidden)
    dX, g = layer_backward_dense(dY, X, gather_params(params, cfg), cfg)
    return to_sharded(dX, lay), shard_params(g, cfg)


def layer_flops(cfg: LayerConfig):
    """Algorithmic FLOPs of one forward and one backward (causal attention
    counts the unmasked half): linears 2M(3h^2 + h^2 + 2hf) forward, twice
    that backward; attention 2 * (2 s^2 d / 2) * b * H forward (QK^T and PV),
    twice that backward."""
    M, h, f = cfg.M, cfg.hidden, cfg.ffn
    lin = 2 * M * (3 * h * h + h * h + 2 * h * f)
    att = 2 * (2 * cfg.seq * cfg.seq * cfg.d // 2) * cfg.batch * cfg.heads
    return {"fwd": lin + att, "bwd": 2 * lin + 2 * att, "total": 3 * lin + 3 * att}
