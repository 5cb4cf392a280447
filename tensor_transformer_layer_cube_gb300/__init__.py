"""tensor_transformer_layer_cube_gb300 - Python binding of ``libtp3d.so``.

The library (``include/tp3d.h``) computes the 3-D tensor-parallel linear, MLP
block and GPT decoder layer of "Maximizing Parallelism in Distributed
Training for Huge Neural Networks" over a virtual q x q x q device cube held
in one GB300's memory, plus bit-exact resharding between row, column, 2-D
block, cube and replicated layouts ("On Optimizing the Communication of Model
Parallelism", §2), in hand-written sm_103a kernels.

This module only marshals arguments: every function has the name of the C
entry point it calls and returns its status code (0 = TP3D_OK).  Tensor
arguments may be torch tensors (their ``data_ptr()`` is passed), raw device
pointers (int) or None.  ``stream`` may be a ``torch.cuda.Stream``, a raw
``cudaStream_t`` (int) or None for torch's current stream.  Nothing here
computes: if ``libtp3d.so`` has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB as LIB_PATH
from .build import build

__all__ = [
    "build", "lib", "Tp3dError", "check", "STATUS", "layout",
    "tp3d_create", "tp3d_destroy", "tp3d_status_string", "tp3d_sync_status", "tp3d_reshard",
    "tp3d_linear", "tp3d_mlp", "tp3d_mlp_noalloc", "tp3d_layer_workspace_bytes", "tp3d_layer_fwd", "tp3d_layer_bwd",
    "tp3d_layout", "tp3d_layer_cfg", "tp3d_layer_params", "tp3d_layer_grads",
    "TP3D_F32", "TP3D_BF16", "CUBE_A", "CUBE_B", "CUBE_C", "CUBE_B_SWAP", "ROW", "COL", "BLOCK2D", "REPLICATED",
]

STATUS = {0: "TP3D_OK", 1: "TP3D_EINVAL", 2: "TP3D_ESHAPE", 3: "TP3D_EALIGN", 4: "TP3D_EDTYPE",
          5: "TP3D_ECUDA", 6: "TP3D_ETIMEOUT", 7: "TP3D_EUNSUPPORTED", 8: "TP3D_EOVERLAP"}
TP3D_F32, TP3D_BF16 = 0, 1
CUBE_A, CUBE_B, CUBE_C, CUBE_B_SWAP, ROW, COL, BLOCK2D, REPLICATED = range(8)


class tp3d_layout(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("q", ctypes.c_int32), ("a", ctypes.c_int32), ("b", ctypes.c_int32)]


class tp3d_layer_cfg(ctypes.Structure):
    _fields_ = [("q", ctypes.c_int32), ("batch", ctypes.c_int32), ("seq", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("heads", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("eps", ctypes.c_float)]


PARAM_NAMES = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b", "w_1", "b_1", "w_2", "b_2")


class tp3d_layer_params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in PARAM_NAMES]


class tp3d_layer_grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in PARAM_NAMES]


class Tp3dError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


def check(status: int, what: str = "") -> None:
    if status != 0:
        raise Tp3dError(status, what)


def layout(kind: int, q: int = 0, a: int = 0, b: int = 0) -> tp3d_layout:
    return tp3d_layout(kind, q, a, b)


_lib = None

_SIGS = {
    "tp3d_create": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)]),
    "tp3d_destroy": (None, [ctypes.c_void_p]),
    "tp3d_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tp3d_sync_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "tp3d_reshard": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_size_t, tp3d_layout,
                                    ctypes.c_void_p, tp3d_layout, ctypes.c_void_p, ctypes.c_void_p]),
    "tp3d_linear": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "tp3d_mlp": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "tp3d_mlp_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p]),
    "tp3d_layer_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(tp3d_layer_cfg)]),
    "tp3d_layer_fwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(tp3d_layer_cfg),
                                      ctypes.POINTER(tp3d_layer_params), ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p]),
    "tp3d_layer_bwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(tp3d_layer_cfg),
                                      ctypes.POINTER(tp3d_layer_params), ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(tp3d_layer_grads),
                                      ctypes.c_void_p]),
}


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m tensor_transformer_layer_cube_gb300.build`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _lib = h
    return _lib


def _p(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def tp3d_create(device: int = 0) -> int:
    """Returns the context handle (int); raises on failure."""
    h = ctypes.c_void_p()
    check(lib().tp3d_create(device, ctypes.byref(h)), "tp3d_create")
    return h.value


def tp3d_destroy(ctx: int) -> None:
    lib().tp3d_destroy(ctx)


def tp3d_status_string(status: int) -> str:
    return lib().tp3d_status_string(status).decode()


def tp3d_sync_status(ctx: int, stream=None) -> int:
    return lib().tp3d_sync_status(ctx, _s(stream))


def tp3d_reshard(ctx, R, C, elem_bytes, src_l: tp3d_layout, src, dst_l: tp3d_layout, dst, stream=None) -> int:
    return lib().tp3d_reshard(ctx, R, C, elem_bytes, src_l, _p(src), dst_l, _p(dst), _s(stream))


def tp3d_linear(ctx, q, y, M, N, K, dtype, A, B, bias, act, C, stream=None) -> int:
    return lib().tp3d_linear(ctx, q, y, M, N, K, dtype, _p(A), _p(B), _p(bias), act, _p(C), _s(stream))


def tp3d_mlp(ctx, q, M, h, f, dtype, X, W1, b1, W2, b2, Y1, Y, stream=None) -> int:
    return lib().tp3d_mlp(ctx, q, M, h, f, dtype, _p(X), _p(W1), _p(b1), _p(W2), _p(b2), _p(Y1), _p(Y), _s(stream))


def tp3d_mlp_noalloc(ctx, q, M, h, f, dtype, X, W1, b1, W2, b2, Y, stream=None) -> int:
    """tp3d_mlp for callers that cannot allocate: the hidden activation lives
    in the library's own fixed 16 MiB device array (M * f <= 8388608)."""
    return lib().tp3d_mlp_noalloc(ctx, q, M, h, f, dtype, _p(X), _p(W1), _p(b1), _p(W2), _p(b2), _p(Y), _s(stream))


def tp3d_layer_workspace_bytes(cfg: tp3d_layer_cfg) -> int:
    return lib().tp3d_layer_workspace_bytes(ctypes.byref(cfg))


def _params(struct, d):
    return struct(*[_p(d.get(n)) for n in PARAM_NAMES])


def tp3d_layer_fwd(ctx, cfg: tp3d_layer_cfg, params: dict, X, Y, workspace, stream=None) -> int:
    p = _params(tp3d_layer_params, params)
    return lib().tp3d_layer_fwd(ctx, ctypes.byref(cfg), ctypes.byref(p), _p(X), _p(Y), _p(workspace), _s(stream))


def tp3d_layer_bwd(ctx, cfg: tp3d_layer_cfg, params: dict, X, workspace, dY, dX, grads: dict, stream=None) -> int:
    p = _params(tp3d_layer_params, params)
    g = _params(tp3d_layer_grads, grads)
    return lib().tp3d_layer_bwd(ctx, ctypes.byref(cfg), ctypes.byref(p), _p(X), _p(workspace), _p(dY), _p(dX),
                                ctypes.byref(g), _s(stream))
