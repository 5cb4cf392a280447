"""tensor_transformer_layer_cube_gb300 - Python binding of ``libtp3d.so``.

The library (``include/tp3d.h``) computes the 3-D tensor-parallel linear, MLP
block and GPT decoder layer of "Maximizing Parallelism in Distributed
Training for Huge Neural Networks" over a virtual q x q x q device cube held
in one GB300's memory, plus bit-exact resharding between row, column, 2-D
block, cube and replicated layouts ("On Optimizing the Communication of Model
Parallelism", §2), in hand-written sm_103a kernels; and (``include/tp3d_plan.h``)
the host-side planners: the cross-mesh resharding planner of that page's
§3.2 and a pipeline-bubble simulator.

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
    "tp3d_set_wait_limit_ns", "tp3d_inject_load_stall",
    "tp3d_linear", "tp3d_mlp", "tp3d_mlp_plan", "tp3d_mlp_noalloc", "tp3d_layer_workspace_bytes", "tp3d_layer_fwd", "tp3d_layer_bwd",
    "tp3d_layout", "tp3d_layer_cfg", "tp3d_layer_params", "tp3d_layer_grads",
    "TP3D_F32", "TP3D_BF16", "CUBE_A", "CUBE_B", "CUBE_C", "CUBE_B_SWAP", "ROW", "COL", "BLOCK2D", "REPLICATED",
    "tp3d_rect", "tp3d_mesh_spec", "tp3d_cmr_options", "tp3d_cmr_result", "tp3d_pipe_cfg", "tp3d_pipe_op",
    "tp3d_pipe_result", "tp3d_layout_rects", "tp3d_mesh_rects", "tp3d_cmr_plan_create", "tp3d_cmr_plan_destroy",
    "tp3d_cmr_plan_num_tasks", "tp3d_cmr_plan_task", "tp3d_cmr_plan_lower_bound", "tp3d_cmr_schedule",
    "tp3d_pipeline_simulate", "tp3d_mlp_layout", "TP3D_SCHEME_1D", "TP3D_SCHEME_2D", "TP3D_SCHEME_3D", "TP3D_SPEC_R", "TP3D_SPEC_S0", "TP3D_SPEC_S1", "TP3D_SPEC_S01", "TP3D_CMR_NAIVE",
    "TP3D_CMR_LOAD_BALANCE", "TP3D_CMR_DFS", "TP3D_CMR_RANDOM_GREEDY", "TP3D_PIPE_GPIPE", "TP3D_PIPE_1F1B",
    "TP3D_PIPE_INTERLEAVED",
]

STATUS = {0: "TP3D_OK", 1: "TP3D_EINVAL", 2: "TP3D_ESHAPE", 3: "TP3D_EALIGN", 4: "TP3D_EDTYPE",
          5: "TP3D_ECUDA", 6: "TP3D_ETIMEOUT", 7: "TP3D_EUNSUPPORTED", 8: "TP3D_EOVERLAP",
          9: "TP3D_ERANGE"}
TP3D_F32, TP3D_BF16 = 0, 1
CUBE_A, CUBE_B, CUBE_C, CUBE_B_SWAP, ROW, COL, BLOCK2D, REPLICATED = range(8)
TP3D_SPEC_R, TP3D_SPEC_S0, TP3D_SPEC_S1, TP3D_SPEC_S01 = range(4)
TP3D_CMR_NAIVE, TP3D_CMR_LOAD_BALANCE, TP3D_CMR_DFS, TP3D_CMR_RANDOM_GREEDY = range(4)
TP3D_PIPE_GPIPE, TP3D_PIPE_1F1B, TP3D_PIPE_INTERLEAVED = range(3)
TP3D_SCHEME_1D, TP3D_SCHEME_2D, TP3D_SCHEME_3D = 1, 2, 3


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


class tp3d_rect(ctypes.Structure):
    _fields_ = [("row0", ctypes.c_int64), ("rows", ctypes.c_int64), ("col0", ctypes.c_int64),
                ("cols", ctypes.c_int64)]


class tp3d_mesh_spec(ctypes.Structure):
    _fields_ = [("m1", ctypes.c_int32), ("m2", ctypes.c_int32), ("row_spec", ctypes.c_int32),
                ("col_spec", ctypes.c_int32)]


class tp3d_cmr_options(ctypes.Structure):
    _fields_ = [("algo", ctypes.c_int32), ("trials", ctypes.c_int32), ("seed", ctypes.c_uint64),
                ("node_limit", ctypes.c_int64)]


class tp3d_cmr_result(ctypes.Structure):
    _fields_ = [("makespan", ctypes.c_int64), ("nodes", ctypes.c_int64), ("complete", ctypes.c_int32),
                ("rounds", ctypes.c_int32)]


class tp3d_pipe_cfg(ctypes.Structure):
    _fields_ = [("schedule", ctypes.c_int32), ("p", ctypes.c_int32), ("m", ctypes.c_int32), ("v", ctypes.c_int32),
                ("t_f", ctypes.c_int64), ("t_b", ctypes.c_int64)]


class tp3d_pipe_op(ctypes.Structure):
    _fields_ = [("device", ctypes.c_int32), ("microbatch", ctypes.c_int32), ("chunk", ctypes.c_int32),
                ("backward", ctypes.c_int32), ("start", ctypes.c_int64), ("end", ctypes.c_int64)]


class tp3d_pipe_result(ctypes.Structure):
    _fields_ = [("makespan", ctypes.c_int64), ("busy", ctypes.c_int64), ("idle", ctypes.c_int64),
                ("bubble", ctypes.c_double), ("max_in_flight", ctypes.c_int32)]


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
    "tp3d_set_wait_limit_ns": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint64]),
    "tp3d_inject_load_stall": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64]),
    "tp3d_reshard": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_size_t, tp3d_layout,
                                    ctypes.c_void_p, tp3d_layout, ctypes.c_void_p, ctypes.c_void_p]),
    "tp3d_linear": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "tp3d_mlp": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "tp3d_mlp_plan": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "tp3d_mlp_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p]),
    "tp3d_mlp_layout": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p]),
    "tp3d_layer_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(tp3d_layer_cfg)]),
    "tp3d_layer_fwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(tp3d_layer_cfg),
                                      ctypes.POINTER(tp3d_layer_params), ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p]),
    "tp3d_layer_bwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(tp3d_layer_cfg),
                                      ctypes.POINTER(tp3d_layer_params), ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(tp3d_layer_grads),
                                      ctypes.c_void_p]),
    "tp3d_layout_rects": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, tp3d_layout, ctypes.POINTER(tp3d_rect),
                                         ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "tp3d_mesh_rects": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, tp3d_mesh_spec, ctypes.POINTER(tp3d_rect),
                                       ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "tp3d_cmr_plan_create": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.POINTER(tp3d_rect), ctypes.c_int32, ctypes.c_int32,
                                            ctypes.POINTER(tp3d_rect), ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.POINTER(ctypes.c_void_p)]),
    "tp3d_cmr_plan_destroy": (None, [ctypes.c_void_p]),
    "tp3d_cmr_plan_num_tasks": (ctypes.c_int32, [ctypes.c_void_p]),
    "tp3d_cmr_plan_task": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(tp3d_rect),
                                          ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32),
                                          ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                          ctypes.POINTER(ctypes.c_int32)]),
    "tp3d_cmr_plan_lower_bound": (ctypes.c_int64, [ctypes.c_void_p]),
    "tp3d_cmr_schedule": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(tp3d_cmr_options),
                                         ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                         ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(tp3d_cmr_result)]),
    "tp3d_pipeline_simulate": (ctypes.c_int, [ctypes.POINTER(tp3d_pipe_cfg), ctypes.POINTER(tp3d_pipe_op),
                                              ctypes.c_int64, ctypes.POINTER(tp3d_pipe_result)]),
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


def tp3d_set_wait_limit_ns(ctx: int, ns: int) -> int:
    return lib().tp3d_set_wait_limit_ns(ctx, ns)


def tp3d_inject_load_stall(ctx: int, stages: int) -> int:
    return lib().tp3d_inject_load_stall(ctx, stages)


def tp3d_reshard(ctx, R, C, elem_bytes, src_l: tp3d_layout, src, dst_l: tp3d_layout, dst, stream=None) -> int:
    return lib().tp3d_reshard(ctx, R, C, elem_bytes, src_l, _p(src), dst_l, _p(dst), _s(stream))


def tp3d_linear(ctx, q, y, M, N, K, dtype, A, B, bias, act, C, stream=None) -> int:
    return lib().tp3d_linear(ctx, q, y, M, N, K, dtype, _p(A), _p(B), _p(bias), act, _p(C), _s(stream))


def tp3d_mlp(ctx, q, M, h, f, dtype, X, W1, b1, W2, b2, Y1, Y, stream=None) -> int:
    return lib().tp3d_mlp(ctx, q, M, h, f, dtype, _p(X), _p(W1), _p(b1), _p(W2), _p(b2), _p(Y1), _p(Y), _s(stream))


def tp3d_mlp_plan(ctx, q, M, h, f):
    """(status, launches, splits): how tp3d_mlp runs a block of these sizes."""
    n, s = ctypes.c_int(0), ctypes.c_int(0)
    st = lib().tp3d_mlp_plan(ctx, q, M, h, f, ctypes.byref(n), ctypes.byref(s))
    return st, n.value, s.value


def tp3d_mlp_noalloc(ctx, q, M, h, f, dtype, X, W1, b1, W2, b2, Y, stream=None) -> int:
    """tp3d_mlp for callers that cannot allocate: the hidden activation lives
    in the library's own fixed 16 MiB device array (M * f <= 8388608)."""
    return lib().tp3d_mlp_noalloc(ctx, q, M, h, f, dtype, _p(X), _p(W1), _p(b1), _p(W2), _p(b2), _p(Y), _s(stream))


def tp3d_mlp_layout(ctx, scheme, p, M, h, f, dtype, X, W1, b1, W2, b2, Y1, Y, stream=None) -> int:
    """The MLP block in the 1-D (Megatron), 2-D (SUMMA) or 3-D (cube) layout."""
    return lib().tp3d_mlp_layout(ctx, scheme, p, M, h, f, dtype, _p(X), _p(W1), _p(b1), _p(W2), _p(b2), _p(Y1),
                                 _p(Y), _s(stream))


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


# ---------------------------------------------------------------------------
# Host-side planners (include/tp3d_plan.h): no GPU involved.  Rectangles are
# (row0, rows, col0, cols) tuples.
# ---------------------------------------------------------------------------

def _rects_out(fn, R, C, spec):
    n = ctypes.c_int32(0)
    st = fn(R, C, spec, None, 0, ctypes.byref(n))
    if n.value <= 0:
        return st, []
    arr = (tp3d_rect * n.value)()
    st = fn(R, C, spec, arr, n.value, ctypes.byref(n))
    return st, [(r.row0, r.rows, r.col0, r.cols) for r in arr] if st == 0 else []


def tp3d_layout_rects(R, C, l: tp3d_layout):
    """(status, rectangles of the layout's shards in shard order)."""
    return _rects_out(lib().tp3d_layout_rects, R, C, l)


def tp3d_mesh_rects(R, C, s: tp3d_mesh_spec):
    """(status, rectangles of the mesh devices in mesh order)."""
    return _rects_out(lib().tp3d_mesh_rects, R, C, s)


def _rect_array(rects):
    arr = (tp3d_rect * len(rects))()
    for k, r in enumerate(rects):
        arr[k] = tp3d_rect(*r)
    return arr


def tp3d_cmr_plan_create(R, C, elem_bytes, src_rects, src_first, dst_rects, dst_first, devices_per_host):
    """(status, plan handle or None)."""
    h = ctypes.c_void_p()
    st = lib().tp3d_cmr_plan_create(R, C, elem_bytes, _rect_array(src_rects), len(src_rects), src_first,
                                    _rect_array(dst_rects), len(dst_rects), dst_first, devices_per_host,
                                    ctypes.byref(h))
    return st, h.value


def tp3d_cmr_plan_destroy(plan) -> None:
    lib().tp3d_cmr_plan_destroy(plan)


def tp3d_cmr_plan_num_tasks(plan) -> int:
    return lib().tp3d_cmr_plan_num_tasks(plan)


def tp3d_cmr_plan_task(plan, i, max_senders, max_receivers):
    """(status, slice, duration, sender devices, receiver devices) of task i;
    max_senders / max_receivers: the create call's source / destination
    device counts."""
    r, d = tp3d_rect(), ctypes.c_int64()
    ns, nr = ctypes.c_int32(), ctypes.c_int32()
    sa, ra = (ctypes.c_int32 * max_senders)(), (ctypes.c_int32 * max_receivers)()
    st = lib().tp3d_cmr_plan_task(plan, i, ctypes.byref(r), ctypes.byref(d), sa, ctypes.byref(ns), ra,
                                  ctypes.byref(nr))
    if st != 0:
        return st, None, None, [], []
    return st, (r.row0, r.rows, r.col0, r.cols), d.value, list(sa[:ns.value]), list(ra[:nr.value])


def tp3d_cmr_plan_lower_bound(plan) -> int:
    return lib().tp3d_cmr_plan_lower_bound(plan)


def tp3d_cmr_schedule(plan, algo, trials=1, seed=0, node_limit=1):
    """(status, sender host per task, global order, start time per task,
    tp3d_cmr_result)."""
    n = max(lib().tp3d_cmr_plan_num_tasks(plan), 0)
    snd, order, start = (ctypes.c_int32 * n)(), (ctypes.c_int32 * n)(), (ctypes.c_int64 * n)()
    res = tp3d_cmr_result()
    opt = tp3d_cmr_options(algo, trials, seed, node_limit)
    st = lib().tp3d_cmr_schedule(plan, ctypes.byref(opt), snd, order, start, ctypes.byref(res))
    return st, list(snd), list(order), list(start), res


def tp3d_pipeline_simulate(cfg: tp3d_pipe_cfg, want_ops: bool = False):
    """(status, tp3d_pipe_result, list of tp3d_pipe_op or None)."""
    res = tp3d_pipe_result()
    if not want_ops:
        return lib().tp3d_pipeline_simulate(ctypes.byref(cfg), None, 0, ctypes.byref(res)), res, None
    n = 2 * max(cfg.p, 0) * max(cfg.m, 0) * max(cfg.v, 0)
    ops = (tp3d_pipe_op * max(n, 1))()
    st = lib().tp3d_pipeline_simulate(ctypes.byref(cfg), ops, n, ctypes.byref(res))
    return st, res, list(ops[:n]) if st == 0 else None
