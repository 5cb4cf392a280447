#!/usr/bin/env python
"""Benchmark of the 3-D tensor-parallel layer cube on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload layer_q2|mlp_q2|mlp_q4|reshard]

Prints ONE JSON line (rank 0).  A step is one pass of the workload's whole
hot path over one batch of synthetic input already resident in HBM; every
timed step is bracketed by CUDA events on the launching stream and followed,
outside the events, by a 256 MiB write that flushes L2 and a 256 MiB read
that writes the flush's dirty lines back before the next step.  `value` is the
whole-job throughput (all ranks' work / the slowest rank's time).  `e2e` is
the same metric through the public C-ABI call with the step's input copied
from pinned host memory and its result copied back inside the timed region.
Extra objects: `roofline` (dominant kernel, timed live with CUDA events),
`cpu_baseline` (the fp64 oracle on a bounded sample on the host cores),
`reshard` (the resharding sweep among row-4, column-4, 2x2 block, q=2 cube
and 4-replica layouts of an 8192 x 8192 bf16 matrix, GB/s), `clocks`
(nvidia-smi samples taken during the timed region).

Multi-GPU: the cube is virtual and lives in one GPU's memory, so the path
does not shard across GPUs: N ranks run N independent replicas, with no
collective on the data path ("scaling": "weak").

`--impl reference` times the fp64 CPU oracle (the reference arm of this
build) on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "3D-partitioned layer TFLOP/s (% bf16 peak); resharding GB/s (% of HBM)"
DEFAULT_WORKLOAD = "layer_q2"

WORKLOADS = {
    "linear_f32_q2": dict(kind="linear_f32", q=2, M=64, N=64, K=64,
                          name="3-D linear C=A.B on a q=2 cube (8 virtual devices), M=N=K=64, fp32"),
    "mlp_q2": dict(kind="mlp", q=2, M=2048, h=1024, f=4096,
                   name="Megatron MLP (column-split Linear+GELU, row-split Linear) on a q=2 cube: "
                        "tokens 2048, hidden 1024, ffn 4096, bf16"),
    "layer_q2": dict(kind="layer", q=2, batch=4, seq=1024, hidden=2048, heads=16, ffn=8192,
                     name="GPT decoder layer fwd+bwd on a q=2 cube: batch 4, seq 1024, hidden 2048, "
                          "16 heads, ffn 8192, bf16"),
    "mlp_q4": dict(kind="mlp", q=4, M=8192, h=4096, f=16384,
                   name="MLP on a q=4 cube (64 virtual devices): tokens 8192, hidden 4096, ffn 16384, bf16"),
    "reshard": dict(kind="reshard", R=8192, C=8192,
                    name="resharding sweep, 8192x8192 bf16, 20 ordered pairs of ROW4 COL4 BLK2x2 CUBE_A(q=2) REP4"),
    "reshard_q3": dict(kind="reshard", R=8190, C=8190, q3=True,
                       name="resharding sweep, 8190x8190 bf16, 30 ordered pairs of CUBE_A CUBE_B CUBE_C (q=3) "
                            "ROW3 COL3 REP3 (block rows of 5460, 1820 and 16380 bytes: not 16-byte aligned)"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU baseline sample budget")
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads and the CPU baseline")
    ap.add_argument("--no-graph", action="store_true",
                    help="time direct C-ABI calls instead of replaying a CUDA graph of the step")
    ap.add_argument("--probe-only", action="store_true",
                    help="only launch the dominant kernel three times (for profiler captures)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sustained": d["bf16_tflops_sustained"],
                "source": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        rows = [r.split(", ") for r in open(self.path).read().strip().splitlines() if r.count(",") >= 9]
        os.unlink(self.path)
        return rows

    @staticmethod
    def summarize(rows, t0, t1):
        def ts(r):
            try:
                return time.mktime(time.strptime(r[0].split(".")[0], "%Y/%m/%d %H:%M:%S")) + float("0." + r[0].split(".")[1])
            except (ValueError, IndexError):
                return None
        inside = [r for r in rows if ts(r) is not None and t0 - 0.05 <= ts(r) <= t1 + 0.05]
        note = "samples inside the timed region"
        if not inside:
            inside = rows
            note = "timed region shorter than the sampling period: all samples of the run"
        sm = [float(r[2]) for r in inside if r[2].strip().replace(".", "").isdigit()]
        mx = [float(r[3]) for r in inside if r[3].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in inside for k in range(4) if r[6 + k].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "note": note}


# ----------------------------------------------------------------- workloads
def _randn(torch, n, dev, g, std=1.0):
    return (torch.randn(n, device=dev, generator=g) * std).to(torch.bfloat16)


class MlpBench:
    """Config 2 / 4: tp3d_mlp (linear 1 with bias + GELU, linear 2 with bias)."""

    def __init__(self, t, ctx, dev, w, seed=20262):
        import torch
        self.t, self.ctx, self.w = t, ctx, w
        q, M, h, f = w["q"], w["M"], w["h"], w["f"]
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        bf = torch.bfloat16
        self.X = _randn(torch, M * h, dev, g)
        self.W1 = _randn(torch, h * f, dev, g, 0.02)
        self.W2 = _randn(torch, f * h, dev, g, 0.02)
        self.b1 = torch.zeros(f, device=dev, dtype=bf)
        self.b2 = torch.zeros(h, device=dev, dtype=bf)
        self.Y1 = torch.empty(M * f, device=dev, dtype=bf)
        self.Y = torch.empty(M * h, device=dev, dtype=bf)
        self.units = 4.0 * M * h * f
        # one chained launch for a small block, else two GEMM launches
        st, n, splits = t.tp3d_mlp_plan(ctx, q, M, h, f)
        t.check(st, "tp3d_mlp_plan")
        self.launches, self.splits = n, splits
        self.unit, self.scale = "TFLOP/s", 1e12
        self.X_host = self.X.cpu().pin_memory()
        self.Y_host = torch.empty(M * h, dtype=bf).pin_memory()

    def step(self):
        w = self.w
        self.t.check(self.t.tp3d_mlp(self.ctx, w["q"], w["M"], w["h"], w["f"], self.t.TP3D_BF16, self.X, self.W1,
                                     self.b1, self.W2, self.b2, self.Y1, self.Y), "tp3d_mlp")

    def e2e_step(self):
        self.X.copy_(self.X_host, non_blocking=True)
        self.step()
        self.Y_host.copy_(self.Y, non_blocking=True)

    def e2e_bytes(self):
        return self.X.numel() * 2, self.Y.numel() * 2, "X copied from pinned host memory, tp3d_mlp, Y copied back"

    def kernel_probe(self):
        w = self.w
        if self.launches == 1:  # the whole block is the one kernel
            fl = 4.0 * w["M"] * w["h"] * w["f"]
            return self.step, fl, (f"gemm_chain_kernel (the MLP block as one persistent launch of CTA pairs: "
                                   f"linear 1 + bias + GELU feeding linear 2 + bias, second contraction in "
                                   f"{self.splits} part(s); M={w['M']}, h={w['h']}, f={w['f']}, q={w['q']}), "
                                   f"{fl / 1e9:.2f} GFLOP per launch")

        def launch():
            self.t.check(self.t.tp3d_linear(self.ctx, w["q"], 0, w["M"], w["h"], w["f"], self.t.TP3D_BF16, self.X,
                                            self.W1, self.b1, 1, self.Y1), "tp3d_linear")
        fl = 2.0 * w["M"] * w["h"] * w["f"]
        return launch, fl, (f"gemm_tc2_kernel (CTA-pair tcgen05 GEMM): 3-D linear 1 of the MLP (M={w['M']}, "
                            f"N={w['h']}, K={w['f']}, q={w['q']}, bias+GELU epilogue), {fl / 1e9:.2f} GFLOP per launch")


class LayerBench:
    """Config 3: tp3d_layer_fwd + tp3d_layer_bwd of the pre-LN GPT layer."""

    def __init__(self, t, ctx, dev, w, seed=20263):
        import torch
        self.t, self.ctx, self.w = t, ctx, w
        q, b, s, h, H, f = w["q"], w["batch"], w["seq"], w["hidden"], w["heads"], w["ffn"]
        M = b * s
        self.M, self.h, self.f, self.q = M, h, f, q
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        bf = torch.bfloat16
        shapes = {"w_qkv": h * 3 * h, "w_o": h * h, "w_1": h * f, "w_2": f * h}
        self.params = {k: _randn(torch, n, dev, g, 0.02) for k, n in shapes.items()}
        for k, n in (("b_qkv", 3 * h), ("b_o", h), ("b_1", f), ("b_2", h), ("ln1_b", h), ("ln2_b", h)):
            self.params[k] = torch.zeros(n, device=dev, dtype=bf)
        for k in ("ln1_g", "ln2_g"):
            self.params[k] = torch.ones(h, device=dev, dtype=bf)
        self.grads = {k: torch.empty_like(v) for k, v in self.params.items()}
        self.X = _randn(torch, M * h, dev, g)
        self.dY = _randn(torch, M * h, dev, g)
        self.Y = torch.empty(M * h, device=dev, dtype=bf)
        self.dX = torch.empty(M * h, device=dev, dtype=bf)
        self.cfg = t.tp3d_layer_cfg(q, b, s, h, H, f, t.TP3D_BF16, 1e-5)
        nb = t.tp3d_layer_workspace_bytes(self.cfg)
        if nb == 0:
            raise SystemExit("layer configuration rejected")
        self.ws = torch.empty(nb, device=dev, dtype=torch.uint8)
        d = h // H
        lin = 2.0 * M * (3 * h * h + h * h + 2 * h * f)
        att = 2.0 * (2.0 * s * s * d / 2) * b * H  # causal: the unmasked half of QK^T and PV
        self.fwd_flops = lin + att
        self.units = 3 * lin + 3 * att  # backward = twice the forward's products
        # library kernels per step: forward 7 (2 LN, 4 GEMM, attention);
        # backward 19 (8 GEMM, 3 attention, 2 LN rows, 2 LN column sums, 4
        # bias column sums; each column sum finishes its own reduction)
        self.launches = 9 + 19  # forward 9 (W_qkv max and fp16 copy, 2 LN, 4 GEMMs, attention), backward 19
        self.unit, self.scale = "TFLOP/s", 1e12
        self.X_host = self.X.cpu().pin_memory()
        self.dY_host = self.dY.cpu().pin_memory()
        self.dX_host = torch.empty(M * h, dtype=bf).pin_memory()

    def fwd(self):
        self.t.check(self.t.tp3d_layer_fwd(self.ctx, self.cfg, self.params, self.X, self.Y, self.ws), "tp3d_layer_fwd")

    def bwd(self):
        self.t.check(self.t.tp3d_layer_bwd(self.ctx, self.cfg, self.params, self.X, self.ws, self.dY, self.dX,
                                           self.grads), "tp3d_layer_bwd")

    def step(self):
        self.fwd()
        self.bwd()

    def e2e_step(self):
        import torch
        cur = torch.cuda.current_stream()
        if not hasattr(self, "copy_stream"):
            self.copy_stream = torch.cuda.Stream()
        # X first, alone on the host-to-device engine (the forward waits for it);
        # dY, needed only by the backward, then copies beside the forward
        self.X.copy_(self.X_host, non_blocking=True)
        self.copy_stream.wait_stream(cur)
        with torch.cuda.stream(self.copy_stream):
            self.dY.copy_(self.dY_host, non_blocking=True)
        self.fwd()
        cur.wait_stream(self.copy_stream)
        self.bwd()
        self.dX_host.copy_(self.dX, non_blocking=True)

    def e2e_bytes(self):
        return (2 * self.X.numel() * 2, self.dX.numel() * 2,
                "X then dY copied from pinned host memory (dY's copy beside the forward), tp3d_layer_fwd + "
                "tp3d_layer_bwd, dX copied back")

    def kernel_probe(self):
        """The layer's largest GEMM (MLP linear 1 with bias + GELU), same shape and epilogue."""
        import torch
        p = self.params
        Y1 = torch.empty(self.M * self.f, device=self.X.device, dtype=torch.bfloat16)

        def launch():
            self.t.check(self.t.tp3d_linear(self.ctx, self.q, 0, self.M, self.h, self.f, self.t.TP3D_BF16, self.X,
                                            p["w_1"], p["b_1"], 1, Y1), "tp3d_linear")
        fl = 2.0 * self.M * self.h * self.f
        return launch, fl, (f"gemm_tc2_kernel (CTA-pair tcgen05 GEMM): the layer's MLP linear 1 (M={self.M}, "
                            f"N={self.h}, K={self.f}, q={self.q}, bias+GELU epilogue) through tp3d_linear, "
                            f"{fl / 1e9:.2f} GFLOP per launch")


class LinearF32Bench:
    """Config 1: tp3d_linear in fp32 on the CUDA cores (latency-bound)."""

    def __init__(self, t, ctx, dev, w, seed=20261):
        import torch
        self.t, self.ctx, self.w = t, ctx, w
        M, N, K = w["M"], w["N"], w["K"]
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.A = torch.randn(M * N, device=dev, generator=g)
        self.B = torch.randn(N * K, device=dev, generator=g)
        self.C = torch.empty(M * K, device=dev)
        self.units = 2.0 * M * N * K
        self.launches = 1
        self.unit, self.scale = "GFLOP/s", 1e9

    def step(self):
        w = self.w
        self.t.check(self.t.tp3d_linear(self.ctx, w["q"], 0, w["M"], w["N"], w["K"], self.t.TP3D_F32, self.A, self.B,
                                        None, 0, self.C), "tp3d_linear f32")


class ReshardBench:
    def __init__(self, t, ctx, dev, w, seed=20265):
        import torch
        self.t, self.ctx = t, ctx
        R, C = w["R"], w["C"]
        self.R, self.C = R, C
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        L = t.layout
        if w.get("q3"):
            self.lays = [("CUBE_A", L(t.CUBE_A, 3), 1), ("CUBE_B", L(t.CUBE_B, 3), 1), ("CUBE_C", L(t.CUBE_C, 3), 1),
                         ("ROW3", L(t.ROW, 0, 3), 1), ("COL3", L(t.COL, 0, 3), 1), ("REP3", L(t.REPLICATED, 0, 3), 3)]
        else:
            self.lays = [("ROW4", L(t.ROW, 0, 4), 1), ("COL4", L(t.COL, 0, 4), 1),
                         ("BLK2x2", L(t.BLOCK2D, 0, 2, 2), 1), ("CUBE_A", L(t.CUBE_A, 2), 1),
                         ("REP4", L(t.REPLICATED, 0, 4), 4)]
        vals = torch.randint(-256, 257, (R * C,), device=dev, generator=g).to(torch.bfloat16)
        self.src = {}
        for name, lay, copies in self.lays:
            buf = torch.empty(R * C * copies, device=dev, dtype=torch.bfloat16)
            t.check(t.tp3d_reshard(ctx, R, C, 2, t.layout(t.ROW, 0, 1), vals, lay, buf), "reshard setup")
            self.src[name] = buf
        self.dst = {name: torch.empty_like(self.src[name]) for name, _, _ in self.lays}
        self.pairs = [(a, b) for a in self.lays for b in self.lays if a[0] != b[0]]
        # bytes moved: one full read (a replicated source is read once) + every destination copy written
        self.pair_bytes = [R * C * 2 * (1 + b[2]) for a, b in self.pairs]
        self.units = float(sum(self.pair_bytes))
        self.launches = len(self.pairs)
        self.unit, self.scale = "GB/s", 1e9

    def launch_pair(self, k):
        (an, al, _), (bn, bl, _) = self.pairs[k]
        self.t.check(self.t.tp3d_reshard(self.ctx, self.R, self.C, 2, al, self.src[an], bl, self.dst[bn]), "reshard")

    def step(self):
        for k in range(len(self.pairs)):
            self.launch_pair(k)


BENCHES = {"mlp": MlpBench, "layer": LayerBench, "linear_f32": LinearF32Bench, "reshard": ReshardBench}


def flush_l2(flush):
    """Flush L2 between timed steps: write 256 MiB (the first half of the
    buffer), then read the other 256 MiB, so that the write's dirty lines are
    written back here, outside the timed region, and not by the next step's
    kernels."""
    h = flush.numel() // 2
    flush[:h].add_(1)
    flush[h:].sum()


def time_steps(torch, fn, steps, warmup, flush, stream):
    """Per-step CUDA-event durations (ms), L2 flushed between steps (outside the events)."""
    for _ in range(warmup):
        fn()
        flush_l2(flush)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
        flush_l2(flush)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def capture(torch, fn, stream):
    """A CUDA graph of one call of fn (C-ABI launches on the current stream),
    for the timed loop to replay: the same kernels on the same buffers, without
    the host's per-launch work between them."""
    s = torch.cuda.Stream()
    s.wait_stream(stream)
    with torch.cuda.stream(s):
        fn()
    stream.wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def cpu_baseline_mlp(w, seconds):
    """The oracle (plain numpy fp64) on a bounded sample: the MLP is
    row-separable, so the sample is a block of rows run repeatedly."""
    import numpy as np
    from oracle import mlp as OM

    rng = np.random.default_rng(0)
    h, f = w["h"], w["f"]
    rows = min(w["M"], 512)
    X = rng.standard_normal((rows, h))
    W1 = 0.02 * rng.standard_normal((h, f))
    W2 = 0.02 * rng.standard_normal((f, h))
    b1, b2 = np.zeros(f), np.zeros(h)
    t0 = time.perf_counter()
    n = 0
    while True:
        OM.mlp_rows_dense(X, W1, b1, W2, b2)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or n >= 1000:
            break
    fl = 4.0 * rows * h * f * n
    return {"value": fl / el / 1e12, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{n} x MLP forward on {rows} of {w['M']} token rows (row-separable), float64 numpy, "
                      f"{el:.1f} s"}


def _oracle_layer_sample(w):
    import numpy as np
    from oracle import layer as OY

    cfg = OY.LayerConfig(p=w["q"], batch=1, seq=w["seq"], hidden=w["hidden"], heads=w["heads"], ffn=w["ffn"])
    rng = np.random.default_rng(0)
    h, f = cfg.hidden, cfg.ffn
    P = {k: 0.02 * rng.standard_normal(sh) for k, sh in OY.weight_shapes(cfg).items()}
    for k, n in (("b_qkv", 3 * h), ("b_o", h), ("b_1", f), ("b_2", h), ("ln1_b", h), ("ln2_b", h)):
        P[k] = np.zeros(n)
    P["ln1_g"], P["ln2_g"] = np.ones(h), np.ones(h)
    X = rng.standard_normal((cfg.M, h))
    dY = rng.standard_normal((cfg.M, h))

    def run():
        OY.layer_forward_dense(X, P, cfg)
        OY.layer_backward_dense(dY, X, P, cfg)
    return run, float(OY.layer_flops(cfg)["total"]), cfg


def cpu_baseline_layer(w, seconds):
    """The oracle's layer forward + backward on one of the batch's sequences
    (a bounded sample of the same workload), repeated up to the budget."""
    run, fl, cfg = _oracle_layer_sample(w)
    t0 = time.perf_counter()
    n = 0
    while True:
        run()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or n >= 100:
            break
    return {"value": fl * n / el / 1e12, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{n} x layer forward + backward on 1 of {w['batch']} sequences (seq {cfg.seq}), float64 "
                      f"numpy, {el:.1f} s (the oracle's backward recomputes its forward)"}


# DRAM bytes (read + write) of one launch of the layer's linear-1 probe, from
# an ncu capture (dram__bytes_read.sum + dram__bytes_write.sum) of that
# launch; valid only while the GEMM sources, byte for byte as written, hash
# to the value they had when it was taken (any edit voids it until the
# figure is captured again).
GEMM_TRAFFIC = {"workload": "layer_q2", "bytes": 50484736 + 27985408, "sources_sha256_16": "4d6e12f37d417884",
                "note": "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch; output lines still in "
                        "L2 when the kernel ends are not counted (reads equal the algorithmic inputs)"}
GEMM_SOURCES = ("gemm_tc.cu", "gemm.cuh", "common.cuh", "layout.cuh", "api.cu")


def gemm_sources_hash(read=None):
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        path = os.path.join("tensor_transformer_layer_cube_gb300", "csrc", f)
        if read is None:
            with open(os.path.join(ROOT, path), encoding="utf-8") as fh:
                text = fh.read()
        else:
            text = read(path)
        h.update(text.encode())
    return h.hexdigest()[:16]


def roofline_probe(torch, wb, steps, flush, stream, pk, workload=None):
    launch, fl, kname = wb.kernel_probe()
    kd = time_steps(torch, launch, max(10, steps), 3, flush, stream)
    ach = fl / (statistics.mean(kd) / 1e3) / 1e12
    traffic, tnote = None, "no ncu capture of the current kernel source for this workload"
    if workload == GEMM_TRAFFIC["workload"] and gemm_sources_hash() == GEMM_TRAFFIC["sources_sha256_16"]:
        traffic, tnote = GEMM_TRAFFIC["bytes"], GEMM_TRAFFIC["note"]
    return {"bound": "tensor", "achieved": ach, "peak": pk["bf16"], "unit": "TFLOP/s", "frac": ach / pk["bf16"],
            "traffic": traffic, "traffic_note": tnote, "kernel": kname,
            "peak_source": f"bf16_tflops ({pk['source']}, burst)", "launch_ms": statistics.mean(kd)}


def reshard_summary(torch, rb, flush, stream, pk, name="reshard", reps=5):
    per = []
    for k in range(len(rb.pairs)):
        d = time_steps(torch, lambda k=k: rb.launch_pair(k), reps, 2, flush, stream)
        per.append(statistics.median(d))
    gbs = [rb.pair_bytes[k] / (per[k] / 1e3) / 1e9 for k in range(len(per))]
    tot = rb.units / (sum(per) / 1e3) / 1e9
    # a plain device copy of the same 128 MiB (torch), the practical ceiling for one launch of this size
    a = torch.empty(rb.R * rb.C, device=flush.device, dtype=torch.bfloat16)
    b = torch.empty_like(a)
    cd = time_steps(torch, lambda: b.copy_(a), reps, 2, flush, stream)
    copy_gbs = 2 * a.numel() * 2 / (statistics.median(cd) / 1e3) / 1e9
    del a, b
    kern = ("reshard_vec_kernel" if not WORKLOADS[name].get("q3") else
            "reshard_staged_kernel (rows staged through shared memory by bulk copies and realigned)")
    return {
        "value": tot, "unit": "GB/s", "frac_of_measured_hbm": tot / pk["hbm"], "frac_of_8TBs": tot / 8000.0,
        "min_pair_gbs": min(gbs), "min_pair_frac": min(gbs) / pk["hbm"], "max_pair_gbs": max(gbs),
        "ms_per_sweep": sum(per), "torch_copy_same_bytes_gbs": copy_gbs,
        "pairs": {f"{rb.pairs[k][0][0]}->{rb.pairs[k][1][0]}": {"gbs": round(gbs[k], 1),
                                                                 "frac": round(gbs[k] / pk["hbm"], 4)}
                  for k in range(len(gbs))},
        "roofline": {"bound": "hbm", "achieved": tot, "peak": pk["hbm"], "unit": "GB/s", "frac": tot / pk["hbm"],
                     "traffic": None, "kernel": f"{kern} (sweep average; bytes = read once + every destination "
                                                "copy written)",
                     "peak_source": f"hbm_gbs ({pk['source']})"},
        "workload": WORKLOADS[name]["name"]}


def host_planner_summary(t):
    """The library's host-side planners, timed on the CPU: the cross-mesh
    resharding planner on a 8192 x 8192 bf16 activation handed from a
    (8, 16) mesh S1 R (16 row slices, each held on all 8 source hosts) to a
    (8, 16) mesh S01 R (16 devices per host), and the pipeline simulator on
    the printed bubble-table configurations.  The oracle's planner is timed
    beside it as the CPU baseline."""
    from oracle import cmr as OC
    from oracle import layouts as OL

    R = C = 8192
    _, src = t.tp3d_mesh_rects(R, C, t.tp3d_mesh_spec(8, 16, t.TP3D_SPEC_S1, t.TP3D_SPEC_R))
    _, dst = t.tp3d_mesh_rects(R, C, t.tp3d_mesh_spec(8, 16, t.TP3D_SPEC_S01, t.TP3D_SPEC_R))
    st, plan = t.tp3d_cmr_plan_create(R, C, 2, src, 0, dst, 128, 16)
    t.check(st, "tp3d_cmr_plan_create")
    out = {"instance": "8192 x 8192 bf16, (8, 16) S1 R on devices 0-127 -> (8, 16) S01 R on devices 128-255, "
                       "16 devices per host; durations in bytes at unit bandwidth",
           "tasks": t.tp3d_cmr_plan_num_tasks(plan), "lower_bound": t.tp3d_cmr_plan_lower_bound(plan)}
    algos = {"naive": (t.TP3D_CMR_NAIVE, {}), "load_balance": (t.TP3D_CMR_LOAD_BALANCE, {}),
             "random_greedy": (t.TP3D_CMR_RANDOM_GREEDY, {"trials": 16, "seed": 20260}),
             "dfs": (t.TP3D_CMR_DFS, {"node_limit": 200000})}
    for name, (algo, kw) in algos.items():
        reps, t0 = 0, time.perf_counter()
        while True:
            st, _, _, _, res = t.tp3d_cmr_schedule(plan, algo, **kw)
            t.check(st, "tp3d_cmr_schedule")
            reps += 1
            if time.perf_counter() - t0 > 0.2:
                break
        out[name] = {"makespan_over_lower_bound": res.makespan / out["lower_bound"],
                     "us_per_plan": (time.perf_counter() - t0) / reps * 1e6}
        if name == "dfs":
            out[name].update({"nodes": res.nodes, "complete": bool(res.complete)})
    t.tp3d_cmr_plan_destroy(plan)
    t0 = time.perf_counter()
    tasks = OC.make_tasks(OL.MeshSpec(8, 16, ("S1", "R")), OL.MeshSpec(8, 16, ("S01", "R")), R, C, 2, 0, 128, 16)
    OC.random_greedy(tasks, 16, 20260)
    out["cpu_baseline"] = {"kind": "oracle", "cores": 1, "what": "oracle unit tasks + randomised greedy, same "
                           "instance", "us_per_plan": (time.perf_counter() - t0) * 1e6}
    rows = []
    for sch, p, m, v in (("gpipe", 4, 8, 1), ("1f1b", 4, 8, 1), ("interleaved", 4, 8, 2), ("interleaved", 4, 8, 4),
                         ("1f1b", 8, 32, 1), ("interleaved", 8, 32, 4), ("gpipe", 16, 32, 1), ("1f1b", 16, 64, 1)):
        code = {"gpipe": t.TP3D_PIPE_GPIPE, "1f1b": t.TP3D_PIPE_1F1B, "interleaved": t.TP3D_PIPE_INTERLEAVED}[sch]
        t0 = time.perf_counter()
        st, res, _ = t.tp3d_pipeline_simulate(t.tp3d_pipe_cfg(code, p, m, v, 4, 8))
        t.check(st, "tp3d_pipeline_simulate")
        rows.append({"schedule": sch, "p": p, "m": m, "v": v, "bubble": res.bubble,
                     "closed_form": (p - 1) / (v * m), "us": (time.perf_counter() - t0) * 1e6})
    out["pipeline"] = rows
    return out


def layout_comparison(torch, t, ctx, dev, flush, stream):
    """The MLP block of the q = 4 workload (tokens 8192, hidden 4096, ffn
    16384; 64 virtual devices) in the three layouts that "Maximizing
    Parallelism in Distributed Training for Huge Neural Networks" compares:
    1-D Megatron (t = 64), 2-D SUMMA (8 x 8) and the 3-D cube (q = 4).  Time
    on this GPU, per-device memory and per-device communication (elements
    received or sent per forward, from each scheme's collectives), and the
    resharding of X between the schemes' input layouts."""
    M, h, f = 8192, 4096, 16384
    bf = torch.bfloat16
    g = torch.Generator(device=dev)
    g.manual_seed(20264)
    X = torch.randn(M * h, device=dev, generator=g).to(bf)
    W1 = (torch.randn(h * f, device=dev, generator=g) * 0.02).to(bf)
    W2 = (torch.randn(f * h, device=dev, generator=g) * 0.02).to(bf)
    b1 = torch.zeros(f, device=dev, dtype=bf)
    b2 = torch.zeros(h, device=dev, dtype=bf)
    Y1 = torch.empty(M * f, device=dev, dtype=bf)
    Y = torch.empty(M * h, device=dev, dtype=bf)
    fl = 4.0 * M * h * f
    out = {"workload": "MLP, tokens 8192, hidden 4096, ffn 16384, bf16, 64 virtual devices (values are layout "
                       "independent for timing: one buffer serves every layout)"}
    for name, scheme, p in (("1d_megatron_t64", t.TP3D_SCHEME_1D, 64), ("2d_summa_8x8", t.TP3D_SCHEME_2D, 8),
                            ("3d_cube_q4", t.TP3D_SCHEME_3D, 4)):
        def step(scheme=scheme, p=p):
            t.check(t.tp3d_mlp_layout(ctx, scheme, p, M, h, f, t.TP3D_BF16, X, W1, b1, W2, b2, Y1, Y),
                    "tp3d_mlp_layout")
        d = time_steps(torch, step, 10, 3, flush, stream)
        ms = statistics.mean(d)
        if scheme == t.TP3D_SCHEME_1D:
            mem = M * h + h * f // p + M * f // p + f * h // p + M * h
            comm = 2 * (p - 1) * M * h // p  # ring all-reduce of Y
        elif scheme == t.TP3D_SCHEME_2D:
            mem = (2 * M * h + 2 * h * f + M * f) // (p * p)
            # SUMMA: q steps, each receiving an A panel along the row and a B panel along the column
            comm = (p - 1) * ((M * h + h * f) + (M * f + f * h)) // (p * p)
        else:
            def lin(Mm, N, K):
                return (Mm // (p * p)) * (N // p) + (N // p) * (K // (p * p)) + (Mm // (p * p)) * (K // p)
            mem = lin(M, h, f) + lin(M, f, h) - (M // (p * p)) * (f // p)  # Y1 counted once
            # per linear: all-gather of A over y, of B over x, reduce-scatter of C over z,
            # each over q - 1 peers' shards
            comm = (p - 1) * (lin(M, h, f) + lin(M, f, h))
        out[name] = {"ms": ms, "tflops": fl / (ms / 1e3) / 1e12, "devices": p if scheme == 1 else p * p if scheme == 2
                     else p ** 3, "mem_elems_per_device": int(mem), "comm_elems_per_device": int(comm)}
    # resharding X (8192 x 4096 bf16) from the cube's layout to the other two
    for name, dst in (("x_cube_to_1d", t.layout(t.REPLICATED, 0, 1)), ("x_cube_to_2d", t.layout(t.BLOCK2D, 0, 8, 8))):
        Xd = torch.empty_like(X)

        def rs(dst=dst, Xd=Xd):
            t.check(t.tp3d_reshard(ctx, M, h, 2, t.layout(t.CUBE_A, 4), X, dst, Xd), "tp3d_reshard")
        d = time_steps(torch, rs, 10, 3, flush, stream)
        out[name] = {"ms": statistics.mean(d), "gbs": 2 * M * h * 2 / (statistics.mean(d) / 1e3) / 1e9}
    return out


def make_bench(t, ctx, dev, name):
    w = WORKLOADS[name]
    return BENCHES[w["kind"]](t, ctx, dev, w)


def slowest_rank_ms(total_ms, world, dist, device):
    """The job's timed total: every rank runs the same replica, so the job
    takes as long as its slowest rank (a MAX all-reduce over the ranks)."""
    if world <= 1 or dist is None:
        return total_ms
    import torch
    tt = torch.tensor([total_ms], device=device, dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_value(world, units, steps, total_ms, scale):
    """Whole-job throughput: the work of all ranks' steps over the slowest
    rank's time (units per second, divided by the metric's scale)."""
    return world * units * steps / (total_ms / 1e3) / scale


def run_ours(args, rank, world, dist):
    import torch

    import tensor_transformer_layer_cube_gb300 as t

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    ctx = t.tp3d_create(local)
    stream = torch.cuda.current_stream()
    flush = torch.zeros(512 * 1024 * 1024 // 4, device=dev, dtype=torch.float32)  # 256 MiB written + 256 MiB read
    w = WORKLOADS[args.workload]
    pk = peaks()
    wb = make_bench(t, ctx, dev, args.workload)
    if args.probe_only:
        launch, _, _ = wb.kernel_probe()
        for _ in range(3):
            launch()
        torch.cuda.synchronize()
        t.check(t.tp3d_sync_status(ctx), "probe")
        t.tp3d_destroy(ctx)
        return

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    use_graph = not args.no_graph and w["kind"] in ("layer", "mlp", "linear_f32")
    step_fn = wb.step
    if use_graph:
        for _ in range(args.warmup):  # one-time host work (attributes, occupancy) before the capture
            wb.step()
        torch.cuda.synchronize()
        graph = capture(torch, wb.step, stream)
        step_fn = graph.replay
    durs = time_steps(torch, step_fn, args.steps, args.warmup, flush, stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        dist.barrier()
    rows = sampler.stop() if rank == 0 else []
    st = t.tp3d_sync_status(ctx)
    if st != 0:
        raise SystemExit(f"device error after the timed region: {t.STATUS[st]}")
    total_ms = slowest_rank_ms(sum(durs), world, dist, dev)
    ms = total_ms / args.steps
    value = job_value(world, wb.units, args.steps, total_ms, wb.scale)

    line = {
        "metric": METRIC, "value": value, "unit": wb.unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w["kind"] != "linear_f32" else "f32",
        "data": "synthetic (seeded device RNG; N(0,1) inputs, N(0,0.02) weights)",
        "config": {"workload": w["name"], "l2": "flushed between timed steps outside the events: a 256 MiB write, "
                                                  "then a 256 MiB read that writes its dirty lines back",
                   "launch": "one CUDA graph per step (the step's C-ABI calls captured once, replayed)" if use_graph
                   else "direct C-ABI calls",
                   "parallelism": "replicas (no data-path collective)" if world > 1
                   else "single GPU, q^3 virtual devices in HBM"},
        "gpu_launches": wb.launches * args.steps,
    }
    if w["kind"] == "layer":
        ffn, bfn = wb.fwd, wb.bwd
        if use_graph:
            ffn, bfn = capture(torch, wb.fwd, stream).replay, capture(torch, wb.bwd, stream).replay
        fd = time_steps(torch, ffn, max(5, args.steps // 2), 2, flush, stream)
        bd = time_steps(torch, bfn, max(5, args.steps // 2), 2, flush, stream)
        fwd_ms = slowest_rank_ms(sum(fd), world, dist, dev) / len(fd)
        bwd_ms = slowest_rank_ms(sum(bd), world, dist, dev) / len(bd)
        line["layer"] = {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
                         "avg_step_time_ms_per_sequence": (fwd_ms + bwd_ms) / w["batch"],
                         "fwd_tflops": wb.fwd_flops / (fwd_ms / 1e3) / 1e12,
                         "bwd_tflops": (wb.units - wb.fwd_flops) / (bwd_ms / 1e3) / 1e12,
                         "flops_per_step": wb.units}
    if hasattr(wb, "e2e_step"):
        edurs = time_steps(torch, wb.e2e_step, max(3, args.steps // 2), 2, flush, stream)
        bi, bo, what = wb.e2e_bytes()
        e_ms = slowest_rank_ms(sum(edurs), world, dist, dev)
        line["e2e"] = {"value": job_value(world, wb.units, len(edurs), e_ms, wb.scale), "unit": wb.unit,
                       "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                       "ms_per_step": e_ms / len(edurs), "what": what + ", per step"}
    if hasattr(wb, "kernel_probe"):
        line["roofline"] = roofline_probe(torch, wb, args.steps, flush, stream, pk, args.workload)
    elif w["kind"] == "reshard":
        sweep = reshard_summary(torch, wb, flush, stream, pk, args.workload)
        line["roofline"] = sweep["roofline"]
        line["sweep"] = sweep

    if rank == 0 and not args.no_extras:
        extras = {}
        for name in WORKLOADS:
            if name == args.workload:
                continue
            eb = make_bench(t, ctx, dev, name)
            if WORKLOADS[name]["kind"] == "reshard":
                extras[name] = reshard_summary(torch, eb, flush, stream, pk, name)
            else:
                d = time_steps(torch, eb.step, 10, 3, flush, stream)
                e = {"value": eb.units / (statistics.mean(d) / 1e3) / eb.scale, "unit": eb.unit,
                     "ms_per_step": statistics.mean(d), "workload": WORKLOADS[name]["name"]}
                if hasattr(eb, "kernel_probe"):
                    e["roofline"] = roofline_probe(torch, eb, 10, flush, stream, pk)
                    e["frac_of_bf16_peak"] = e["value"] / pk["bf16"]
                extras[name] = e
            del eb
            torch.cuda.empty_cache()
        host = host_planner_summary(t)
        layouts = layout_comparison(torch, t, ctx, dev, flush, stream)
        torch.cuda.empty_cache()
        st = t.tp3d_sync_status(ctx)
        if st != 0:
            raise SystemExit(f"device error in the extra workloads: {t.STATUS[st]}")
        # a compact resharding summary near the top of the line; the full
        # objects follow, with `configs` (every other workload) last
        line["reshard"] = {k: {"gbs": round(extras[k]["value"], 1), "frac": round(extras[k]["frac_of_measured_hbm"], 4),
                               "min_pair_frac": round(extras[k]["min_pair_frac"], 4),
                               "frac_of_8TBs": round(extras[k]["frac_of_8TBs"], 4)}
                           for k in extras if WORKLOADS[k]["kind"] == "reshard"}
    if rank == 0:
        line["clocks"] = ClockSampler.summarize(rows, t0, t1) if isinstance(rows, list) else rows
        if not args.no_extras and w["kind"] in ("mlp", "layer"):
            line["cpu_baseline"] = (cpu_baseline_layer if w["kind"] == "layer" else cpu_baseline_mlp)(
                w, args.cpu_seconds)
        if not args.no_extras:
            line["host_planners"] = host
            line["layout_comparison"] = layouts
            line["configs"] = extras
        print(json.dumps(line), flush=True)
    t.tp3d_destroy(ctx)


def run_reference(args, rank):
    """The reference arm: the fp64 oracle on the host cores, one bounded
    sample of the workload per step."""
    if rank != 0:
        return
    import numpy as np

    w = WORKLOADS[args.workload]
    cores = len(os.sched_getaffinity(0))
    if w["kind"] == "layer":
        run, fl, cfg = _oracle_layer_sample(w)
        sample = f"each step: layer forward + backward on 1 of {w['batch']} sequences (seq {cfg.seq}), float64 numpy"
    elif w["kind"] == "mlp":
        from oracle import mlp as OM
        rng = np.random.default_rng(0)
        h, f, rows = w["h"], w["f"], 256
        X = rng.standard_normal((rows, h))
        W1 = 0.02 * rng.standard_normal((h, f))
        W2 = 0.02 * rng.standard_normal((f, h))
        b1, b2 = np.zeros(f), np.zeros(h)

        def run():
            OM.mlp_rows_dense(X, W1, b1, W2, b2)
        fl = 4.0 * rows * h * f
        sample = f"each step: MLP forward on {rows} of {w['M']} token rows (row-separable), float64 numpy"
    else:
        print(json.dumps({"impl": "reference", "unavailable": f"no oracle arm for {args.workload}"}))
        return
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    v = fl * args.steps / el / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w["name"]},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    run_ours(args, rank, world, dist)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
