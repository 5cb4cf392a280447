#!/usr/bin/env python
"""Benchmark of the 3-D tensor-parallel layer cube on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload layer_q2|mlp_q2|mlp_q4|reshard]

Prints ONE JSON line (rank 0).  A step is one pass of the workload's whole
hot path over one batch of synthetic input already resident in HBM; every
timed step is bracketed by CUDA events on the launching stream and followed,
outside the events, by a 256 MiB write that flushes L2.  `value` is the
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
DEFAULT_WORKLOAD = "mlp_q2"

WORKLOADS = {
    "mlp_q2": dict(kind="mlp", q=2, M=2048, h=1024, f=4096,
                   name="Megatron MLP (column-split Linear+GELU, row-split Linear) on a q=2 cube: "
                        "tokens 2048, hidden 1024, ffn 4096, bf16"),
    "mlp_q4": dict(kind="mlp", q=4, M=8192, h=4096, f=16384,
                   name="MLP on a q=4 cube (64 virtual devices): tokens 8192, hidden 4096, ffn 16384, bf16"),
    "layer_q2": dict(kind="layer", q=2, batch=4, seq=1024, hidden=2048, heads=16, ffn=8192,
                     name="GPT decoder layer fwd+bwd on a q=2 cube: batch 4, seq 1024, hidden 2048, "
                          "16 heads, ffn 8192, bf16"),
    "reshard": dict(kind="reshard", R=8192, C=8192,
                    name="resharding sweep, 8192x8192 bf16, 20 ordered pairs of ROW4 COL4 BLK2x2 CUBE_A(q=2) REP4"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU baseline sample budget")
    ap.add_argument("--no-extras", action="store_true", help="skip the reshard sweep and the CPU baseline")
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
class MlpBench:
    def __init__(self, t, ctx, dev, w, seed=20262):
        import torch
        self.t, self.ctx, self.w = t, ctx, w
        q, M, h, f = w["q"], w["M"], w["h"], w["f"]
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        bf = torch.bfloat16
        self.X = torch.randn(M * h, device=dev, generator=g).to(bf)
        self.W1 = (torch.randn(h * f, device=dev, generator=g) * 0.02).to(bf)
        self.W2 = (torch.randn(f * h, device=dev, generator=g) * 0.02).to(bf)
        self.b1 = torch.zeros(f, device=dev, dtype=bf)
        self.b2 = torch.zeros(h, device=dev, dtype=bf)
        self.Y1 = torch.empty(M * f, device=dev, dtype=bf)
        self.Y = torch.empty(M * h, device=dev, dtype=bf)
        self.flops = 4.0 * M * h * f
        self.launches = 2
        self.unit = "TFLOP/s"
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
        return self.X.numel() * 2, self.Y.numel() * 2

    def kernel_probe(self):
        """(launch callable, algorithmic FLOPs per launch, name) of the dominant kernel."""
        w = self.w
        def launch():
            self.t.check(self.t.tp3d_linear(self.ctx, w["q"], 0, w["M"], w["h"], w["f"], self.t.TP3D_BF16, self.X,
                                            self.W1, self.b1, 1, self.Y1), "tp3d_linear")
        return launch, 2.0 * w["M"] * w["h"] * w["f"], (
            f"gemm_tc_kernel: 3-D linear 1 of the MLP (M={w['M']}, N={w['h']}, K={w['f']}, q={w['q']}, "
            f"bias+GELU epilogue), {2.0 * w['M'] * w['h'] * w['f'] / 1e9:.2f} GFLOP per launch")


class ReshardBench:
    def __init__(self, t, ctx, dev, w, seed=20265):
        import torch
        self.t, self.ctx = t, ctx
        R, C = w["R"], w["C"]
        self.R, self.C = R, C
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        L = t.layout
        self.lays = [("ROW4", L(t.ROW, 0, 4), 1), ("COL4", L(t.COL, 0, 4), 1), ("BLK2x2", L(t.BLOCK2D, 0, 2, 2), 1),
                     ("CUBE_A", L(t.CUBE_A, 2), 1), ("REP4", L(t.REPLICATED, 0, 4), 4)]
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
        self.bytes = float(sum(self.pair_bytes))
        self.launches = len(self.pairs)
        self.unit = "GB/s"

    def launch_pair(self, k):
        (an, al, _), (bn, bl, _) = self.pairs[k]
        self.t.check(self.t.tp3d_reshard(self.ctx, self.R, self.C, 2, al, self.src[an], bl, self.dst[bn]), "reshard")

    def step(self):
        for k in range(len(self.pairs)):
            self.launch_pair(k)


def time_steps(torch, fn, steps, warmup, flush, stream):
    """Per-step CUDA-event durations (ms), L2 flushed between steps (outside the events)."""
    for _ in range(warmup):
        fn()
        flush.add_(1)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
        flush.add_(1)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


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
                      f"{el:.1f} s", "seconds": el}


def run_ours(args, rank, world, dist):
    import torch

    import tensor_transformer_layer_cube_gb300 as t

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    ctx = t.tp3d_create(local)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, device=dev, dtype=torch.float32)
    w = WORKLOADS[args.workload]
    pk = peaks()
    if w["kind"] == "mlp":
        wb = MlpBench(t, ctx, dev, w)
    elif w["kind"] == "reshard":
        wb = ReshardBench(t, ctx, dev, w)
    else:
        raise SystemExit(f"workload {args.workload} is not available yet")

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    durs = time_steps(torch, wb.step, args.steps, args.warmup, flush, stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        dist.barrier()
    rows = sampler.stop() if rank == 0 else []
    st = t.tp3d_sync_status(ctx)
    if st != 0:
        raise SystemExit(f"device error after the timed region: {t.STATUS[st]}")
    total_ms = sum(durs)
    if world > 1:
        tt = torch.tensor([total_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    ms = total_ms / args.steps
    units = wb.flops if w["kind"] != "reshard" else wb.bytes
    scale = 1e12 if w["kind"] != "reshard" else 1e9
    value = world * units * args.steps / (total_ms / 1e3) / scale

    # end to end through the public call with host buffers
    e2e = None
    if hasattr(wb, "e2e_step"):
        edurs = time_steps(torch, wb.e2e_step, max(3, args.steps // 2), 2, flush, stream)
        bi, bo = wb.e2e_bytes()
        e2e = {"value": units / (statistics.mean(edurs) / 1e3) / scale * world, "unit": wb.unit,
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "ms_per_step": statistics.mean(edurs),
               "what": "X copied from pinned host memory, tp3d_mlp, Y copied back, per step"}

    # roofline of the dominant kernel, timed live
    roof = None
    if w["kind"] == "mlp":
        launch, fl, kname = wb.kernel_probe()
        kd = time_steps(torch, launch, max(10, args.steps), 3, flush, stream)
        ach = fl / (statistics.mean(kd) / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": pk["bf16"], "unit": "TFLOP/s", "frac": ach / pk["bf16"],
                "traffic": None, "kernel": kname, "peak_source": f"bf16_tflops ({pk['source']}, burst)",
                "launch_ms": statistics.mean(kd)}

    extras = {}
    if rank == 0 and not args.no_extras and w["kind"] != "reshard":
        rb = ReshardBench(t, ctx, dev, WORKLOADS["reshard"])
        per = []
        for k in range(len(rb.pairs)):
            d = time_steps(torch, lambda k=k: rb.launch_pair(k), 5, 2, flush, stream)
            per.append(statistics.median(d))
        gbs = [rb.pair_bytes[k] / (per[k] / 1e3) / 1e9 for k in range(len(per))]
        tot = rb.bytes / (sum(per) / 1e3) / 1e9
        extras["reshard"] = {
            "value": tot, "unit": "GB/s", "frac_of_measured_hbm": tot / pk["hbm"], "frac_of_8TBs": tot / 8000.0,
            "min_pair_gbs": min(gbs), "max_pair_gbs": max(gbs),
            "pairs": {f"{rb.pairs[k][0][0]}->{rb.pairs[k][1][0]}": round(gbs[k], 1) for k in range(len(gbs))},
            "workload": WORKLOADS["reshard"]["name"], "kernel": "reshard_vec_kernel",
            "bytes_convention": "read once + every destination copy written"}
        del rb

    line = {
        "metric": METRIC, "value": value, "unit": wb.unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded device RNG; N(0,1) inputs, N(0,0.02) weights)",
        "config": {"workload": w["name"], "l2": "flushed between timed steps (256 MiB write outside the events)",
                   "parallelism": "replicas" if world > 1 else "single GPU, q^3 virtual devices in HBM"},
        "gpu_launches": wb.launches * args.steps,
    }
    if e2e:
        line["e2e"] = e2e
    if roof:
        line["roofline"] = roof
    line.update(extras)
    if rank == 0:
        line["clocks"] = ClockSampler.summarize(rows, t0, t1) if isinstance(rows, list) else rows
        if not args.no_extras and w["kind"] == "mlp":
            line["cpu_baseline"] = cpu_baseline_mlp(w, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    t.tp3d_destroy(ctx)


def run_reference(args, rank):
    if rank != 0:
        return
    import numpy as np
    from oracle import mlp as OM

    w = WORKLOADS[args.workload]
    if w["kind"] != "mlp":
        print(json.dumps({"impl": "reference", "unavailable": f"oracle arm for {args.workload} not built yet"}))
        return
    rng = np.random.default_rng(0)
    h, f = w["h"], w["f"]
    rows = 256
    X = rng.standard_normal((rows, h))
    W1 = 0.02 * rng.standard_normal((h, f))
    W2 = 0.02 * rng.standard_normal((f, h))
    b1, b2 = np.zeros(f), np.zeros(h)
    for _ in range(args.warmup):
        OM.mlp_rows_dense(X, W1, b1, W2, b2)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        OM.mlp_rows_dense(X, W1, b1, W2, b2)
    el = time.perf_counter() - t0
    fl = 4.0 * rows * h * f * args.steps
    v = fl / el / 1e12
    cores = len(os.sched_getaffinity(0))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w["name"]},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: MLP forward on {rows} of {w['M']} token rows (row-separable), "
                                   f"float64 numpy on the host cores"},
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
