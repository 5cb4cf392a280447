"""Pipeline-bubble simulation, restated from "Transformer Training 11: Model
Parallelism" (pipeline parallelism section: the GPipe, 1F1B and interleaved
schedules, the closed forms T = (m + (p - 1)/v)(t_f + t_b) and bubble =
(p - 1)/(v m), and the table of simulated against closed-form bubbles).

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and bench.py's CPU
baseline may import this module; the library never does.

Every device runs its own list of operations in order; an operation starts
when the device is free and its input exists: the forward of micro-batch k on
virtual stage s needs the forward of k on stage s - 1, its backward needs the
backward of k on stage s + 1 (the last stage: its own forward).  Sends take
no time.  With v chunks per device, chunk c of device d is virtual stage
c * p + d and takes t_f / v forward, t_b / v backward.

Orders (from the schedules' published descriptions):
- GPipe (Huang et al. 2019): every forward, then every backward, micro-batches
  ascending.
- 1F1B (Narayanan et al. 2021, §2.2): device d first runs p - d - 1 forwards
  (at most m), then alternates one forward and one backward, then finishes
  the backwards.
- Interleaved 1F1B (same paper, §2.2): forwards go through the micro-batches
  in groups of p, each group through chunks 0 .. v-1; backwards the same
  groups through chunks v-1 .. 0.  Warm-up: 2 (p - d - 1) + (v - 1) p
  forwards (at most m v), then one forward / one backward, then the rest of
  the backwards.  Needs p | m.
"""
from __future__ import annotations


def device_program(schedule: str, p: int, m: int, v: int, d: int):
    """Operations of device d in order: (micro-batch, chunk, is_backward)."""
    if schedule == "gpipe":
        return [(k, 0, False) for k in range(m)] + [(k, 0, True) for k in range(m)]
    if schedule == "1f1b":
        w = min(p - d - 1, m)
        prog = [(k, 0, False) for k in range(w)]
        for k in range(m - w):
            prog += [(w + k, 0, False), (k, 0, True)]
        return prog + [(k, 0, True) for k in range(m - w, m)]
    if schedule == "interleaved":
        assert m % p == 0
        fwd, bwd = [], []
        for g in range(m // p):
            group = range(g * p, g * p + p)
            for c in range(v):
                fwd += [(k, c, False) for k in group]
            for c in reversed(range(v)):
                bwd += [(k, c, True) for k in group]
        w = min(2 * (p - d - 1) + (v - 1) * p, m * v)
        prog = fwd[:w]
        for k in range(m * v - w):
            prog += [fwd[w + k], bwd[k]]
        return prog + bwd[m * v - w:]
    raise ValueError(schedule)


def simulate(schedule: str, p: int, m: int, v: int, t_f: int, t_b: int):
    """Start and end time of every operation, by the definition: end(op) =
    max(end of the device's previous op, end of the op's input) + duration,
    evaluated on demand with an explicit stack."""
    assert t_f % v == 0 and t_b % v == 0
    progs = [device_program(schedule, p, m, v, d) for d in range(p)]
    where = {}  # (stage, micro-batch, backward) -> (device, position)
    for d in range(p):
        for pos, (k, c, b) in enumerate(progs[d]):
            where[(c * p + d, k, b)] = (d, pos)
    S = p * v
    end = {}

    def deps(d, pos):
        k, c, b = progs[d][pos]
        s = c * p + d
        out = [(d, pos - 1)] if pos > 0 else []
        if not b and s > 0:
            out.append(where[(s - 1, k, False)])
        if b:
            out.append(where[(s + 1, k, True)] if s < S - 1 else where[(s, k, False)])
        return out

    start = {}
    for d in range(p):
        for pos in range(len(progs[d])):
            stack = [(d, pos)]
            while stack:
                node = stack[-1]
                if node in end:
                    stack.pop()
                    continue
                todo = [x for x in deps(*node) if x not in end]
                if todo:
                    stack.extend(todo)
                    continue
                stack.pop()
                k, c, b = progs[node[0]][node[1]]
                st = max([end[x] for x in deps(*node)], default=0)
                start[node] = st
                end[node] = st + (t_b if b else t_f) // v
    ops = [(d, k, c, int(b), start[(d, pos)], end[(d, pos)])
           for d in range(p) for pos, (k, c, b) in enumerate(progs[d])]
    return ops


def bubble(schedule: str, p: int, m: int, v: int, t_f: int, t_b: int):
    """(makespan, bubble = idle / busy per device, most chunk activations
    held at once on a device)."""
    ops = simulate(schedule, p, m, v, t_f, t_b)
    makespan = max(o[5] for o in ops)
    busy = m * (t_f + t_b)
    held = 0
    for d in range(p):
        cur = 0
        for o in (o for o in ops if o[0] == d):
            cur += -1 if o[3] else 1
            held = max(held, cur)
    return makespan, (makespan - busy) / busy, held


def closed_form_bubble(p: int, m: int, v: int) -> float:
    """(p - 1) / (v m)."""
    return (p - 1) / (v * m)
