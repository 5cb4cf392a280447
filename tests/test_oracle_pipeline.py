"""Pins of the pipeline-bubble oracle (oracle/pipeline.py): the table of
simulated against closed-form bubbles printed in "Transformer Training 11:
Model Parallelism" (pipeline parallelism section), the closed form
T = (m + (p - 1)/v)(t_f + t_b) itself, the page's statements on activation
memory, and the dependency rules of every simulated operation."""
import json
import os

import pytest

from oracle import pipeline as P

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "pipeline_bubble_table.json")))


@pytest.mark.parametrize("row", GOLD["rows"], ids=lambda r: f"{r['schedule']}-p{r['p']}-m{r['m']}-v{r['v']}")
def test_printed_table(row):
    v = row["v"]
    # forward 1 unit, backward 2 units per chunk, and the same scaled by v
    for t_f, t_b in ((v, 2 * v), (4, 8)):
        _, b, _ = P.bubble(row["schedule"], row["p"], row["m"], v, t_f, t_b)
        assert round(b, GOLD["printed_digits"]) == pytest.approx(row["simulated"], abs=1e-12)
        assert round(P.closed_form_bubble(row["p"], row["m"], v), 4) == pytest.approx(row["closed_form"])


def _grid():
    for p in (1, 2, 3, 4, 6):
        for m in (1, 2, 5, 8, 12):
            yield "gpipe", p, m, 1
            yield "1f1b", p, m, 1
            if m % p == 0:
                for v in (2, 3, 4):
                    yield "interleaved", p, m, v


@pytest.mark.parametrize("ratio", [1, 2, 3])
def test_closed_form_makespan(ratio):
    for sch, p, m, v in _grid():
        t_f = 12
        t_b = ratio * t_f
        mk, b, _ = P.bubble(sch, p, m, v, t_f, t_b)
        # T v = (m v + p - 1)(t_f + t_b)
        assert mk * v == (m * v + p - 1) * (t_f + t_b), (sch, p, m, v, ratio)
        assert b == pytest.approx((p - 1) / (v * m))


def test_single_device_has_no_bubble():
    for sch in ("gpipe", "1f1b"):
        mk, b, _ = P.bubble(sch, 1, 7, 1, 3, 5)
        assert mk == 7 * 8 and b == 0


def test_activation_memory():
    # GPipe holds every micro-batch's activations; 1F1B at most p of them
    for p, m in ((4, 8), (8, 32), (3, 2)):
        assert P.bubble("gpipe", p, m, 1, 1, 2)[2] == m
        assert P.bubble("1f1b", p, m, 1, 1, 2)[2] == min(p, m)


@pytest.mark.parametrize("sch,p,m,v", [("gpipe", 4, 6, 1), ("1f1b", 5, 7, 1), ("interleaved", 3, 6, 2),
                                       ("interleaved", 4, 8, 4)])
def test_every_operation_waits_for_its_input(sch, p, m, v):
    t_f, t_b = 4 * v, 8 * v
    ops = P.simulate(sch, p, m, v, t_f, t_b)
    assert len(ops) == 2 * p * m * v
    end = {}
    for d, k, c, b, st, en in ops:
        assert en - st == (t_b if b else t_f) // v
        end[(c * p + d, k, b)] = (st, en)
    S = p * v
    for (s, k, b), (st, en) in end.items():
        if not b and s > 0:
            assert st >= end[(s - 1, k, 0)][1]
        if b:
            assert st >= end[(s + 1, k, 1)][1] if s < S - 1 else st >= end[(s, k, 0)][1]
    for d in range(p):
        iv = sorted((o[4], o[5]) for o in ops if o[0] == d)
        assert all(a[1] <= b_[0] for a, b_ in zip(iv, iv[1:]))
