"""Parity of the library's host-side planners (include/tp3d_plan.h) with the
oracle: layout rectangles, cross-mesh resharding unit tasks and schedules
("On Optimizing the Communication of Model Parallelism" §2 and §3.2) and the
pipeline-bubble simulator ("Transformer Training 11: Model Parallelism").

These entry points are plain host code: they run here, without a GPU.  All
outputs are integers (rectangles, devices, hosts, orders, byte-time units)
and must match exactly; where several schedules are optimal (the depth-first
search) the optimum's makespan is compared and the schedule checked for
validity."""
import itertools
import json
import os

import pytest

import tensor_transformer_layer_cube_gb300 as t
from oracle import cmr as OC
from oracle import layouts as L
from oracle import pipeline as OP

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    t.build()
    t.lib()


def _rects(layout_obj, R, C):
    return [(rs.start, rs.stop - rs.start, cs.start, cs.stop - cs.start) for rs, cs in layout_obj.slices(R, C)]


LAYOUTS = {
    "CUBE_A": (lambda q: t.layout(t.CUBE_A, q), L.CUBE_A),
    "CUBE_B": (lambda q: t.layout(t.CUBE_B, q), L.CUBE_B),
    "CUBE_C": (lambda q: t.layout(t.CUBE_C, q), L.CUBE_C),
    "CUBE_B_SWAP": (lambda q: t.layout(t.CUBE_B_SWAP, q), L.CUBE_B_SWAP),
}


@pytest.mark.parametrize("name", sorted(LAYOUTS))
@pytest.mark.parametrize("q", [1, 2, 3])
def test_cube_rects(name, q):
    R, C = 36 * q * q, 12 * q * q
    st, got = t.tp3d_layout_rects(R, C, LAYOUTS[name][0](q))
    assert st == 0
    assert got == _rects(LAYOUTS[name][1](q), R, C)


@pytest.mark.parametrize("lib_l,orc", [
    (t.layout(t.ROW, 0, 4), L.ROW(4)), (t.layout(t.COL, 0, 3), L.COL(3)),
    (t.layout(t.BLOCK2D, 0, 2, 3), L.BLOCK(2, 3)), (t.layout(t.REPLICATED, 0, 3), L.REP(3))])
def test_mesh_layout_rects(lib_l, orc):
    st, got = t.tp3d_layout_rects(24, 36, lib_l)
    assert st == 0 and got == _rects(orc, 24, 36)


SPECS = {"R": t.TP3D_SPEC_R, "S0": t.TP3D_SPEC_S0, "S1": t.TP3D_SPEC_S1, "S01": t.TP3D_SPEC_S01}


@pytest.mark.parametrize("m1,m2", [(2, 2), (2, 4), (1, 4), (3, 1)])
def test_mesh_spec_rects(m1, m2):
    R, C = 48, 24
    for rs, cs in itertools.product(SPECS, SPECS):
        axes = {"R": set(), "S0": {0}, "S1": {1}, "S01": {0, 1}}
        st, got = t.tp3d_mesh_rects(R, C, t.tp3d_mesh_spec(m1, m2, SPECS[rs], SPECS[cs]))
        if axes[rs] & axes[cs]:
            assert st == 1, (rs, cs)
            continue
        assert st == 0, (rs, cs)
        assert got == _rects(L.MeshSpec(m1, m2, (rs, cs)), R, C), (rs, cs)


def _lib_layout(kind):
    kinds = {
        "ROW4": (t.layout(t.ROW, 0, 4), L.ROW(4)),
        "COL4": (t.layout(t.COL, 0, 4), L.COL(4)),
        "BLK2x2": (t.layout(t.BLOCK2D, 0, 2, 2), L.BLOCK(2, 2)),
        "CUBE_A2": (t.layout(t.CUBE_A, 2), L.CUBE_A(2)),
        "REP4": (t.layout(t.REPLICATED, 0, 4), L.REP(4)),
    }
    return kinds[kind]


def _mesh(m1, m2, rs, cs):
    return t.tp3d_mesh_spec(m1, m2, SPECS[rs], SPECS[cs]), L.MeshSpec(m1, m2, (rs, cs))


def _side(spec, R, C):
    lib_spec, orc = spec
    fn = t.tp3d_mesh_rects if isinstance(lib_spec, t.tp3d_mesh_spec) else t.tp3d_layout_rects
    st, rects = fn(R, C, lib_spec)
    assert st == 0
    return rects, orc


def _plan(src, dst, R, C, esz, src_first, dst_first, dph):
    (sr, so), (dr, do) = _side(src, R, C), _side(dst, R, C)
    st, plan = t.tp3d_cmr_plan_create(R, C, esz, sr, src_first, dr, dst_first, dph)
    assert st == 0, t.STATUS[st]
    tasks = OC.make_tasks(so, do, R, C, esz, src_first, dst_first, dph)
    return plan, tasks, len(sr), len(dr)


def _compare_plan(plan, tasks, ns, nd):
    assert t.tp3d_cmr_plan_num_tasks(plan) == len(tasks)
    for i, want in enumerate(tasks):
        st, sl, dur, snd, rcv = t.tp3d_cmr_plan_task(plan, i, ns, nd)
        assert st == 0
        assert sl == want["slice"] and dur == want["dur"]
        assert snd == want["src_devs"] and rcv == want["dst_devs"]
    assert t.tp3d_cmr_plan_lower_bound(plan) == OC.lower_bound(tasks)


def _compare_schedules(plan, tasks, seeds=(0, 1, 20260), trials=(1, 3, 8)):
    st, s, o, start, res = t.tp3d_cmr_schedule(plan, t.TP3D_CMR_NAIVE)
    ws, wo = OC.naive(tasks)
    assert st == 0 and (s, o) == (ws, wo)
    wstart, wmk = OC.list_schedule(tasks, wo, ws)
    assert start == wstart and res.makespan == wmk
    st, s, o, start, res = t.tp3d_cmr_schedule(plan, t.TP3D_CMR_LOAD_BALANCE)
    ws, wo = OC.load_balance(tasks)
    assert st == 0 and (s, o) == (ws, wo)
    wstart, wmk = OC.list_schedule(tasks, wo, ws)
    assert start == wstart and res.makespan == wmk
    for seed in seeds:
        for tr in trials:
            st, s, o, start, res = t.tp3d_cmr_schedule(plan, t.TP3D_CMR_RANDOM_GREEDY, trials=tr, seed=seed)
            ws, wo, rounds = OC.random_greedy(tasks, tr, seed)
            assert st == 0 and (s, o) == (ws, wo), (seed, tr)
            wstart, wmk = OC.list_schedule(tasks, wo, ws)
            assert start == wstart and res.makespan == wmk and res.rounds == len(rounds)
            assert OC.check_schedule(tasks, s, start) == wmk


PAIRS = list(itertools.permutations(["ROW4", "COL4", "BLK2x2", "CUBE_A2", "REP4"], 2))


@pytest.mark.parametrize("a,b", PAIRS, ids=[f"{a}->{b}" for a, b in PAIRS])
@pytest.mark.parametrize("dph", [1, 2, 4])
def test_reshard_pairs_plan_and_schedules(a, b, dph):
    nsrc = 8 if a == "CUBE_A2" else 4
    dst_first = -(-nsrc // dph) * dph  # first device of the next host
    plan, tasks, ns, nd = _plan(_lib_layout(a), _lib_layout(b), 64, 64, 2, 0, dst_first, dph)
    try:
        _compare_plan(plan, tasks, ns, nd)
        _compare_schedules(plan, tasks)
    finally:
        t.tp3d_cmr_plan_destroy(plan)


def test_figure2_plans():
    src = (t.layout(t.ROW, 0, 4), L.ROW(4))
    dst = _mesh(2, 2, "S0", "R")
    plan, tasks, ns, nd = _plan(src, dst, 4, 4, 4, 0, 4, 1)
    try:
        _compare_plan(plan, tasks, ns, nd)
        _compare_schedules(plan, tasks)
        st, _, _, _, res = t.tp3d_cmr_schedule(plan, t.TP3D_CMR_DFS, node_limit=10 ** 6)
        assert st == 0 and res.complete == 1 and res.makespan == OC.optimum(tasks) == 32
    finally:
        t.tp3d_cmr_plan_destroy(plan)


def test_large_replicated_mesh_plan():
    # a 64 x 2048 activation (bf16) from a (4, 8) mesh S0 R - replicated over
    # 8 devices per host - to an (8, 4) mesh S1 S0, 8 devices per host
    src, dst = _mesh(4, 8, "S0", "R"), _mesh(8, 4, "S1", "S0")
    plan, tasks, ns, nd = _plan(src, dst, 64, 2048, 2, 0, 32, 8)
    try:
        _compare_plan(plan, tasks, ns, nd)
        _compare_schedules(plan, tasks, seeds=(5,), trials=(4,))
    finally:
        t.tp3d_cmr_plan_destroy(plan)


def test_many_tasks_with_replicated_holders():
    # (2, 8) mesh R S1 (8 unique column slices, 2 holders each, 4 devices per
    # host) to a (4, 4) mesh S0 S1: 8 tasks over 4 source hosts, 16 receivers
    src, dst = _mesh(2, 8, "R", "S1"), _mesh(4, 4, "S0", "S1")
    plan, tasks, ns, nd = _plan(src, dst, 32, 64, 4, 0, 16, 4)
    try:
        _compare_plan(plan, tasks, ns, nd)
        _compare_schedules(plan, tasks)
    finally:
        t.tp3d_cmr_plan_destroy(plan)


@pytest.mark.parametrize("case", [
    ((2, 2, "S0", "R"), (1, 2, "R", "S01"), 1),
    ((2, 2, "R", "S0"), (2, 1, "S0", "R"), 1),
    ((1, 4, "R", "R"), (2, 2, "S0", "S1"), 2),
    ((2, 2, "S01", "R"), (1, 3, "R", "S1"), 1),
])
def test_dfs_reaches_the_optimum(case):
    (a1, a2, ar, ac), (b1, b2, br, bc), dph = case
    src, dst = _mesh(a1, a2, ar, ac), _mesh(b1, b2, br, bc)
    nsrc = a1 * a2
    dst_first = -(-nsrc // dph) * dph
    plan, tasks, ns, nd = _plan(src, dst, 12, 12, 2, 0, dst_first, dph)
    try:
        assert len(tasks) <= 6
        st, s, o, start, res = t.tp3d_cmr_schedule(plan, t.TP3D_CMR_DFS, node_limit=10 ** 7)
        assert st == 0 and res.complete == 1
        assert res.makespan == OC.optimum(tasks)
        assert OC.check_schedule(tasks, s, start) == res.makespan
        assert sorted(o) == list(range(len(tasks)))
    finally:
        t.tp3d_cmr_plan_destroy(plan)


def test_dfs_node_limit_returns_a_valid_schedule():
    src, dst = _mesh(2, 8, "R", "S1"), _mesh(4, 4, "S0", "S1")
    plan, tasks, ns, nd = _plan(src, dst, 32, 64, 4, 0, 16, 4)
    try:
        st, s, o, start, res = t.tp3d_cmr_schedule(plan, t.TP3D_CMR_DFS, node_limit=50)
        assert st == 0 and res.nodes <= 50
        assert OC.check_schedule(tasks, s, start) == res.makespan
        ns_, no = OC.naive(tasks)
        ls, lo = OC.load_balance(tasks)
        assert res.makespan <= min(OC.list_schedule(tasks, no, ns_)[1], OC.list_schedule(tasks, lo, ls)[1])
    finally:
        t.tp3d_cmr_plan_destroy(plan)


def test_plan_errors():
    _, row = t.tp3d_layout_rects(8, 8, t.layout(t.ROW, 0, 4))
    _, col = t.tp3d_layout_rects(8, 8, t.layout(t.COL, 0, 4))
    assert t.tp3d_cmr_plan_create(8, 8, 2, row, 0, col, 2, 1)[0] == 8          # device ranges overlap
    assert t.tp3d_cmr_plan_create(8, 8, 2, row, 0, col, 4, 8)[0] == 1          # one host holds both meshes
    assert t.tp3d_cmr_plan_create(8, 8, 0, row, 0, col, 4, 1)[0] == 1          # element size
    bad = list(row)
    bad[1] = (0, 2, 0, 8)                                                       # rows 2-3 never held
    assert t.tp3d_cmr_plan_create(8, 8, 2, bad, 0, col, 4, 1)[0] == 2
    bad[1] = (1, 2, 0, 8)                                                       # overlapping slices
    assert t.tp3d_cmr_plan_create(8, 8, 2, bad, 0, col, 4, 1)[0] == 2
    assert t.tp3d_cmr_plan_create(8, 8, 2, row, 0, [(0, 9, 0, 8)], 4, 1)[0] == 2  # leaves the matrix
    st, plan = t.tp3d_cmr_plan_create(8, 8, 2, row, 0, col, 4, 1)
    assert st == 0
    try:
        assert t.tp3d_cmr_schedule(plan, 9)[0] == 1
        assert t.tp3d_cmr_schedule(plan, t.TP3D_CMR_RANDOM_GREEDY, trials=0)[0] == 1
        assert t.tp3d_cmr_schedule(plan, t.TP3D_CMR_DFS, node_limit=0)[0] == 1
        assert t.tp3d_cmr_plan_task(plan, 4, 4, 4)[0] == 1
    finally:
        t.tp3d_cmr_plan_destroy(plan)
    assert t.tp3d_layout_rects(6, 8, t.layout(t.ROW, 0, 4))[0] == 2
    assert t.tp3d_mesh_rects(8, 8, t.tp3d_mesh_spec(3, 1, t.TP3D_SPEC_S0, t.TP3D_SPEC_R))[0] == 2


# ---------------------------------------------------------------------------
# pipeline-bubble simulator
# ---------------------------------------------------------------------------

SCHED = {"gpipe": t.TP3D_PIPE_GPIPE, "1f1b": t.TP3D_PIPE_1F1B, "interleaved": t.TP3D_PIPE_INTERLEAVED}


def _pipe_cases():
    for p in (1, 2, 3, 4, 5):
        for m in (1, 3, 4, 8, 10):
            yield "gpipe", p, m, 1
            yield "1f1b", p, m, 1
            if m % p == 0:
                for v in (1, 2, 3):
                    yield "interleaved", p, m, v


@pytest.mark.parametrize("t_f,t_b", [(6, 12), (6, 6), (12, 18)])
def test_pipeline_matches_oracle(t_f, t_b):
    for sch, p, m, v in _pipe_cases():
        st, res, ops = t.tp3d_pipeline_simulate(t.tp3d_pipe_cfg(SCHED[sch], p, m, v, t_f, t_b), want_ops=True)
        assert st == 0, (sch, p, m, v)
        want = OP.simulate(sch, p, m, v, t_f, t_b)
        got = [(o.device, o.microbatch, o.chunk, o.backward, o.start, o.end) for o in ops]
        assert got == want, (sch, p, m, v)
        mk, b, held = OP.bubble(sch, p, m, v, t_f, t_b)
        assert (res.makespan, res.max_in_flight) == (mk, held)
        assert res.busy == m * (t_f + t_b) and res.idle == p * (mk - res.busy)
        assert res.bubble == pytest.approx(b, abs=1e-15)


def test_pipeline_printed_table():
    gold = json.load(open(os.path.join(HERE, "golden", "pipeline_bubble_table.json")))
    for row in gold["rows"]:
        st, res, _ = t.tp3d_pipeline_simulate(
            t.tp3d_pipe_cfg(SCHED[row["schedule"]], row["p"], row["m"], row["v"], 4, 8))
        assert st == 0
        assert round(res.bubble, gold["printed_digits"]) == pytest.approx(row["simulated"], abs=1e-12)


def test_pipeline_errors():
    sim = lambda *a: t.tp3d_pipeline_simulate(t.tp3d_pipe_cfg(*a))[0]  # noqa: E731
    assert sim(t.TP3D_PIPE_1F1B, 4, 8, 2, 4, 8) == 1        # chunks outside the interleaved schedule
    assert sim(t.TP3D_PIPE_INTERLEAVED, 4, 6, 2, 4, 8) == 2  # p does not divide m
    assert sim(t.TP3D_PIPE_INTERLEAVED, 4, 8, 3, 4, 9) == 2  # v does not divide t_f
    assert sim(7, 4, 8, 1, 4, 8) == 1
    assert sim(t.TP3D_PIPE_GPIPE, 0, 8, 1, 4, 8) == 1
    assert sim(t.TP3D_PIPE_GPIPE, 4, 8, 1, 0, 8) == 1


def test_replicated_source_plan():
    src, dst = _mesh(4, 8, "S1", "R"), _mesh(4, 8, "S01", "R")
    plan, tasks, ns, nd = _plan(src, dst, 64, 32, 2, 0, 32, 8)
    try:
        _compare_plan(plan, tasks, ns, nd)
        _compare_schedules(plan, tasks)
        st, s, o, start, res = t.tp3d_cmr_schedule(plan, t.TP3D_CMR_DFS, node_limit=10 ** 5)
        assert st == 0 and res.makespan == t.tp3d_cmr_plan_lower_bound(plan) == 2 * 8 * 32 * 2
    finally:
        t.tp3d_cmr_plan_destroy(plan)
