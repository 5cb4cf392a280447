"""Pins of the cross-mesh resharding planner oracle (oracle/cmr.py) to facts
outside itself: the worked example of "On Optimizing the Communication of
Model Parallelism" §2 (Figure 2), closed forms of simple instances, Graham's
bound for longest-processing-time-first list scheduling, an independent brute
force of the pure load-balance problem, the published SplitMix64 outputs,
and a validity checker of Eq. 2-3."""
import json
import os
import random

import pytest

from oracle import cmr as O
from oracle import layouts as L

HERE = os.path.dirname(os.path.abspath(__file__))


def _task(dur, src_hosts, dst_hosts):
    return {"slice": None, "dur": dur, "src_devs": list(src_hosts), "dst_devs": list(dst_hosts),
            "src_hosts": sorted(src_hosts), "dst_hosts": sorted(dst_hosts)}


def _all_schedules(tasks, seed=7):
    out = {"naive": O.naive(tasks), "load_balance": O.load_balance(tasks)}
    s, o, _ = O.random_greedy(tasks, 4, seed)
    out["random_greedy"] = (s, o)
    return out


def test_splitmix64_published_outputs():
    gold = json.load(open(os.path.join(HERE, "golden", "splitmix64_seed0.json")))
    got = [O.splitmix64_at(gold["seed"], k) for k in range(len(gold["outputs_hex"]))]
    assert got == [int(x, 16) for x in gold["outputs_hex"]]


def test_figure2_task1_schedules_take_two_slice_times():
    # four 1 x 4 row slices; devices 4, 5 need the top two, 6, 7 the bottom two:
    # each receiver takes two slices one after the other, and nothing forces more
    s0r = L.MeshSpec(2, 2, ("S0", "R"))
    tasks = O.make_tasks(L.ROW(4), s0r, 4, 4, 4, 0, 4, 1)
    T = 4 * 4
    assert [t["dur"] for t in tasks] == [T] * 4
    assert O.lower_bound(tasks) == 2 * T
    assert O.optimum(tasks) == 2 * T
    for name, (s, o) in _all_schedules(tasks).items():
        start, mk = O.list_schedule(tasks, o, s)
        assert O.check_schedule(tasks, s, start) == mk == 2 * T, name


def test_figure2_task2_two_disjoint_tasks_run_together():
    s0r = L.MeshSpec(2, 2, ("S0", "R"))
    tasks = O.make_tasks(s0r, L.ROW(4), 4, 4, 2, 4, 0, 1)
    assert [t["src_hosts"] for t in tasks] == [[4, 5], [6, 7]]
    assert [t["dst_hosts"] for t in tasks] == [[0, 1], [2, 3]]
    for name, (s, o) in _all_schedules(tasks).items():
        start, mk = O.list_schedule(tasks, o, s)
        assert O.check_schedule(tasks, s, start) == mk == 2 * 8, name


def test_one_receiver_serialises_everything():
    # every slice goes to the single destination device: the makespan is the sum
    tasks = O.make_tasks(L.BLOCK(2, 2), L.REP(1), 8, 8, 2, 0, 4, 1)
    total = 8 * 8 * 2
    assert sum(t["dur"] for t in tasks) == total
    assert O.optimum(tasks) == total
    for name, (s, o) in _all_schedules(tasks).items():
        assert O.list_schedule(tasks, o, s)[1] == total, name


def test_disjoint_hosts_run_in_parallel():
    tasks = O.make_tasks(L.ROW(4), L.ROW(4), 16, 8, 2, 0, 4, 1)
    for name, (s, o) in _all_schedules(tasks).items():
        assert O.list_schedule(tasks, o, s)[1] == 4 * 8 * 2, name


def test_host_grouping():
    # 8 source devices on hosts 0-1, 8 destination devices on hosts 2-3 (4 per host)
    tasks = O.make_tasks(L.ROW(8), L.COL(8), 16, 16, 2, 0, 8, 4)
    assert [t["src_hosts"] for t in tasks] == [[0]] * 4 + [[1]] * 4
    assert all(t["dst_hosts"] == [2, 3] and t["dst_devs"] == list(range(8, 16)) for t in tasks)


def _assign_brute_force(durs, m):
    """min over task -> host maps of the largest host load (P||Cmax)."""
    best = None
    n = len(durs)
    for code in range(m ** n):
        load = [0] * m
        c = code
        for d in durs:
            load[c % m] += d
            c //= m
        best = max(load) if best is None else min(best, max(load))
    return best


@pytest.mark.parametrize("seed", range(12))
def test_load_balance_within_grahams_bound(seed):
    # senders unrestricted, receivers all distinct: Eq. 1-3 reduce to P||Cmax,
    # LPT is within (4/3 - 1/(3m)) of the optimum (Graham 1969), and the
    # exhaustive optimum equals the brute force over assignments
    rng = random.Random(seed)
    m = rng.randint(2, 3)
    n = rng.randint(3, 5)
    durs = [rng.randint(1, 20) for _ in range(n)]
    tasks = [_task(d, range(m), [100 + i]) for i, d in enumerate(durs)]
    opt = _assign_brute_force(durs, m)
    assert O.optimum(tasks) == opt
    s, o = O.load_balance(tasks)
    start, mk = O.list_schedule(tasks, o, s)
    assert O.check_schedule(tasks, s, start) == mk
    assert opt <= mk <= (4 / 3 - 1 / (3 * m)) * opt + 1e-9
    assert O.lower_bound(tasks) <= opt


@pytest.mark.parametrize("n,m", [(5, 2), (6, 3), (4, 4), (7, 3)])
def test_equal_tasks_load_balance_is_optimal(n, m):
    T = 5
    tasks = [_task(T, range(m), [100 + i]) for i in range(n)]
    s, o = O.load_balance(tasks)
    mk = O.list_schedule(tasks, o, s)[1]
    assert mk == -(-n // m) * T == _assign_brute_force([T] * n, m)
    assert O.lower_bound(tasks) <= mk


@pytest.mark.parametrize("seed", range(8))
def test_optimum_bounds_every_schedule(seed):
    rng = random.Random(100 + seed)
    hosts_src, hosts_dst = list(range(3)), list(range(10, 14))
    tasks = []
    for _ in range(rng.randint(2, 5)):
        src = rng.sample(hosts_src, rng.randint(1, 2))
        dst = rng.sample(hosts_dst, rng.randint(1, 3))
        tasks.append(_task(rng.randint(1, 9), src, dst))
    opt = O.optimum(tasks)
    assert O.lower_bound(tasks) <= opt
    for name, (s, o) in _all_schedules(tasks, seed).items():
        start, mk = O.list_schedule(tasks, o, s)
        assert O.check_schedule(tasks, s, start) == mk >= opt, name


def test_random_greedy_rounds_are_disjoint_and_maximal():
    src = L.MeshSpec(2, 4, ("S0", "S1"))
    dst = L.MeshSpec(4, 2, ("S1", "S0"))
    tasks = O.make_tasks(src, dst, 64, 64, 2, 0, 8, 1)
    s, o, rounds = O.random_greedy(tasks, 5, 3)
    assert sorted(o) == list(range(len(tasks)))
    placed = set()
    for rnd in rounds:
        used = set()
        for t in rnd:
            hosts = {s[t]} | set(tasks[t]["dst_hosts"])
            assert not hosts & used
            used |= hosts
        for t in range(len(tasks)):
            if t in placed or t in rnd:
                continue
            # any task left for a later round conflicts with this round
            blocked = set(tasks[t]["dst_hosts"]) & used or set(tasks[t]["src_hosts"]) <= used
            assert blocked
        placed |= set(rnd)
    start, mk = O.list_schedule(tasks, o, s)
    assert O.check_schedule(tasks, s, start) == mk >= O.lower_bound(tasks)
    assert O.random_greedy(tasks, 5, 3)[1] == o  # deterministic in the seed


def test_check_schedule_rejects_overlap_and_wrong_sender():
    tasks = [_task(4, [0], [5]), _task(4, [1], [5])]
    with pytest.raises(AssertionError):
        O.check_schedule(tasks, [0, 1], [0, 2])     # both use receiver 5 during [2, 4)
    with pytest.raises(AssertionError):
        O.check_schedule(tasks, [1, 1], [0, 4])     # host 1 does not hold slice 0
    assert O.check_schedule(tasks, [0, 1], [0, 4]) == 8


def test_replicated_source_spreads_the_senders():
    # 8 row slices (S1 over the second axis of a (4, 8) mesh, replicated over
    # its first), 8 devices per host: every slice has one holder on each of
    # hosts 0-3.  The destination (4, 8) S01 R puts the receivers of slices
    # 2k and 2k+1 on host 4+k.  By hand:
    # - naive: host 0 sends all 8, one after the other: 8 T;
    # - load balance only: slice k from host k % 4 (2 T of sending each), but
    #   in plan order slices 4 and 5 wait for hosts 0 and 1 and slice 5 also
    #   for receiver host 6: it runs in [2T, 3T): 3 T;
    # - randomised greedy: rounds of 4 host-disjoint tasks, 2 rounds: 2 T,
    #   the receive-load bound.
    src = L.MeshSpec(4, 8, ("S1", "R"))
    dst = L.MeshSpec(4, 8, ("S01", "R"))
    tasks = O.make_tasks(src, dst, 64, 32, 2, 0, 32, 8)
    T = 8 * 32 * 2
    assert len(tasks) == 8 and all(t["dur"] == T and t["src_hosts"] == [0, 1, 2, 3] for t in tasks)
    assert [t["dst_hosts"] for t in tasks] == [[4 + k // 2] for k in range(8)]
    assert O.lower_bound(tasks) == 2 * T
    s, o = O.naive(tasks)
    assert O.list_schedule(tasks, o, s)[1] == 8 * T
    s, o = O.load_balance(tasks)
    assert s == [k % 4 for k in range(8)]
    assert O.list_schedule(tasks, o, s)[1] == 3 * T
    s, o, rounds = O.random_greedy(tasks, 4, 11)
    start, mk = O.list_schedule(tasks, o, s)
    assert O.check_schedule(tasks, s, start) == mk == 2 * T and len(rounds) == 2
