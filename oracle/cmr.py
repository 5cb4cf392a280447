"""Cross-mesh resharding planner, restated from "On Optimizing the
Communication of Model Parallelism" (arXiv 2211.05322).

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and bench.py's CPU
baseline may import this module; the library never does.

- Unit tasks (§2, 'Data slice' and 'Cross-mesh resharding'):
  ``layouts.unit_tasks`` gives one task per unique source slice DS_i, its
  holders N_i and the destination devices M_i whose slice overlaps it.
- Hosts (§3.2): balancing and scheduling work on hosts, host(d) =
  d // devices_per_host; n_i and m_i are the host sets of N_i and M_i.
- Duration T_i (reading): the slice's bytes, i.e. the time to send it once at
  unit bandwidth, which the pipelined broadcast of §3.1 approaches for many
  partitions.
- Eq. 1-3 (§3.2): choose n_i* in n_i and start times S_i so that tasks that
  share a sender or receiver host do not overlap; minimise max_i S_i + T_i.
  A schedule here is a sender per task plus a global order, start times
  following from the order by list scheduling (each task starts when the
  previous tasks on its hosts have ended) - the reduction stated in §3.2
  'Depth First Search (DFS) with Pruning'.
- Algorithms (§3.2): naive (lowest-indexed holder, one fixed order), load
  balance only (longest task first to the least-loaded holder host), the
  optimum the DFS searches for (here by exhaustive enumeration, for tiny
  instances), and greedy search with randomisation (rounds of mutually
  non-overlapping tasks, the largest of several random orders per round).

Readings where the page is silent: the size of a
round is the number of hosts it involves; a task joining a round is sent by
its free holder host with the least send load so far (ties: lowest host);
ties between equal candidate rounds keep the first trial; random orders sort
the remaining tasks by a SplitMix64 key of (seed, round, trial, task).
"""
from __future__ import annotations

import itertools

from . import layouts as L

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def splitmix64_at(seed: int, ctr: int) -> int:
    """Output number ``ctr`` (0-based) of SplitMix64 seeded with ``seed``
    (Steele, Lea and Flood, OOPSLA 2014): state seed + (ctr + 1) * gamma
    through the generator's mixing function."""
    z = (seed + (ctr + 1) * GAMMA) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def make_tasks(src, dst, R: int, C: int, elem_bytes: int, src_first: int, dst_first: int,
               devices_per_host: int):
    """Unit tasks with their hosts and durations, in first-holder order."""
    out = []
    for rs, cs, srcs, dsts in L.unit_tasks(src, dst, R, C, src_offset=src_first, dst_offset=dst_first):
        rows, cols = rs.stop - rs.start, cs.stop - cs.start
        out.append({
            "slice": (rs.start, rows, cs.start, cols),
            "dur": rows * cols * elem_bytes,
            "src_devs": sorted(srcs),
            "dst_devs": sorted(dsts),
            "src_hosts": sorted({d // devices_per_host for d in srcs}),
            "dst_hosts": sorted({d // devices_per_host for d in dsts}),
        })
    return out


def list_schedule(tasks, order, sender):
    """Start times of a global order (list scheduling) and the makespan."""
    free = {}
    start = [0] * len(tasks)
    makespan = 0
    for i in order:
        hosts = [sender[i]] + tasks[i]["dst_hosts"]
        s = max(free.get(h, 0) for h in hosts)
        start[i] = s
        for h in hosts:
            free[h] = s + tasks[i]["dur"]
        makespan = max(makespan, s + tasks[i]["dur"])
    return start, makespan


def check_schedule(tasks, sender, start):
    """Eq. 2: every sender holds its slice; Eq. 3: no two tasks sharing a
    host overlap in time.  Returns the makespan (Eq. 1)."""
    busy = {}
    for i, t in enumerate(tasks):
        assert sender[i] in t["src_hosts"], f"task {i}: host {sender[i]} does not hold the slice"
        assert start[i] >= 0
        for h in [sender[i]] + t["dst_hosts"]:
            busy.setdefault(h, []).append((start[i], start[i] + t["dur"]))
    for h, iv in busy.items():
        iv.sort()
        for (a0, a1), (b0, b1) in zip(iv, iv[1:]):
            assert a1 <= b0, f"host {h}: [{a0}, {a1}) overlaps [{b0}, {b1})"
    return max((start[i] + t["dur"] for i, t in enumerate(tasks)), default=0)


def naive(tasks):
    """§3.2 'Naive algorithm': the lowest-indexed holder sends; tasks in plan order."""
    return [t["src_hosts"][0] for t in tasks], list(range(len(tasks)))


def load_balance(tasks):
    """§3.2 'Load balance only': by descending T_i, each task to the holder
    host with the lightest send load so far."""
    order = sorted(range(len(tasks)), key=lambda i: (-tasks[i]["dur"], i))
    load = {}
    sender = [None] * len(tasks)
    for i in order:
        h = min(tasks[i]["src_hosts"], key=lambda x: (load.get(x, 0), x))
        sender[i] = h
        load[h] = load.get(h, 0) + tasks[i]["dur"]
    return sender, order


def random_greedy(tasks, trials: int, seed: int):
    """§3.2 'Greedy Search with Randomization'.  Returns (sender, order,
    rounds), rounds being the list of task sets in the order chosen."""
    n = len(tasks)
    remaining = list(range(n))
    load = {}
    sender = [None] * n
    order, rounds = [], []
    k = 0
    while remaining:
        best, best_size = None, -1
        for r in range(trials):
            ctr0 = (k * trials + r) * n
            perm = sorted(remaining, key=lambda t: (splitmix64_at(seed, ctr0 + t), t))
            taken, chosen = set(), []
            for t in perm:
                if any(h in taken for h in tasks[t]["dst_hosts"]):
                    continue
                free = [h for h in tasks[t]["src_hosts"] if h not in taken]
                if not free:
                    continue
                h = min(free, key=lambda x: (load.get(x, 0), x))
                chosen.append((t, h))
                taken.add(h)
                taken.update(tasks[t]["dst_hosts"])
            if len(taken) > best_size:
                best, best_size = chosen, len(taken)
        for t, h in best:
            sender[t] = h
            order.append(t)
            load[h] = load.get(h, 0) + tasks[t]["dur"]
        rounds.append([t for t, _ in best])
        chosen_ids = {t for t, _ in best}
        remaining = [t for t in remaining if t not in chosen_ids]
        k += 1
    return sender, order, rounds


def optimum(tasks):
    """The optimum of Eq. 1-3 by exhaustive enumeration of every global
    order and every sender choice (tiny instances only)."""
    n = len(tasks)
    assert n <= 6, "exhaustive search is for tiny instances"
    best = None
    for choice in itertools.product(*[t["src_hosts"] for t in tasks]):
        for order in itertools.permutations(range(n)):
            _, mk = list_schedule(tasks, order, list(choice))
            if best is None or mk < best:
                best = mk
    return best


def lower_bound(tasks) -> int:
    """Largest of: a host's receive load; the send load forced on a host by
    tasks only it holds; total send work spread over all holder hosts."""
    recv, forced, holders = {}, {}, set()
    total = 0
    for t in tasks:
        for h in t["dst_hosts"]:
            recv[h] = recv.get(h, 0) + t["dur"]
        if len(t["src_hosts"]) == 1:
            h = t["src_hosts"][0]
            forced[h] = forced.get(h, 0) + t["dur"]
        holders.update(t["src_hosts"])
        total += t["dur"]
    spread = -(-total // len(holders)) if holders else 0
    return max([spread] + list(recv.values()) + list(forced.values()))
