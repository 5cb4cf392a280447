// planner.cpp - host-side planners: layout rectangles, the cross-mesh
// resharding planner ("On Optimizing the Communication of Model
// Parallelism", §2 unit tasks and §3.2 load balancing and scheduling) and the
// pipeline-bubble simulator ("Transformer Training 11: Model Parallelism",
// pipeline parallelism).  Plain C++: no CUDA call.
#include <stdint.h>

#include <algorithm>
#include <new>
#include <vector>

#include "../../include/tp3d_plan.h"
#include "layout.cuh"

namespace {

using tp3d::Grid;

#define PLAN_TRY(x)                     \
  do {                                  \
    tp3d_status s_ = (x);               \
    if (s_ != TP3D_OK) return s_;       \
  } while (0)

// ---------------------------------------------------------------------------
// Rectangles
// ---------------------------------------------------------------------------

// Mesh axes a dimension spec splits over: bit 0 = axis 0, bit 1 = axis 1.
int spec_axes(int32_t spec) {
  switch (spec) {
    case TP3D_SPEC_R: return 0;
    case TP3D_SPEC_S0: return 1;
    case TP3D_SPEC_S1: return 2;
    case TP3D_SPEC_S01: return 3;
    default: return -1;
  }
}

// The interval of `extent` that mesh device (a, b) holds under `spec`.
tp3d_status spec_part(int32_t spec, int64_t extent, int32_t m1, int32_t m2, int32_t a, int32_t b, int64_t* start,
                      int64_t* len) {
  int64_t parts = 1, idx = 0;
  switch (spec) {
    case TP3D_SPEC_R: break;
    case TP3D_SPEC_S0: parts = m1; idx = a; break;
    case TP3D_SPEC_S1: parts = m2; idx = b; break;
    case TP3D_SPEC_S01: parts = (int64_t)m1 * m2; idx = (int64_t)a * m2 + b; break;
    default: return TP3D_EINVAL;
  }
  if (extent % parts != 0) return TP3D_ESHAPE;
  *len = extent / parts;
  *start = idx * *len;
  return TP3D_OK;
}

bool same_rect(const tp3d_rect& x, const tp3d_rect& y) {
  return x.row0 == y.row0 && x.rows == y.rows && x.col0 == y.col0 && x.cols == y.cols;
}

bool intersects(const tp3d_rect& x, const tp3d_rect& y) {
  return x.row0 < y.row0 + y.rows && y.row0 < x.row0 + x.rows && x.col0 < y.col0 + y.cols &&
         y.col0 < x.col0 + x.cols;
}

// The distinct rectangles of one side must tile the R x C matrix exactly.
tp3d_status check_partition(const tp3d_rect* r, int32_t n, int64_t R, int64_t C) {
  std::vector<tp3d_rect> u;
  for (int32_t k = 0; k < n; ++k) {
    const tp3d_rect& x = r[k];
    if (x.rows < 1 || x.cols < 1 || x.row0 < 0 || x.col0 < 0 || x.row0 + x.rows > R || x.col0 + x.cols > C)
      return TP3D_ESHAPE;
    bool seen = false;
    for (const tp3d_rect& y : u) seen = seen || same_rect(x, y);
    if (!seen) u.push_back(x);
  }
  int64_t area = 0;
  for (size_t a = 0; a < u.size(); ++a) {
    area += u[a].rows * u[a].cols;
    for (size_t b = a + 1; b < u.size(); ++b)
      if (intersects(u[a], u[b])) return TP3D_ESHAPE;
  }
  return area == R * C ? TP3D_OK : TP3D_ESHAPE;
}

// ---------------------------------------------------------------------------
// SplitMix64 (Steele, Lea and Flood, "Fast Splittable Pseudorandom Number
// Generators", OOPSLA 2014): the state advances by the odd constant gamma and
// each output is the state passed through the 64-bit mixing function.  Output
// number `ctr` (0-based) of the sequence seeded with `seed` is therefore a
// pure function of (seed, ctr): a counter-based generator.
// ---------------------------------------------------------------------------

constexpr uint64_t kGamma = 0x9e3779b97f4a7c15ull;

uint64_t splitmix64_at(uint64_t seed, uint64_t ctr) {
  uint64_t z = seed + (ctr + 1) * kGamma;
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

}  // namespace

// ---------------------------------------------------------------------------
// Cross-mesh resharding plan
// ---------------------------------------------------------------------------

struct tp3d_cmr_plan {
  struct Task {
    tp3d_rect slice;
    int64_t dur;                    // T_i: bytes of the slice
    std::vector<int32_t> src_dev;   // N_i (devices), ascending
    std::vector<int32_t> dst_dev;   // M_i (devices), ascending
    std::vector<int32_t> src_host;  // n_i (hosts), ascending, distinct
    std::vector<int32_t> dst_host;  // m_i (hosts), ascending, distinct
  };
  std::vector<Task> tasks;
  int32_t n_hosts = 0;  // host numbers are 0 .. n_hosts - 1
};

namespace {

void push_host(std::vector<int32_t>& v, int32_t h) {
  if (v.empty() || v.back() != h) v.push_back(h);
}

// List scheduling of a global order (Eq. 3): each task starts when the last
// earlier task on its sender host or any of its receiver hosts has ended.
int64_t list_schedule(const tp3d_cmr_plan& P, const int32_t* order, const int32_t* sender, int64_t* start) {
  std::vector<int64_t> avail(P.n_hosts, 0);
  int64_t makespan = 0;
  for (size_t k = 0; k < P.tasks.size(); ++k) {
    const int32_t i = order[k];
    const auto& t = P.tasks[i];
    int64_t s = avail[sender[i]];
    for (int32_t h : t.dst_host) s = std::max(s, avail[h]);
    start[i] = s;
    const int64_t f = s + t.dur;
    avail[sender[i]] = f;
    for (int32_t h : t.dst_host) avail[h] = f;
    makespan = std::max(makespan, f);
  }
  return makespan;
}

void schedule_naive(const tp3d_cmr_plan& P, int32_t* sender, int32_t* order) {
  for (size_t i = 0; i < P.tasks.size(); ++i) {
    sender[i] = P.tasks[i].src_host.front();
    order[i] = (int32_t)i;
  }
}

// Load balance only: tasks by descending duration (ties by index), each to
// the holder host with the least send load so far (ties: lowest host).
void schedule_load_balance(const tp3d_cmr_plan& P, int32_t* sender, int32_t* order) {
  const int32_t n = (int32_t)P.tasks.size();
  for (int32_t i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order, order + n, [&](int32_t a, int32_t b) { return P.tasks[a].dur > P.tasks[b].dur; });
  std::vector<int64_t> load(P.n_hosts, 0);
  for (int32_t k = 0; k < n; ++k) {
    const auto& t = P.tasks[order[k]];
    int32_t best = t.src_host.front();
    for (int32_t h : t.src_host)
      if (load[h] < load[best]) best = h;
    sender[order[k]] = best;
    load[best] += t.dur;
  }
}

// Greedy search with randomisation: each round keeps, of `trials` random
// orders of the remaining tasks, the set of mutually host-disjoint tasks a
// greedy pass over the order collects that involves the most hosts (ties:
// the first trial).  A task joins the set when none of its receiver hosts is
// taken and one of its holder hosts is free: the free holder with the least
// send load so far (ties: lowest host) sends it.
int32_t schedule_random_greedy(const tp3d_cmr_plan& P, int32_t trials, uint64_t seed, int32_t* sender,
                               int32_t* order) {
  const int32_t n = (int32_t)P.tasks.size();
  std::vector<int32_t> remaining(n);
  for (int32_t i = 0; i < n; ++i) remaining[i] = i;
  std::vector<int64_t> load(P.n_hosts, 0);
  std::vector<char> busy(P.n_hosts, 0);
  std::vector<std::pair<uint64_t, int32_t>> keyed;
  std::vector<std::pair<int32_t, int32_t>> sel, best;
  int32_t placed = 0, round = 0;
  while (!remaining.empty()) {
    int64_t best_size = -1;
    for (int32_t r = 0; r < trials; ++r) {
      keyed.clear();
      const uint64_t base = ((uint64_t)round * (uint64_t)trials + (uint64_t)r) * (uint64_t)n;
      for (int32_t t : remaining) keyed.emplace_back(splitmix64_at(seed, base + (uint64_t)t), t);
      std::sort(keyed.begin(), keyed.end());
      std::fill(busy.begin(), busy.end(), 0);
      sel.clear();
      int64_t size = 0;
      for (const auto& kt : keyed) {
        const auto& t = P.tasks[kt.second];
        bool free_dst = true;
        for (int32_t h : t.dst_host) free_dst = free_dst && !busy[h];
        if (!free_dst) continue;
        int32_t pick = -1;
        for (int32_t h : t.src_host)
          if (!busy[h] && (pick < 0 || load[h] < load[pick])) pick = h;
        if (pick < 0) continue;
        sel.emplace_back(kt.second, pick);
        busy[pick] = 1;
        for (int32_t h : t.dst_host) busy[h] = 1;
        size += 1 + (int64_t)t.dst_host.size();
      }
      if (size > best_size) {
        best_size = size;
        best = sel;
      }
    }
    std::vector<char> taken(n, 0);
    for (const auto& th : best) {
      order[placed++] = th.first;
      sender[th.first] = th.second;
      load[th.second] += P.tasks[th.first].dur;
      taken[th.first] = 1;
    }
    std::vector<int32_t> rest;
    for (int32_t t : remaining)
      if (!taken[t]) rest.push_back(t);
    remaining.swap(rest);
    ++round;
  }
  return round;
}

// Depth-first search with pruning over both decisions: which task comes next
// in the global order, and which holder host sends it.  A branch is cut when
// a lower bound on its completion time reaches the best complete schedule
// found so far; the bound is, for every host, the time it is busy until plus
// the durations of the remaining tasks it must receive (a sum of task
// durations on one host, as Eq. 4).  Starts from the better of the naive and
// load-balance schedules; stops after `node_limit` nodes.
struct Dfs {
  const tp3d_cmr_plan& P;
  int64_t node_limit;
  int64_t nodes = 0;
  bool stopped = false;
  int64_t best;
  std::vector<int32_t> best_order, best_sender;
  std::vector<int32_t> cur_order, cur_sender;
  std::vector<int64_t> avail, rem_recv;
  std::vector<char> done;

  Dfs(const tp3d_cmr_plan& p, int64_t limit) : P(p), node_limit(limit) {}

  void run(int32_t depth, int64_t cur) {
    if (nodes >= node_limit) {
      stopped = true;
      return;
    }
    ++nodes;
    const int32_t n = (int32_t)P.tasks.size();
    if (depth == n) {
      if (cur < best) {
        best = cur;
        best_order = cur_order;
        best_sender = cur_sender;
      }
      return;
    }
    int64_t lb = cur;
    for (int32_t h = 0; h < P.n_hosts; ++h) lb = std::max(lb, avail[h] + rem_recv[h]);
    if (lb >= best) return;
    std::vector<int64_t> saved;
    for (int32_t i = 0; i < n && !stopped; ++i) {
      if (done[i]) continue;
      const auto& t = P.tasks[i];
      for (int32_t h : t.src_host) {
        int64_t s = avail[h];
        for (int32_t r : t.dst_host) s = std::max(s, avail[r]);
        const int64_t f = s + t.dur;
        saved.assign(1, avail[h]);
        for (int32_t r : t.dst_host) saved.push_back(avail[r]);
        avail[h] = f;
        for (int32_t r : t.dst_host) {
          avail[r] = f;
          rem_recv[r] -= t.dur;
        }
        done[i] = 1;
        cur_order.push_back(i);
        cur_sender[i] = h;
        run(depth + 1, std::max(cur, f));
        cur_order.pop_back();
        done[i] = 0;
        for (size_t k = 0; k < t.dst_host.size(); ++k) {
          avail[t.dst_host[k]] = saved[k + 1];
          rem_recv[t.dst_host[k]] += t.dur;
        }
        avail[h] = saved[0];
        if (stopped) break;
      }
    }
  }
};

}  // namespace

extern "C" {

tp3d_status tp3d_layout_rects(int64_t R, int64_t C, tp3d_layout l, tp3d_rect* rects, int32_t capacity,
                              int32_t* count) {
  if (!count) return TP3D_EINVAL;
  Grid g;
  PLAN_TRY(tp3d::make_grid(l, R, C, &g));
  const int32_t n = l.kind == TP3D_REPLICATED ? g.copies : g.nshards();
  *count = n;
  if (!rects || capacity < n) return TP3D_EINVAL;
  if (l.kind == TP3D_REPLICATED) {
    for (int32_t k = 0; k < n; ++k) rects[k] = tp3d_rect{0, R, 0, C};
    return TP3D_OK;
  }
  for (int32_t br = 0; br < g.rb; ++br)
    for (int32_t bc = 0; bc < g.cb; ++bc) rects[g.shard(br, bc)] = tp3d_rect{br * g.bh, g.bh, bc * g.bw, g.bw};
  return TP3D_OK;
}

tp3d_status tp3d_mesh_rects(int64_t R, int64_t C, tp3d_mesh_spec s, tp3d_rect* rects, int32_t capacity,
                            int32_t* count) {
  if (!count || R < 1 || C < 1 || s.m1 < 1 || s.m2 < 1 || (int64_t)s.m1 * s.m2 > (1 << 24)) return TP3D_EINVAL;
  const int ra = spec_axes(s.row_spec), ca = spec_axes(s.col_spec);
  if (ra < 0 || ca < 0 || (ra & ca) != 0) return TP3D_EINVAL;
  const int32_t n = s.m1 * s.m2;
  *count = n;
  for (int32_t a = 0; a < s.m1; ++a)
    for (int32_t b = 0; b < s.m2; ++b) {
      int64_t r0, nr, c0, nc;
      PLAN_TRY(spec_part(s.row_spec, R, s.m1, s.m2, a, b, &r0, &nr));
      PLAN_TRY(spec_part(s.col_spec, C, s.m1, s.m2, a, b, &c0, &nc));
      if (rects && capacity >= n) rects[a * s.m2 + b] = tp3d_rect{r0, nr, c0, nc};
    }
  return (rects && capacity >= n) ? TP3D_OK : TP3D_EINVAL;
}

tp3d_status tp3d_cmr_plan_create(int64_t R, int64_t C, int64_t elem_bytes, const tp3d_rect* src, int32_t n_src,
                                 int32_t src_first, const tp3d_rect* dst, int32_t n_dst, int32_t dst_first,
                                 int32_t devices_per_host, tp3d_cmr_plan** out) {
  if (!out) return TP3D_EINVAL;
  *out = nullptr;
  if (!src || !dst || n_src < 1 || n_dst < 1 || R < 1 || C < 1 || elem_bytes < 1 || devices_per_host < 1 ||
      src_first < 0 || dst_first < 0 || (int64_t)src_first + n_src > INT32_MAX ||
      (int64_t)dst_first + n_dst > INT32_MAX)
    return TP3D_EINVAL;
  if (src_first < dst_first + n_dst && dst_first < src_first + n_src) return TP3D_EOVERLAP;
  const int32_t sh0 = src_first / devices_per_host, sh1 = (src_first + n_src - 1) / devices_per_host;
  const int32_t dh0 = dst_first / devices_per_host, dh1 = (dst_first + n_dst - 1) / devices_per_host;
  if (sh0 <= dh1 && dh0 <= sh1) return TP3D_EINVAL;  // a host with devices of both meshes
  PLAN_TRY(check_partition(src, n_src, R, C));
  PLAN_TRY(check_partition(dst, n_dst, R, C));

  tp3d_cmr_plan* P = new (std::nothrow) tp3d_cmr_plan;
  if (!P) return TP3D_EINVAL;
  P->n_hosts = std::max(sh1, dh1) + 1;
  std::vector<int32_t> task_of(n_src, -1);
  for (int32_t k = 0; k < n_src; ++k) {
    int32_t found = -1;
    for (int32_t e = 0; e < k && found < 0; ++e)
      if (same_rect(src[e], src[k])) found = task_of[e];
    const int32_t dev = src_first + k;
    if (found >= 0) {
      task_of[k] = found;
      auto& t = P->tasks[found];
      t.src_dev.push_back(dev);
      push_host(t.src_host, dev / devices_per_host);
      continue;
    }
    tp3d_cmr_plan::Task t;
    t.slice = src[k];
    t.dur = src[k].rows * src[k].cols * elem_bytes;
    t.src_dev.push_back(dev);
    t.src_host.push_back(dev / devices_per_host);
    for (int32_t e = 0; e < n_dst; ++e)
      if (intersects(src[k], dst[e])) {
        t.dst_dev.push_back(dst_first + e);
        push_host(t.dst_host, (dst_first + e) / devices_per_host);
      }
    task_of[k] = (int32_t)P->tasks.size();
    P->tasks.push_back(std::move(t));
  }
  *out = P;
  return TP3D_OK;
}

void tp3d_cmr_plan_destroy(tp3d_cmr_plan* plan) { delete plan; }

int32_t tp3d_cmr_plan_num_tasks(const tp3d_cmr_plan* plan) { return plan ? (int32_t)plan->tasks.size() : -1; }

tp3d_status tp3d_cmr_plan_task(const tp3d_cmr_plan* plan, int32_t i, tp3d_rect* slice, int64_t* duration,
                               int32_t* senders, int32_t* n_senders, int32_t* receivers, int32_t* n_receivers) {
  if (!plan || i < 0 || i >= (int32_t)plan->tasks.size()) return TP3D_EINVAL;
  const auto& t = plan->tasks[i];
  if (slice) *slice = t.slice;
  if (duration) *duration = t.dur;
  if (n_senders) *n_senders = (int32_t)t.src_dev.size();
  if (n_receivers) *n_receivers = (int32_t)t.dst_dev.size();
  if (senders) std::copy(t.src_dev.begin(), t.src_dev.end(), senders);
  if (receivers) std::copy(t.dst_dev.begin(), t.dst_dev.end(), receivers);
  return TP3D_OK;
}

int64_t tp3d_cmr_plan_lower_bound(const tp3d_cmr_plan* plan) {
  if (!plan) return -1;
  std::vector<int64_t> recv(plan->n_hosts, 0), forced(plan->n_hosts, 0);
  std::vector<char> holder(plan->n_hosts, 0);
  int64_t total = 0, lb = 0;
  for (const auto& t : plan->tasks) {
    for (int32_t h : t.dst_host) recv[h] += t.dur;
    if (t.src_host.size() == 1) forced[t.src_host[0]] += t.dur;
    for (int32_t h : t.src_host) holder[h] = 1;
    total += t.dur;
  }
  int64_t holders = 0;
  for (int32_t h = 0; h < plan->n_hosts; ++h) {
    lb = std::max(lb, std::max(recv[h], forced[h]));
    holders += holder[h];
  }
  return std::max(lb, (total + holders - 1) / holders);
}

tp3d_status tp3d_cmr_schedule(const tp3d_cmr_plan* plan, const tp3d_cmr_options* opt, int32_t* sender_host,
                              int32_t* order, int64_t* start, tp3d_cmr_result* result) {
  if (!plan || !opt || !sender_host || !order || !start || !result) return TP3D_EINVAL;
  const tp3d_cmr_plan& P = *plan;
  *result = tp3d_cmr_result{0, 0, 0, 0};
  switch (opt->algo) {
    case TP3D_CMR_NAIVE:
      schedule_naive(P, sender_host, order);
      break;
    case TP3D_CMR_LOAD_BALANCE:
      schedule_load_balance(P, sender_host, order);
      break;
    case TP3D_CMR_RANDOM_GREEDY:
      if (opt->trials < 1) return TP3D_EINVAL;
      result->rounds = schedule_random_greedy(P, opt->trials, opt->seed, sender_host, order);
      break;
    case TP3D_CMR_DFS: {
      if (opt->node_limit < 1) return TP3D_EINVAL;
      const size_t n = P.tasks.size();
      std::vector<int32_t> s1(n), o1(n), s2(n), o2(n);
      std::vector<int64_t> st(n);
      schedule_naive(P, s1.data(), o1.data());
      schedule_load_balance(P, s2.data(), o2.data());
      const int64_t m1 = list_schedule(P, o1.data(), s1.data(), st.data());
      const int64_t m2 = list_schedule(P, o2.data(), s2.data(), st.data());
      Dfs d(P, opt->node_limit);
      d.best = m2 < m1 ? m2 : m1;
      d.best_order = m2 < m1 ? o2 : o1;
      d.best_sender = m2 < m1 ? s2 : s1;
      d.cur_sender.assign(n, -1);
      d.avail.assign(P.n_hosts, 0);
      d.rem_recv.assign(P.n_hosts, 0);
      d.done.assign(n, 0);
      for (const auto& t : P.tasks)
        for (int32_t h : t.dst_host) d.rem_recv[h] += t.dur;
      d.run(0, 0);
      std::copy(d.best_order.begin(), d.best_order.end(), order);
      std::copy(d.best_sender.begin(), d.best_sender.end(), sender_host);
      result->nodes = d.nodes;
      result->complete = d.stopped ? 0 : 1;
      break;
    }
    default:
      return TP3D_EINVAL;
  }
  result->makespan = list_schedule(P, order, sender_host, start);
  return TP3D_OK;
}

// ---------------------------------------------------------------------------
// Pipeline-bubble simulator
// ---------------------------------------------------------------------------

tp3d_status tp3d_pipeline_simulate(const tp3d_pipe_cfg* cfg, tp3d_pipe_op* ops, int64_t capacity,
                                   tp3d_pipe_result* result) {
  if (!cfg || !result) return TP3D_EINVAL;
  const int32_t p = cfg->p, m = cfg->m, v = cfg->v, sched = cfg->schedule;
  if (p < 1 || m < 1 || v < 1 || cfg->t_f < 1 || cfg->t_b < 1 || p > 4096 || m > (1 << 20) || v > 64)
    return TP3D_EINVAL;
  if (sched != TP3D_PIPE_GPIPE && sched != TP3D_PIPE_1F1B && sched != TP3D_PIPE_INTERLEAVED) return TP3D_EINVAL;
  if (sched != TP3D_PIPE_INTERLEAVED && v != 1) return TP3D_EINVAL;
  if (cfg->t_f % v != 0 || cfg->t_b % v != 0) return TP3D_ESHAPE;
  if (sched == TP3D_PIPE_INTERLEAVED && m % p != 0) return TP3D_ESHAPE;
  const int64_t per_dev = 2 * (int64_t)m * v, total = per_dev * p;
  if (ops && capacity < total) return TP3D_EINVAL;
  const int64_t tf = cfg->t_f / v, tb = cfg->t_b / v;

  struct Op {
    int32_t mb, chunk, bwd;
  };
  // operation order of every device
  std::vector<std::vector<Op>> prog(p);
  for (int32_t d = 0; d < p; ++d) {
    auto& o = prog[d];
    o.reserve(per_dev);
    if (sched == TP3D_PIPE_GPIPE) {
      for (int32_t k = 0; k < m; ++k) o.push_back({k, 0, 0});
      for (int32_t k = 0; k < m; ++k) o.push_back({k, 0, 1});
    } else if (sched == TP3D_PIPE_1F1B) {
      const int32_t w = std::min(p - d - 1, m);
      for (int32_t k = 0; k < w; ++k) o.push_back({k, 0, 0});
      for (int32_t k = 0; k < m - w; ++k) {
        o.push_back({w + k, 0, 0});
        o.push_back({k, 0, 1});
      }
      for (int32_t k = m - w; k < m; ++k) o.push_back({k, 0, 1});
    } else {
      // interleaved: forward op k runs chunk (k / p) % v of micro-batch
      // (k / (p v)) p + k % p; backward op k the chunks in reverse
      const int64_t n = (int64_t)m * v;
      auto fwd = [&](int64_t k) {
        return Op{(int32_t)((k / ((int64_t)p * v)) * p + k % p), (int32_t)((k / p) % v), 0};
      };
      auto bwd = [&](int64_t k) {
        return Op{(int32_t)((k / ((int64_t)p * v)) * p + k % p), (int32_t)(v - 1 - (k / p) % v), 1};
      };
      const int64_t w = std::min<int64_t>(2 * (int64_t)(p - d - 1) + (int64_t)(v - 1) * p, n);
      for (int64_t k = 0; k < w; ++k) o.push_back(fwd(k));
      for (int64_t k = 0; k < n - w; ++k) {
        o.push_back(fwd(w + k));
        o.push_back(bwd(k));
      }
      for (int64_t k = n - w; k < n; ++k) o.push_back(bwd(k));
    }
  }
  // end times of every (stage, micro-batch) forward and backward; stage
  // s = chunk * p + device; -1 = not yet run
  const int64_t S = (int64_t)p * v;
  std::vector<int64_t> fend(S * m, -1), bend(S * m, -1);
  std::vector<int64_t> next(p, 0), free_at(p, 0);
  std::vector<int32_t> in_flight(p, 0), max_in_flight(p, 0);
  std::vector<int64_t> op_start(total), op_end(total);
  int64_t remaining = total, makespan = 0;
  while (remaining > 0) {
    bool progress = false;
    for (int32_t d = 0; d < p; ++d) {
      while (next[d] < per_dev) {
        const Op& o = prog[d][next[d]];
        const int64_t s = (int64_t)o.chunk * p + d;
        int64_t ready;
        if (!o.bwd) {
          ready = s == 0 ? 0 : fend[(s - 1) * m + o.mb];
        } else {
          ready = s == S - 1 ? fend[s * m + o.mb] : bend[(s + 1) * m + o.mb];
        }
        if (ready < 0) break;
        const int64_t st = std::max(ready, free_at[d]);
        const int64_t en = st + (o.bwd ? tb : tf);
        (o.bwd ? bend : fend)[s * m + o.mb] = en;
        free_at[d] = en;
        op_start[(int64_t)d * per_dev + next[d]] = st;
        op_end[(int64_t)d * per_dev + next[d]] = en;
        in_flight[d] += o.bwd ? -1 : 1;
        max_in_flight[d] = std::max(max_in_flight[d], in_flight[d]);
        makespan = std::max(makespan, en);
        ++next[d];
        --remaining;
        progress = true;
      }
    }
    if (!progress) return TP3D_EINVAL;  // an order whose dependencies cannot be met
  }
  if (ops) {
    for (int32_t d = 0; d < p; ++d)
      for (int64_t k = 0; k < per_dev; ++k) {
        const Op& o = prog[d][k];
        ops[(int64_t)d * per_dev + k] =
            tp3d_pipe_op{d, o.mb, o.chunk, o.bwd, op_start[(int64_t)d * per_dev + k], op_end[(int64_t)d * per_dev + k]};
      }
  }
  const int64_t busy = (int64_t)m * (cfg->t_f + cfg->t_b);
  result->makespan = makespan;
  result->busy = busy;
  result->idle = (int64_t)p * (makespan - busy);
  result->bubble = (double)(makespan - busy) / (double)busy;
  result->max_in_flight = *std::max_element(max_in_flight.begin(), max_in_flight.end());
  return TP3D_OK;
}

}  // extern "C"
