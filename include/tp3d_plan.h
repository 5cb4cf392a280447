/* tp3d_plan.h - host-side planners of libtp3d.so (no GPU involved).
 *
 * 1. Cross-mesh resharding planner, after "On Optimizing the Communication of
 *    Model Parallelism" (arXiv 2211.05322):
 *    - §2 'Data slice' / 'Cross-mesh resharding': a resharding task between
 *      two disjoint device meshes splits into one unit communication task per
 *      unique data slice DS_i of the source layout, sent from one of the
 *      devices N_i that hold it to the destination devices M_i whose slice
 *      overlaps it;
 *    - §3.2 'Load balancing and scheduling' (Eq. 1-3): pick a sender host
 *      n_i* in n_i for every task and start times S_i so that tasks sharing a
 *      sender or receiver host do not overlap, minimising max_i (S_i + T_i);
 *      solved by the four algorithms of that section: naive, load balance
 *      only (greedy, longest task first), depth-first search with pruning,
 *      and greedy search with randomisation.
 * 2. Pipeline-bubble simulator, after "Transformer Training 11: Model
 *    Parallelism" (pipeline parallelism section and its table of simulated
 *    against closed-form bubbles): a discrete-event simulation of GPipe,
 *    1F1B and interleaved 1F1B schedules.
 *
 * Everything here is plain host C++ inside libtp3d.so: no CUDA call, so it
 * runs on a machine without a GPU.  All sizes and times are integers, so
 * results are exact and reproducible across machines.
 */
#ifndef TP3D_PLAN_H_
#define TP3D_PLAN_H_

#include <stdint.h>

#include "tp3d.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------------ */
/* Rectangles of a layout                                                     */
/* ------------------------------------------------------------------------ */

/* The part of the R x C matrix one device holds: rows [row0, row0 + rows),
 * columns [col0, col0 + cols).                                              */
typedef struct {
  int64_t row0, rows, col0, cols;
} tp3d_rect;

/* Per-dimension sharding of a matrix over a 2-D device mesh (m1, m2) (CMR
 * §2 'Device mesh', 'Sharding spec'): R = replicated, S0 / S1 = split over
 * mesh axis 0 / 1, S01 = split over both (axis 0 major).  Mesh device
 * (a, b) is number a * m2 + b.                                              */
typedef enum {
  TP3D_SPEC_R = 0,
  TP3D_SPEC_S0 = 1,
  TP3D_SPEC_S1 = 2,
  TP3D_SPEC_S01 = 3
} tp3d_dim_spec;

typedef struct {
  int32_t m1, m2;        /* mesh shape, m1 * m2 devices                     */
  int32_t row_spec;      /* tp3d_dim_spec of the rows                        */
  int32_t col_spec;      /* tp3d_dim_spec of the columns                     */
} tp3d_mesh_spec;

/* Writes the rectangle of every shard of layout `l` (shard order; a
 * REPLICATED layout gives `a` full-matrix rectangles) into rects[0 .. n),
 * n = *count.  capacity < n: nothing written, *count = n, TP3D_EINVAL.
 * Errors: TP3D_EINVAL for a bad layout, TP3D_ESHAPE when R or C is not
 * divisible by the layout's block counts.                                   */
tp3d_status tp3d_layout_rects(int64_t R, int64_t C, tp3d_layout l, tp3d_rect* rects, int32_t capacity,
                              int32_t* count);

/* The same for a 2-D mesh sharding spec: m1 * m2 rectangles in mesh device
 * order.  A spec may not use a mesh axis twice (S0 S0, S01 S1, ...):
 * TP3D_EINVAL.                                                              */
tp3d_status tp3d_mesh_rects(int64_t R, int64_t C, tp3d_mesh_spec s, tp3d_rect* rects, int32_t capacity,
                            int32_t* count);

/* ------------------------------------------------------------------------ */
/* Cross-mesh resharding plan                                                 */
/* ------------------------------------------------------------------------ */

typedef struct tp3d_cmr_plan tp3d_cmr_plan;

/* Builds the unit communication tasks of resharding an R x C matrix of
 * `elem_bytes`-byte elements from the source mesh (devices src_first ..
 * src_first + n_src - 1, device src_first + k holding src[k]) to the
 * destination mesh (dst_first + k holding dst[k]).
 *
 * One task per distinct source rectangle, in the order of its first holder;
 * its senders are all source devices holding that rectangle, its receivers
 * every destination device whose rectangle overlaps it (ascending).  Hosts
 * group devices: host(d) = d / devices_per_host; scheduling works on hosts
 * (CMR §3.2), and no host may hold devices of both meshes.  A task's
 * duration T_i is its byte count: the time to send the slice once at unit
 * bandwidth, which the pipelined broadcast of CMR §3.1 approaches.
 *
 * Errors: TP3D_EINVAL for null pointers, counts < 1, devices_per_host < 1,
 * elem_bytes < 1, negative device numbers or a host shared by both meshes;
 * TP3D_EOVERLAP when the two device ranges intersect; TP3D_ESHAPE when a
 * rectangle leaves the matrix or the distinct rectangles of either side do
 * not partition it exactly.  The plan owns copies of everything.            */
tp3d_status tp3d_cmr_plan_create(int64_t R, int64_t C, int64_t elem_bytes, const tp3d_rect* src, int32_t n_src,
                                 int32_t src_first, const tp3d_rect* dst, int32_t n_dst, int32_t dst_first,
                                 int32_t devices_per_host, tp3d_cmr_plan** out);
void tp3d_cmr_plan_destroy(tp3d_cmr_plan* plan);

/* Number of unit tasks, -1 for a null plan.                                  */
int32_t tp3d_cmr_plan_num_tasks(const tp3d_cmr_plan* plan);

/* Task i: its slice, duration (bytes), and the sender / receiver DEVICES
 * (global numbers, ascending) into caller arrays of capacity n_src / n_dst
 * of the create call (always enough).  Null arrays are skipped.             */
tp3d_status tp3d_cmr_plan_task(const tp3d_cmr_plan* plan, int32_t i, tp3d_rect* slice, int64_t* duration,
                               int32_t* senders, int32_t* n_senders, int32_t* receivers, int32_t* n_receivers);

/* A lower bound on the makespan of any schedule: the largest of the
 * receive load of a host (sum of T_i of the tasks it receives), the send
 * load forced on a host by tasks it alone holds, and the total send work
 * divided (rounded up) over the hosts that hold any slice.                  */
int64_t tp3d_cmr_plan_lower_bound(const tp3d_cmr_plan* plan);

typedef enum {
  TP3D_CMR_NAIVE = 0,          /* lowest holder sends; tasks in plan order                 */
  TP3D_CMR_LOAD_BALANCE = 1,   /* longest task first to the least-loaded holder host        */
  TP3D_CMR_DFS = 2,            /* branch and bound over sender and order, node-limited      */
  TP3D_CMR_RANDOM_GREEDY = 3   /* rounds of non-overlapping tasks, largest of random trials */
} tp3d_cmr_algo;

typedef struct {
  int32_t algo;         /* tp3d_cmr_algo                                               */
  int32_t trials;       /* RANDOM_GREEDY: random orders tried per round (>= 1)         */
  uint64_t seed;        /* RANDOM_GREEDY: SplitMix64 seed                              */
  int64_t node_limit;   /* DFS: search nodes before it stops with the best found (>= 1) */
} tp3d_cmr_options;

typedef struct {
  int64_t makespan;     /* max_i S_i + T_i (Eq. 1)                                     */
  int64_t nodes;        /* DFS: nodes expanded; else 0                                 */
  int32_t complete;     /* DFS: 1 when the search finished (the makespan is optimal)   */
  int32_t rounds;       /* RANDOM_GREEDY: rounds of non-overlapping tasks; else 0      */
} tp3d_cmr_result;

/* Schedules the plan.  Writes, for every task i, the sending host
 * sender_host[i] (a host holding the slice, Eq. 2) and its start time
 * start[i]; order[0 .. n) is the global order the start times follow.
 * Start times come from list scheduling that order: each task starts when
 * the last earlier task on its sender host or any receiver host ends, so no
 * two tasks sharing a host overlap (Eq. 3).
 *
 * RANDOM_GREEDY draws its random task orders from SplitMix64 (Steele, Lea
 * and Flood, OOPSLA 2014) used as a counter-based generator: the key of
 * task t in trial r of round k is output number (k * trials + r) * n + t of
 * the sequence seeded with `seed`; a trial visits the remaining tasks by
 * ascending (key, t).
 * Errors: TP3D_EINVAL for null arguments, an unknown algorithm, trials < 1
 * or node_limit < 1.                                                        */
tp3d_status tp3d_cmr_schedule(const tp3d_cmr_plan* plan, const tp3d_cmr_options* opt, int32_t* sender_host,
                              int32_t* order, int64_t* start, tp3d_cmr_result* result);

/* ------------------------------------------------------------------------ */
/* Pipeline-bubble simulator                                                  */
/* ------------------------------------------------------------------------ */

typedef enum {
  TP3D_PIPE_GPIPE = 0,        /* all forwards, then all backwards (Huang et al. 2019)        */
  TP3D_PIPE_1F1B = 1,         /* warm-up forwards, then one forward / one backward           */
  TP3D_PIPE_INTERLEAVED = 2   /* 1F1B over v chunks per device (Narayanan et al. 2021)       */
} tp3d_pipe_schedule;

typedef struct {
  int32_t schedule;   /* tp3d_pipe_schedule                                              */
  int32_t p;          /* devices (pipeline stages)                                       */
  int32_t m;          /* micro-batches per step                                          */
  int32_t v;          /* chunks of layers per device (1 unless INTERLEAVED)              */
  int64_t t_f, t_b;   /* forward / backward time of one micro-batch through one device's
                         whole share of layers; a chunk takes t_f / v and t_b / v         */
} tp3d_pipe_cfg;

typedef struct {
  int32_t device, microbatch, chunk, backward;
  int64_t start, end;
} tp3d_pipe_op;

typedef struct {
  int64_t makespan;      /* end of the last operation                               */
  int64_t busy;          /* compute time of one device: m * (t_f + t_b)             */
  int64_t idle;          /* sum over devices of makespan - busy                     */
  double bubble;         /* idle / (p * busy)                                       */
  int32_t max_in_flight; /* most micro-batch chunks whose forward has run and
                            backward not yet, on any device (activations held)   */
} tp3d_pipe_result;

/* Simulates one training step: every device runs its operations in the
 * schedule's order, each starting once the device is free and its input is
 * ready (the forward of the previous stage, or the backward of the next
 * stage; the last stage's backward follows its own forward).  Sends take no
 * time.  `ops` (nullable) receives all 2 * p * m * v operations, device by
 * device in execution order; capacity must then be at least that.
 * Errors: TP3D_EINVAL for a null cfg / result, an unknown schedule, p, m,
 * v < 1, v != 1 outside INTERLEAVED, t_f or t_b < 1, or a too small ops
 * buffer; TP3D_ESHAPE when v does not divide t_f and t_b, or (INTERLEAVED)
 * p does not divide m.                                                      */
tp3d_status tp3d_pipeline_simulate(const tp3d_pipe_cfg* cfg, tp3d_pipe_op* ops, int64_t capacity,
                                   tp3d_pipe_result* result);

#ifdef __cplusplus
}
#endif

#endif /* TP3D_PLAN_H_ */
