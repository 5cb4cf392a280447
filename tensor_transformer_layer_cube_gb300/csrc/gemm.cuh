// gemm.cuh - the sharded, batched GEMM that every 3-D linear, every backward
// product and the attention products are expressed in.
//
// For z in [0, Z):  C_z (M x N) = epilogue(alpha * A_z (M x K) . B_z (K x N))
//
// Each operand is a matrix stored in one of the ABI layouts (a uniform grid
// of row-major shards, `Grid`).  A_z, B_z, C_z are windows of those stored
// matrices at offsets that depend on z (used by attention, where z = batch *
// heads + head); for the 3-D linear Z = 1 and the windows are the whole
// matrices.  An operand is "MN-major" when its stored matrix has the M (or
// N) dimension contiguous, i.e. it is stored as K x M (K x N), "K-major"
// when stored as M x K (N x K).
//
// This is how the cube's communication steps become addressing
// ("Maximizing Parallelism in Distributed Training for Huge Neural Networks",
// §3.1.1 and Algorithm 1): the all-gather of A_il over y and of B_lj over x
// are reads from the q shards that hold them; the contraction loop runs over
// every depth index l in ascending order inside one accumulator, which is the
// reduce-scatter over z; the epilogue writes each device's rows of C_ij into
// its own output shard.
//
// Tiles never straddle a shard: along each dimension the host gives a
// segment length (a common divisor of the block sizes of every operand in
// that dimension and of the per-batch extent); tiles are laid out inside
// segments, and the last tile of a segment may be partial.  Partial tiles are
// correct because (a) along M and N the epilogue masks its stores to the
// segment, and (b) along K the operand whose block ends at the segment end
// reads zeros past it (TMA out-of-bounds fill), so the extra products are 0.
#pragma once

#include "common.cuh"

namespace tp3d {

struct Operand {
  Grid g;            // stored matrix
  const void* ptr;   // device pointer
  int32_t mn_major;  // A/B only: stored as K x (M or N)
  // offsets of the batch-z window along the operand's two logical dims
  // (A: m, k; B: k, n; C: m, n): off(z) = (z / Hz) * hi + (z % Hz) * lo + base
  int64_t hi1, lo1, base1;
  int64_t hi2, lo2, base2;
};

enum EpiAct : int32_t { EPI_NONE = 0, EPI_GELU = 1, EPI_GELU_BWD = 2 };

enum Causal : int32_t {
  CAUSAL_NONE = 0,
  CAUSAL_SKIP_UPPER = 1,  // output m x n = queries x keys: skip tiles with every key > every query
  CAUSAL_K_LE_M = 2,      // contraction over keys: only k <= m contributes
  CAUSAL_K_GE_M = 3       // contraction over queries with m = key: only k >= m contributes
};

struct Epilogue {
  int32_t act;          // EpiAct
  int32_t out_f32;      // C stored as fp32 instead of the input dtype
  float alpha;          // scale of the product
  const float* alpha_dev;  // or null: a device scalar that multiplies alpha
  int64_t f16_cols;     // C's columns below this are written as fp16 (a value
                        // beyond fp16's range raises TP3D_ERANGE), the rest as
                        // bf16; a multiple of 32
  unsigned* amax_out;   // or null: atomic max of |C| over the columns from
                        // f16_cols on, as the bits of a non-negative float
  const void* bias;     // vector indexed by C's stored column, or null
  const void* resid;    // matrix in C's layout added after the activation, or null
  const void* gin;      // EPI_GELU_BWD: the GELU input, in C's layout
  void* zsave;          // pre-activation value written here (C's layout), or null
};

struct GemmProblem {
  int32_t Z, Hz;
  int32_t in_f16;             // A and B hold fp16 (else bf16); both always share a type
  int64_t M, N, K;            // per-batch extents
  int64_t segM, segN, segK;   // segment lengths (divide M, N, K)
  int32_t causal;             // Causal
  Operand a, b, c;
  Epilogue epi;
  int* err;                   // device error area (error word, wait limit)
  int64_t stall_after;        // test hook: the producer stops after this many stages (-1: never)
};

TP3D_HD int64_t op_off(int64_t hi, int64_t lo, int64_t base, int32_t z, int32_t Hz) {
  return (int64_t)(z / Hz) * hi + (int64_t)(z % Hz) * lo + base;
}

// Host entry points (gemm_tc.cu, gemm_simt.cu).
tp3d_status gemm_bf16_tc(const tp3d_ctx* ctx, const GemmProblem& P, cudaStream_t s);
tp3d_status gemm_f32_simt(const tp3d_ctx* ctx, const GemmProblem& P, cudaStream_t s);

// Two GEMMs in one launch, the second's A being the first's output (the MLP
// block; gemm_tc.cu).  chain_plan says whether (P0, P1) qualify and how the
// launch divides them; gemm_chain_tc runs it on a device scratch of
// scratch_bytes whose first counter_bytes hold counters that start at zero
// (each launch leaves them zero again).
struct ChainShape {
  int64_t units0, units1, n_ready, n_fix;
  int32_t splits, ready_target, clusters;
  size_t counter_bytes, scratch_bytes;
};
bool chain_plan(const tp3d_ctx* ctx, const GemmProblem& P0, const GemmProblem& P1, ChainShape* sh);
tp3d_status gemm_chain_tc(const tp3d_ctx* ctx, const GemmProblem& P0, const GemmProblem& P1, const ChainShape& sh,
                          void* scratch, cudaStream_t s);

// Fills segment lengths from the operand grids; returns TP3D_ESHAPE if the
// blocks of the operands do not nest or the extents do not divide.
tp3d_status plan_segments(GemmProblem& P);

}  // namespace tp3d
