// layout.cuh - layout algebra of the sharded matrices (host and device).
//
// Every layout of the ABI is a uniform grid of rb x cb rectangular blocks over
// the R x C matrix plus a map from block (br, bc) to the shard that stores it
// ("Maximizing Parallelism in Distributed Training for Huge Neural Networks",
// §3.1.1 Load Balancing, for the cube layouts; "On Optimizing the
// Communication of Model Parallelism", §2, for the mesh sharding specs).
// Shards are dense row-major bh x bw blocks stored back to back in shard
// order; a replicated layout stores `copies` full copies.
//
// Cube layouts, device (i, j, l) = shard (i*q + j)*q + l:
//   CUBE_A       block rows i*q + j (q^2 of them), block cols l (q)
//   CUBE_B       block rows l (q),  block cols j*q + i (q^2)
//   CUBE_C       block rows i*q + l (q^2), block cols j (q)
//   CUBE_B_SWAP  block rows j (q),  block cols l*q + i (q^2)
#pragma once

#include <stdint.h>

#include "../../include/tp3d.h"

#if defined(__CUDACC__)
#define TP3D_HD __host__ __device__ __forceinline__
#else
#define TP3D_HD inline
#endif

namespace tp3d {

struct Grid {
  int32_t kind;    // tp3d_layout_kind
  int32_t q;       // cube edge (cube kinds)
  int32_t rb, cb;  // blocks per column / per row of blocks
  int64_t R, C;    // matrix size
  int64_t bh, bw;  // block (shard) size
  int32_t copies;  // REPLICATED: number of copies, else 1

  TP3D_HD int64_t shard_elems() const { return bh * bw; }
  TP3D_HD int32_t nshards() const { return rb * cb; }

  // shard number of block (br, bc)
  TP3D_HD int32_t shard(int32_t br, int32_t bc) const {
    switch (kind) {
      case TP3D_CUBE_A: return br * q + bc;                                     // (i q + j) q + l
      case TP3D_CUBE_B: return ((bc % q) * q + bc / q) * q + br;                // i = bc%q, j = bc/q, l = br
      case TP3D_CUBE_C: return ((br / q) * q + bc) * q + br % q;                // i = br/q, l = br%q, j = bc
      case TP3D_CUBE_B_SWAP: return ((bc % q) * q + br) * q + bc / q;           // j = br, l = bc/q, i = bc%q
      case TP3D_ROW: return br;
      case TP3D_COL: return bc;
      case TP3D_BLOCK2D: return br * cb + bc;
      default: return 0;  // REPLICATED: one block
    }
  }

  // element offset of global (r, c) in copy 0
  TP3D_HD int64_t offset(int64_t r, int64_t c) const {
    const int64_t br = r / bh, bc = c / bw;
    return (int64_t)shard((int32_t)br, (int32_t)bc) * (bh * bw) + (r - br * bh) * bw + (c - bc * bw);
  }

  // offset of the first element of block (br, bc)
  TP3D_HD int64_t block_base(int32_t br, int32_t bc) const {
    return (int64_t)shard(br, bc) * (bh * bw);
  }

  TP3D_HD int64_t total_elems() const { return R * C * (int64_t)copies; }
};

// Host: build the grid of a layout for an R x C matrix.  Returns TP3D_OK,
// TP3D_EINVAL (bad kind / q / counts) or TP3D_ESHAPE (not divisible).
inline tp3d_status make_grid(tp3d_layout l, int64_t R, int64_t C, Grid* g) {
  if (R <= 0 || C <= 0) return TP3D_EINVAL;
  Grid x{};
  x.kind = l.kind;
  x.q = l.q;
  x.R = R;
  x.C = C;
  x.copies = 1;
  const int64_t q = l.q;
  switch (l.kind) {
    case TP3D_CUBE_A:
    case TP3D_CUBE_C:
      if (q < 1 || q > 16) return TP3D_EINVAL;
      x.rb = (int32_t)(q * q);
      x.cb = (int32_t)q;
      break;
    case TP3D_CUBE_B:
    case TP3D_CUBE_B_SWAP:
      if (q < 1 || q > 16) return TP3D_EINVAL;
      x.rb = (int32_t)q;
      x.cb = (int32_t)(q * q);
      break;
    case TP3D_ROW:
      if (l.a < 1) return TP3D_EINVAL;
      x.rb = l.a;
      x.cb = 1;
      break;
    case TP3D_COL:
      if (l.a < 1) return TP3D_EINVAL;
      x.rb = 1;
      x.cb = l.a;
      break;
    case TP3D_BLOCK2D:
      if (l.a < 1 || l.b < 1) return TP3D_EINVAL;
      x.rb = l.a;
      x.cb = l.b;
      break;
    case TP3D_REPLICATED:
      if (l.a < 1) return TP3D_EINVAL;
      x.rb = 1;
      x.cb = 1;
      x.copies = l.a;
      break;
    default:
      return TP3D_EINVAL;
  }
  if (R % x.rb != 0 || C % x.cb != 0) return TP3D_ESHAPE;
  x.bh = R / x.rb;
  x.bw = C / x.cb;
  *g = x;
  return TP3D_OK;
}

inline tp3d_layout cube(int kind, int q) {
  tp3d_layout l;
  l.kind = kind;
  l.q = q;
  l.a = 0;
  l.b = 0;
  return l;
}

}  // namespace tp3d
