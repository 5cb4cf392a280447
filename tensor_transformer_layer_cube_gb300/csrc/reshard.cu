// reshard.cu - bit-exact layout conversion between the ABI layouts
// ("On Optimizing the Communication of Model Parallelism", §2, cross-mesh
// resharding; the cube layouts of "Maximizing Parallelism in Distributed
// Training for Huge Neural Networks", §3.1.1).
//
// On one GPU every unit communication task of the page (one unique source
// slice sent to the destinations that need it) is a rectangle copied between
// two shards of the same HBM.  Both layouts are uniform grids, so the
// rectangles of their common refinement are the cells of a grid with row
// step gcd(bh_src, bh_dst) and column step gcd(bw_src, bw_dst); each cell
// lies inside one source shard and one destination shard.  The kernel walks
// tiles of that refinement: per tile, one source and one destination base
// address, then fully coalesced 16-byte loads and stores (streaming cache
// hints, several in flight per thread).  A replicated destination is written
// `copies` times from one read; a replicated source is read from copy 0.
// Cells narrower than 16 bytes, or unaligned buffers, take the element-wise
// kernel.  No arithmetic touches the data: words are moved as raw bits.
#include "common.cuh"

namespace tp3d {

namespace {

struct ReshardArgs {
  Grid s, d;
  const uint8_t* src;
  uint8_t* dst;
  int64_t RT, CT;        // tile rows / columns (elements), divide the refinement steps
  int64_t tiles_r, tiles_c;
  int64_t dst_copy_stride;  // bytes between destination copies
  int32_t esz;
};

constexpr int kThreads = 256;
constexpr int kUnroll = 8;

__global__ void __launch_bounds__(kThreads) reshard_vec_kernel(const ReshardArgs a) {
  const int64_t ntiles = a.tiles_r * a.tiles_c;
  const int64_t vpr = a.CT * a.esz / 16;  // 16-byte vectors per tile row
  const int64_t nvec = a.RT * vpr;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t tr = t / a.tiles_c, tc = t - tr * a.tiles_c;
    const int64_t r0 = tr * a.RT, c0 = tc * a.CT;
    const uint8_t* sb = a.src + a.s.offset(r0, c0) * a.esz;
    uint8_t* db = a.dst + a.d.offset(r0, c0) * a.esz;
    const int64_t sp = a.s.bw * a.esz, dp = a.d.bw * a.esz;  // row pitches in bytes
    for (int64_t v0 = threadIdx.x; v0 < nvec; v0 += (int64_t)kThreads * kUnroll) {
      uint4 buf[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t v = v0 + (int64_t)u * kThreads;
        if (v < nvec) {
          const int64_t rr = v / vpr, cv = v - rr * vpr;
          buf[u] = __ldcs(reinterpret_cast<const uint4*>(sb + rr * sp) + cv);
        }
      }
      for (int32_t cp = 0; cp < a.d.copies; ++cp) {
        uint8_t* dc = db + cp * a.dst_copy_stride;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t v = v0 + (int64_t)u * kThreads;
          if (v < nvec) {
            const int64_t rr = v / vpr, cv = v - rr * vpr;
            __stcs(reinterpret_cast<uint4*>(dc + rr * dp) + cv, buf[u]);
          }
        }
      }
    }
  }
}

template <typename W>
__global__ void __launch_bounds__(kThreads) reshard_elem_kernel(const ReshardArgs a) {
  const int64_t n = a.s.R * a.s.C;
  const W* src = reinterpret_cast<const W*>(a.src);
  W* dst = reinterpret_cast<W*>(a.dst);
  const int64_t cstride = a.dst_copy_stride / (int64_t)sizeof(W);
  for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < n; e += (int64_t)gridDim.x * kThreads) {
    const int64_t r = e / a.s.C, c = e - r * a.s.C;
    const W w = src[a.s.offset(r, c)];
    const int64_t o = a.d.offset(r, c);
    for (int32_t cp = 0; cp < a.d.copies; ++cp) dst[o + cp * cstride] = w;
  }
}

}  // namespace

tp3d_status reshard(const tp3d_ctx* ctx, int64_t R, int64_t C, size_t esz, tp3d_layout sl, const void* src,
                    tp3d_layout dl, void* dst, cudaStream_t stream) {
  if (!src || !dst) return TP3D_EINVAL;
  if (esz != 1 && esz != 2 && esz != 4 && esz != 8) return TP3D_EINVAL;
  Grid gs, gd;
  TP3D_TRY(make_grid(sl, R, C, &gs));
  TP3D_TRY(make_grid(dl, R, C, &gd));
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) % esz) return TP3D_EALIGN;
  const size_t sbytes = (size_t)gs.total_elems() * esz, dbytes = (size_t)gd.total_elems() * esz;
  if (overlaps(src, sbytes, dst, dbytes)) return TP3D_EOVERLAP;

  ReshardArgs a{};
  a.s = gs;
  a.d = gd;
  a.src = static_cast<const uint8_t*>(src);
  a.dst = static_cast<uint8_t*>(dst);
  a.esz = (int32_t)esz;
  a.dst_copy_stride = R * C * (int64_t)esz;
  const int64_t gr = gcd64(gs.bh, gd.bh), gc = gcd64(gs.bw, gd.bw);
  const int64_t V = 16 / (int64_t)esz;  // elements per 16-byte vector
  const bool vec = (gc % V == 0) && aligned16(src) && aligned16(dst);
  if (vec) {
    a.CT = gcd64(gc, 4096 / (int64_t)esz);  // at most 4 KiB of a row per tile
    a.RT = gcd64(gr, (int64_t)(32768 / (a.CT * esz) > 0 ? 32768 / (a.CT * esz) : 1));
    a.tiles_r = R / a.RT;
    a.tiles_c = C / a.CT;
    const int64_t ntiles = a.tiles_r * a.tiles_c;
    const int64_t grid = ntiles < (int64_t)ctx->num_sms * 8 ? ntiles : (int64_t)ctx->num_sms * 8;
    reshard_vec_kernel<<<(unsigned)grid, kThreads, 0, stream>>>(a);
  } else {
    const int64_t n = R * C;
    int64_t grid = (n + kThreads - 1) / kThreads;
    if (grid > (int64_t)ctx->num_sms * 16) grid = (int64_t)ctx->num_sms * 16;
    switch (esz) {
      case 1: reshard_elem_kernel<uint8_t><<<(unsigned)grid, kThreads, 0, stream>>>(a); break;
      case 2: reshard_elem_kernel<uint16_t><<<(unsigned)grid, kThreads, 0, stream>>>(a); break;
      case 4: reshard_elem_kernel<uint32_t><<<(unsigned)grid, kThreads, 0, stream>>>(a); break;
      default: reshard_elem_kernel<uint64_t><<<(unsigned)grid, kThreads, 0, stream>>>(a); break;
    }
  }
  return cudaGetLastError() == cudaSuccess ? TP3D_OK : TP3D_ECUDA;
}

}  // namespace tp3d
