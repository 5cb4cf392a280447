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
// lies inside one source shard and one destination shard.  No arithmetic
// touches the data: words are moved as raw bits.  A replicated destination
// is written `copies` times from one read; a replicated source is read from
// copy 0.  Three kernels:
//  * reshard_vec_kernel, cells whose rows are whole 16-byte vectors on both
//    sides: tiles of the refinement (at most 32 KiB), one source and one
//    destination base per tile, then coalesced 16-byte loads and stores with
//    streaming cache hints, eight in flight per thread.  A tile row holds a
//    power of two of vectors, so a thread's flat index splits into row and
//    vector with a shift and a mask (32-bit arithmetic).
//  * reshard_staged_kernel, cells whose rows are not 16-byte aligned (the
//    buffers are): the source side of each cell row (up to 2 KiB of it per
//    job) is brought into shared memory by one untiled bulk copy of the
//    16-byte-aligned span that covers it; each warp keeps a ring of three
//    such stages, two jobs in flight, so the data in flight costs no
//    registers.  Each lane then builds whole 16-byte destination vectors from
//    two aligned shared-memory vectors with funnel shifts, so the stores stay
//    16-byte and coalesced; the partial vectors at a row's two ends are
//    written element by element.
//  * reshard_elem_kernel, everything else (narrow cells, unaligned buffers):
//    one element per thread.
#include "common.cuh"

namespace tp3d {

namespace {

// Division of n < 2^31 by a divisor fixed for the launch, as a multiply-high
// and a shift (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994, the round-up method): with 2^(l-1) < d <= 2^l and
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (umulhi(m, n) + n) >> l.
struct FastDiv {
  uint32_t d, m, l;
};
inline FastDiv fast_div(uint32_t d) {
  FastDiv f;
  f.d = d;
  f.l = 0;
  while ((uint64_t(1) << f.l) < d) ++f.l;
  f.m = (uint32_t)((((uint64_t)1 << 32) * ((uint64_t(1) << f.l) - d)) / d + 1);
  return f;
}
#if defined(__CUDACC__)
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  return (__umulhi(f.m, n) + n) >> f.l;
}
#endif

struct ReshardArgs {
  Grid s, d;
  FastDiv s_bh, s_bw, d_bh, d_bw;  // the grids' block sizes, for the staged kernel's addressing
  const uint8_t* src;
  uint8_t* dst;
  int64_t src_bytes;        // bytes of the source buffer (loads stay inside it)
  int64_t dst_copy_stride;  // bytes between destination copies
  int32_t esz;
  // vector kernel: tiles of RT rows x CT columns, 2^lv vectors per tile row
  int32_t RT, CT, tiles_r, tiles_c, lv;
  // staged kernel: cell rows of `seg` elements, C / seg of them per matrix
  // row, each in jobs of at most kJobBytes destination bytes
  int32_t seg, segs_per_row, jobs_per_seg;
  FastDiv f_spr, f_jps;
  int* err;  // device error word (a bounded wait that runs out)
};

constexpr int kThreads = 256;
constexpr int kUnroll = 8;

__device__ __forceinline__ int64_t grid_offset(const Grid& g, int32_t r, int32_t c) {
  const int32_t br = r / (int32_t)g.bh, bc = c / (int32_t)g.bw;
  return g.block_base(br, bc) + (int64_t)(r - br * (int32_t)g.bh) * g.bw + (c - bc * (int32_t)g.bw);
}
// the same with the block sizes' fast divisors
__device__ __forceinline__ int64_t grid_offset(const Grid& g, const FastDiv& fh, const FastDiv& fw, uint32_t r,
                                               uint32_t c) {
  const uint32_t br = fdiv(r, fh), bc = fdiv(c, fw);
  return g.block_base((int32_t)br, (int32_t)bc) + (int64_t)(r - br * fh.d) * g.bw + (c - bc * fw.d);
}

__global__ void __launch_bounds__(kThreads) reshard_vec_kernel(const ReshardArgs a) {
  const int32_t ntiles = a.tiles_r * a.tiles_c;
  const int32_t vmask = (1 << a.lv) - 1;
  const int32_t nvec = a.RT << a.lv;
  const int64_t sp = a.s.bw * a.esz, dp = a.d.bw * a.esz;  // row pitches in bytes
  for (int32_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int32_t tr = t / a.tiles_c, tc = t - tr * a.tiles_c;
    const int32_t r0 = tr * a.RT, c0 = tc * a.CT;
    const uint8_t* sb = a.src + grid_offset(a.s, r0, c0) * a.esz;
    uint8_t* db = a.dst + grid_offset(a.d, r0, c0) * a.esz;
    for (int32_t v0 = threadIdx.x; v0 < nvec; v0 += kThreads * kUnroll) {
      uint4 buf[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int32_t v = v0 + u * kThreads;
        if (v < nvec) buf[u] = __ldcs(reinterpret_cast<const uint4*>(sb + (v >> a.lv) * sp) + (v & vmask));
      }
      for (int32_t cp = 0; cp < a.d.copies; ++cp) {
        uint8_t* dc = db + cp * a.dst_copy_stride;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int32_t v = v0 + u * kThreads;
          if (v < nvec) __stcs(reinterpret_cast<uint4*>(dc + (v >> a.lv) * dp) + (v & vmask), buf[u]);
        }
      }
    }
  }
}

// Element e of a 16-byte vector (shifts and masks on its four words, so the
// vector stays in registers).
template <typename W>
__device__ __forceinline__ W vec_get(const uint4& v, int e) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (sizeof(W) == 8) {
    return (W)(((uint64_t)w[2 * e + 1] << 32) | w[2 * e]);
  } else if constexpr (sizeof(W) == 4) {
    return (W)w[e];
  } else {
    constexpr int per = 4 / (int)sizeof(W);  // 2 or 4 elements per word
    return (W)(w[e / per] >> (8 * (int)sizeof(W) * (e % per)));
  }
}

// bytes [o, o + 16) of the 32-byte little-endian concatenation lo | hi (o in 0..15)
__device__ __forceinline__ uint4 extract16(const uint4& lo, const uint4& hi, int o) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  const uint32_t sh = (uint32_t)(o & 3) * 8u;
  uint32_t r[4];
  // the word offset o / 4 is the same for the whole warp: each branch indexes
  // the registers with constants
  switch (o >> 2) {
    case 0:
#pragma unroll
      for (int i = 0; i < 4; ++i) r[i] = __funnelshift_r(w[i], w[i + 1], sh);
      break;
    case 1:
#pragma unroll
      for (int i = 0; i < 4; ++i) r[i] = __funnelshift_r(w[i + 1], w[i + 2], sh);
      break;
    case 2:
#pragma unroll
      for (int i = 0; i < 4; ++i) r[i] = __funnelshift_r(w[i + 2], w[i + 3], sh);
      break;
    default:
#pragma unroll
      for (int i = 0; i < 4; ++i) r[i] = __funnelshift_r(w[i + 3], w[i + 4], sh);
      break;
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// Jobs of the staged kernel: chunk c of cell row (r, c0) covers destination
// bytes [D + c kJobBytes, +min(kJobBytes, rest)) and the same source bytes
// from S.  A stage holds 16 bytes of padding, then the source bytes from
// floor16(first source byte) on, at most kJobBytes + 30 of them; the two
// 16-byte reads of the last destination vector reach at most 64 bytes past
// the job, hence the stage size.
constexpr int kJobBytes = 2048;
constexpr int kStageBytes = kJobBytes + 128;
constexpr int kWarpStages = 3;
// the stages, then each warp's three mbarriers, then each warp's abort flag
constexpr int kStagedSmem = (kThreads / 32) * (kWarpStages * (kStageBytes + 8) + 4);

// One warp per job stream (jobs w, w + nwarps, ...), a ring of three stages
// with two jobs in flight.  For job i: wait for its stage, build and store its
// destination vectors (every copy of a replicated destination from the same
// stage), then reuse the stage of job i - 1 for job i + 2.  Every bulk copy
// reads a 16-byte-aligned span inside the source buffer (a span that would
// pass the buffer's end stops at its last whole vector; lanes fetch the few
// bytes after it element by element); every store lies inside its row; every
// wait is bounded.
template <typename W>
__global__ void __launch_bounds__(kThreads) reshard_staged_kernel(const ReshardArgs a) {
  extern __shared__ __align__(128) uint8_t st_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* stage0 = st_smem + warp * kWarpStages * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(st_smem + (kThreads / 32) * kWarpStages * kStageBytes) +
                   warp * kWarpStages;
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(st_smem + (kThreads / 32) * kWarpStages * (kStageBytes + 8)) + warp;
  const int32_t nb = a.seg * a.esz;  // bytes of a cell row (the launcher checks it fits)
  // jobs are numbered in 32 bits (the launcher checks the count fits)
  const uint32_t njobs = (uint32_t)a.s.R * (uint32_t)a.segs_per_row * (uint32_t)a.jobs_per_seg;
  const uint32_t nw = gridDim.x * (kThreads / 32);
  const uint32_t first = blockIdx.x * (kThreads / 32) + warp;
  if (lane == 0) {
    for (int k = 0; k < kWarpStages; ++k) mbar_init(smem_u32(bars + k), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();

  struct Job {
    int64_t S, D0;  // source byte, destination byte (copy 0)
    int32_t n;      // bytes
  };
  auto job = [&](uint32_t i) {
    const uint32_t sg = fdiv(i, a.f_jps);
    const int32_t c = (int32_t)(i - sg * a.f_jps.d);
    const uint32_t r = fdiv(sg, a.f_spr);
    const uint32_t c0 = (sg - r * a.f_spr.d) * (uint32_t)a.seg;
    Job j;
    const int32_t off = c * kJobBytes;
    j.S = grid_offset(a.s, a.s_bh, a.s_bw, r, c0) * a.esz + off;
    j.D0 = grid_offset(a.d, a.d_bh, a.d_bw, r, c0) * a.esz + off;
    j.n = nb - off < kJobBytes ? nb - off : kJobBytes;
    return j;
  };
  // bring job i's source span into stage st
  auto issue = [&](uint32_t i, int st) {
    const Job j = job(i);
    const int64_t lo = j.S & ~(int64_t)15;
    int64_t hi = (j.S + j.n + 15) & ~(int64_t)15;
    const int64_t whole = a.src_bytes & ~(int64_t)15;  // the bulk copy stops at the last whole vector
    if (hi > whole) hi = whole > lo ? whole : lo;
    uint8_t* sb = stage0 + st * kStageBytes + 16;
    // bytes past the last whole vector of the buffer, element by element (generic stores)
    for (int64_t q = hi + lane * a.esz; q < j.S + j.n; q += 32 * a.esz)
      *reinterpret_cast<W*>(sb + (q - lo)) = *reinterpret_cast<const W*>(a.src + q);
    __syncwarp();
    if (lane == 0) {
      const uint32_t bar = smem_u32(bars + st);
      mbar_arrive_expect_tx(bar, (uint32_t)(hi - lo));
      if (hi > lo) bulk_load(smem_u32(sb), a.src + lo, (uint32_t)(hi - lo), bar);
    }
  };
  uint32_t it = 0;  // jobs issued
  for (uint32_t i = first; i < njobs && it < 2; i += nw, ++it) issue(i, (int)it);
  bool ok = true;
  uint32_t done = 0;
  for (uint32_t i = first; i < njobs; i += nw, ++done) {
    const int st = (int)(done % kWarpStages);
    bool got = lane == 0 ? mbar_wait(smem_u32(bars + st), (done / kWarpStages) & 1u, abort_flag, a.err) : false;
    if (!(ok = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0)) break;
    const Job j = job(i);
    const uint8_t* sb = stage0 + st * kStageBytes;  // stage vector jv (the padding is vector 0) at sb + 16 jv
    const int32_t sbase = (int32_t)(j.S & 15);
    for (int32_t cp = 0; cp < a.d.copies; ++cp) {
      const int64_t D = j.D0 + cp * a.dst_copy_stride;
      const int32_t dl = (int32_t)(D & 15);      // D = 16 kb + dl
      const int32_t nv = (dl + j.n + 15) >> 4;   // vectors touching [D, D + n)
      uint8_t* db = a.dst + (D - dl);
      for (int32_t t = lane; t < nv; t += 32) {
        // destination byte 16 (kb + t) takes source byte S + 16 t - dl: stage offset x + 16
        const int32_t x = 16 * t - dl + sbase;  // > -16
        const int32_t jv = (x + 16) >> 4;
        const int o = x & 15;
        const uint4 v0 = *reinterpret_cast<const uint4*>(sb + 16 * jv);
        const uint4 v1 = *reinterpret_cast<const uint4*>(sb + 16 * jv + 16);
        const uint4 v = o == 0 ? v0 : extract16(v0, v1, o);
        uint8_t* dp = db + 16 * t;
        const int32_t b0 = 16 * t - dl;  // byte of the job at the vector's start
        if (b0 >= 0 && b0 + 16 <= j.n) {
          __stcs(reinterpret_cast<uint4*>(dp), v);
        } else {  // a partial vector at either end of the job
#pragma unroll
          for (int e = 0; e < (int)(16 / sizeof(W)); ++e) {
            const int32_t p = b0 + e * (int32_t)sizeof(W);
            if (p >= 0 && p < j.n) reinterpret_cast<W*>(dp)[e] = vec_get<W>(v, e);
          }
        }
      }
    }
    // the stage of this job is read: it takes job done + 3 ... after the
    // generic reads are ordered before the bulk copy's writes
    fence_proxy_async_smem();
    __syncwarp();
    const uint32_t nxt = first + (done + 2) * nw;
    if (nxt < njobs) {
      issue(nxt, (int)((done + 2) % kWarpStages));
      ++it;
    }
  }
  if (!ok && lane == 0) {
    // every bulk copy in flight lands before the CTA may leave
    for (uint32_t q = done; q < it; ++q) {
      const uint32_t bar = smem_u32(bars + (q % kWarpStages));
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(bar, (uint32_t)((q / kWarpStages) & 1)))
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
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

template <template <typename> class K>
void launch_by_size(int esz, unsigned grid, cudaStream_t s, const ReshardArgs& a) {
  switch (esz) {
    case 1: K<uint8_t>::launch(grid, s, a); break;
    case 2: K<uint16_t>::launch(grid, s, a); break;
    case 4: K<uint32_t>::launch(grid, s, a); break;
    default: K<uint64_t>::launch(grid, s, a); break;
  }
}
template <typename W>
struct StagedK {
  static void launch(unsigned g, cudaStream_t s, const ReshardArgs& a) {
    reshard_staged_kernel<W><<<g, kThreads, kStagedSmem, s>>>(a);
  }
  static cudaError_t prepare() {
    return cudaFuncSetAttribute(reshard_staged_kernel<W>, cudaFuncAttributeMaxDynamicSharedMemorySize, kStagedSmem);
  }
};
template <typename W>
struct ElemK {
  static void launch(unsigned g, cudaStream_t s, const ReshardArgs& a) {
    reshard_elem_kernel<W><<<g, kThreads, 0, s>>>(a);
  }
};

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
  // the kernels index rows, columns and tiles in 32 bits
  if (R > INT32_MAX || C > INT32_MAX) return TP3D_EUNSUPPORTED;

  ReshardArgs a{};
  a.s = gs;
  a.d = gd;
  a.src = static_cast<const uint8_t*>(src);
  a.dst = static_cast<uint8_t*>(dst);
  a.src_bytes = (int64_t)R * C * (int64_t)esz;  // copy 0 of a replicated source
  a.esz = (int32_t)esz;
  a.dst_copy_stride = R * C * (int64_t)esz;
  const int64_t gr = gcd64(gs.bh, gd.bh), gc = gcd64(gs.bw, gd.bw);
  const int64_t V = 16 / (int64_t)esz;  // elements per 16-byte vector
  const bool buffers16 = aligned16(src) && aligned16(dst);
  // every cell row starts 16-byte aligned on both sides when both block
  // widths are whole vectors (then so are the shards' sizes and offsets)
  const bool vec = buffers16 && (gs.bw % V == 0) && (gd.bw % V == 0) && (gc % V == 0);
  if (vec) {
    a.CT = (int32_t)gcd64(gc, 4096 / (int64_t)esz);  // at most 4 KiB of a row per tile
    a.RT = (int32_t)gcd64(gr, (int64_t)(32768 / (a.CT * esz) > 0 ? 32768 / (a.CT * esz) : 1));
    a.tiles_r = (int32_t)(R / a.RT);
    a.tiles_c = (int32_t)(C / a.CT);
    const int64_t vpr = (int64_t)a.CT * (int64_t)esz / 16;  // divides 256: a power of two
    int lv = 0;
    while ((int64_t(1) << lv) < vpr) ++lv;
    a.lv = lv;
    const int64_t ntiles = (int64_t)a.tiles_r * a.tiles_c;
    if (ntiles > INT32_MAX) return TP3D_EUNSUPPORTED;
    const int64_t grid = ntiles < (int64_t)ctx->num_sms * 8 ? ntiles : (int64_t)ctx->num_sms * 8;
    reshard_vec_kernel<<<(unsigned)grid, kThreads, 0, stream>>>(a);
  } else if (buffers16 && gc * (int64_t)esz >= 64) {
    a.seg = (int32_t)gc;
    a.segs_per_row = (int32_t)(C / gc);
    a.jobs_per_seg = (int32_t)((gc * (int64_t)esz + kJobBytes - 1) / kJobBytes);
    a.err = ctx->d_err;
    const int64_t njobs = R * (C / gc) * a.jobs_per_seg;
    // job numbers and row / column indices go through the fast divisions (n < 2^31)
    if (njobs > (int64_t)INT32_MAX || gc * (int64_t)esz > INT32_MAX) return TP3D_EUNSUPPORTED;
    a.s_bh = fast_div((uint32_t)gs.bh);
    a.s_bw = fast_div((uint32_t)gs.bw);
    a.d_bh = fast_div((uint32_t)gd.bh);
    a.d_bw = fast_div((uint32_t)gd.bw);
    a.f_spr = fast_div((uint32_t)a.segs_per_row);
    a.f_jps = fast_div((uint32_t)a.jobs_per_seg);
    int64_t grid = (njobs + 7) / 8;
    if (grid > (int64_t)ctx->num_sms * 4) grid = (int64_t)ctx->num_sms * 4;
    cudaError_t e = cudaSuccess;
    switch (esz) {
      case 1: e = StagedK<uint8_t>::prepare(); break;
      case 2: e = StagedK<uint16_t>::prepare(); break;
      case 4: e = StagedK<uint32_t>::prepare(); break;
      default: e = StagedK<uint64_t>::prepare(); break;
    }
    TP3D_CUDA_TRY(e);
    launch_by_size<StagedK>((int)esz, (unsigned)grid, stream, a);
  } else {
    const int64_t n = R * C;
    int64_t grid = (n + kThreads - 1) / kThreads;
    if (grid > (int64_t)ctx->num_sms * 16) grid = (int64_t)ctx->num_sms * 16;
    launch_by_size<ElemK>((int)esz, (unsigned)grid, stream, a);
  }
  return cudaGetLastError() == cudaSuccess ? TP3D_OK : TP3D_ECUDA;
}

}  // namespace tp3d
