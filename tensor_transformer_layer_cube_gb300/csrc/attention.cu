// attention.cu - fused causal attention of the GPT layer on the cube.
//
// "Maximizing Parallelism in Distributed Training for Huge Neural Networks"
// §3.2 puts a Self-Attention block between the two 3-D linears of the first
// block; its core is not partitioned by the page.  Here the heads are read in
// place from the CUBE_C shards of the QKV matrix (the output layout of the
// first linear): head t of sequence b is the window rows [b*s, +s) x columns
// [t*d, +d) (Q), [h + t*d, +d) (K), [2h + t*d, +d) (V).
//
// Q and K arrive in fp16 (the layer writes them so: the softmax's
// sensitivity to its scores' inputs grows with the scores' magnitude, and
// fp16 carries 3 more significant bits than bf16); V, O and dO are bf16.
// Every product takes both operands in one type: S = Q K^T in fp16, the score
// gradients dS in fp16 for dQ = dS K and dK = dS^T Q (scaled by a power of
// two sigma that keeps them inside fp16's range, undone when dQ and dK are
// stored), P in bf16 for O = P V and dV = P^T dO, dP = dO V^T in bf16.
//
// Three persistent tcgen05 kernels, 128-row tiles, warp 0 = TMA
// producer, warp 1 = MMA issuer (and TMEM owner), then one thread per tile
// row (TMEM lane) for the softmax arithmetic:
//  * forward: two query tiles per CTA, one pass over the key tiles at or
//    below the diagonal with an online softmax (S = Q K^T in TMEM, P written
//    back over it, O += P V in TMEM with P read from there, O rescaled only
//    when the row maximum grows by more than 2^8); the row's log-sum-exp is
//    saved for the backward.
//  * backward dK/dV: per key tile, over the query tiles at or above the
//    diagonal: S^T = K Q^T, dP^T = V dO^T (one key row per thread; lse and
//    rowsum(dO O) are per-column values read from shared memory),
//    P^T = exp(S^T - lse), dS^T = P^T (dP^T - rowsum(dO O)) / sqrt(d), then
//    dV += P^T dO and dK += dS^T Q with P^T and dS^T read from TMEM.
//  * backward dQ: per query tile, over the key tiles at or below the
//    diagonal: S, dP, dS as above, dQ += dS K with dS in TMEM (the next key
//    tile's S and dP are computed while dS is formed).
// The score and probability matrices never leave the SM.  Every mbarrier
// wait is bounded; a wait that runs out sets the error word and the CTA
// returns.
#include <cudaTypedefs.h>
#include <math.h>

#include "attention.cuh"

namespace tp3d {

namespace {

constexpr int TR = 128;              // rows of a tile (queries or keys)
constexpr int kComputeWarps = 4;     // forward: row warps per query tile (one per TMEM lane quarter)
// backward: warp 0 producer, warp 1 MMA issuer, warps 2-17 element-wise work,
// four per TMEM lane quarter, each on a quarter of a tile row's 128 columns
constexpr int kBwdComputeWarps = 16;  // backward: element-wise warps, kBwdWpq per TMEM lane quarter
constexpr int kBwdWpq = kBwdComputeWarps / 4;
constexpr int kBwdCpw = 4 / kBwdWpq;    // 32-column chunks of a 128-key (or 128-query) row per warp
constexpr int kBwdThreads = 32 * (2 + kBwdComputeWarps);
constexpr uint32_t kChunk = 16384;   // 128 rows x 64 bf16 columns (one 128-byte swizzle span)
constexpr uint32_t kTile = 2 * kChunk;  // a 128 x 128 bf16 tile
constexpr int kSmem = 7 * kTile + 512 + 1024;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

using bf16 = __nv_bfloat16;

struct Ctx {
  uint32_t base;       // 1024-aligned shared address of the tile area
  uint8_t* base_ptr;
  uint32_t bar0;       // first mbarrier
  volatile int* abort_flag;
  uint32_t* tmem_holder;
};

__device__ __forceinline__ Ctx setup_smem(uint8_t* smem_raw) {
  Ctx c;
  const uint32_t raw = smem_u32(smem_raw);
  c.base = (raw + 1023u) & ~1023u;
  c.base_ptr = smem_raw + (c.base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(c.base_ptr + 7 * kTile);
  c.bar0 = smem_u32(bars);
  c.tmem_holder = reinterpret_cast<uint32_t*>(bars + 40);
  c.abort_flag = reinterpret_cast<volatile int*>(c.tmem_holder + 1);
  return c;
}

// TMA of a 128-row x d-column window at global (row0, col0) of a matrix with
// grid g (the window lies inside one shard): d / 64 boxes of 64 columns.
__device__ __forceinline__ void load_tile(const CUtensorMap* m, const Grid& g, int64_t row0, int64_t col0, int nch,
                                          uint32_t dst, uint32_t bar) {
  // 32-bit division (the launchers check the extents): this runs for every tile loaded
  const int64_t br = (uint32_t)row0 / (uint32_t)g.bh, bc = (uint32_t)col0 / (uint32_t)g.bw;
  const int sh = g.shard((int32_t)br, (int32_t)bc);
  const int c1 = (int)(row0 - br * g.bh), c0 = (int)(col0 - bc * g.bw);
  for (int c = 0; c < nch; ++c) tma_load_3d(dst + c * kChunk, m, bar, c0 + 64 * c, c1, sh);
}

// descriptors of a 128-row tile stored as 64-column swizzled chunks
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int k16) {  // contraction along the columns
  return smem_desc_sw128(tile + (uint32_t)(k16 >> 2) * kChunk + (uint32_t)(k16 & 3) * 32u, 16u, 1024u);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int k16) {  // contraction along the rows
  return smem_desc_sw128(tile + (uint32_t)k16 * 2048u, kChunk, 1024u);
}

__device__ __forceinline__ uint4 pack8f(const float* f) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return v;
}

// The scale sigma of the fp16 score gradients.  With P <= 1 (up to rounding),
// |dP_rk| <= |dO_r| |V_k| and |delta_r| = |dO_r . O_r| <= |dO_r| max_k |V_k|
// (O_r is a convex combination of the V rows), and |V_k| <= sqrt(d) max |V|,
// so (Euclidean norms over a head's d columns)
//   |dS_rk| <= B = 2.1 scale sqrt(d) max_r |dO_r| max |V|.
// sigma = 2^(13 - e) for B < 2^e keeps sigma |dS| below 2^13, a factor 8
// inside fp16's range, and its largest values far above fp16's normal
// minimum; sigma = 1 when B is 0 or not finite.  dmax[0] holds max |dO_r|^2
// (rows and heads), dmax[1] max |V| over every element, as the bits of
// non-negative floats.
__device__ __forceinline__ float ds_sigma(const unsigned* dmax, float scale, int64_t d) {
  const float b = 2.1f * scale * sqrtf((float)d) * sqrtf(__uint_as_float(dmax[0])) * __uint_as_float(dmax[1]);
  if (!(b > 0.0f) || !(b <= 3.0e38f)) return 1.0f;
  int e;
  frexpf(b, &e);  // b = m 2^e, m in [0.5, 1)
  return ldexpf(1.0f, 13 - e);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Ctx& c, int* err, int lane) {
  bool ok = lane == 0 ? mbar_wait(bar, parity, c.abort_flag, err) : false;
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

__device__ __forceinline__ uint32_t tmem_row(uint32_t tmem, int quarter, uint32_t col) {
  return tmem + ((uint32_t)(quarter * 32) << 16) + col;
}

// store 32 fp32 values times mul as bf16 to global row pointer + column offset
// (16-byte aligned): two 32-byte stores where the row is 32-byte aligned (a
// whole sector per lane: each lane writes a different row), else four 16-byte
__device__ __forceinline__ void store_row32(bf16* dst, const uint32_t (&r)[32], float mul = 1.0f) {
  uint4 pk[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    float f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(r[v * 8 + e]) * mul;
    pk[v] = pack8f(f);
  }
  if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
      asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + h * 16), "r"(pk[2 * h].x),
                   "r"(pk[2 * h].y), "r"(pk[2 * h].z), "r"(pk[2 * h].w), "r"(pk[2 * h + 1].x), "r"(pk[2 * h + 1].y),
                   "r"(pk[2 * h + 1].z), "r"(pk[2 * h + 1].w)
                   : "memory");
  } else {
#pragma unroll
    for (int v = 0; v < 4; ++v) *reinterpret_cast<uint4*>(dst + v * 8) = pk[v];
  }
}

__device__ __forceinline__ void mma_tile(uint32_t d_tmem, uint32_t a_tile, bool a_mn, uint32_t b_tile, bool b_mn,
                                         int ksteps, uint32_t idesc, bool accumulate) {
  for (int k = 0; k < ksteps; ++k) {
    const uint64_t ad = a_mn ? desc_mnmajor(a_tile, k) : desc_kmajor(a_tile, k);
    const uint64_t bd = b_mn ? desc_mnmajor(b_tile, k) : desc_kmajor(b_tile, k);
    umma_bf16(d_tmem, ad, bd, idesc, (accumulate || k > 0) ? 1u : 0u);
  }
}

// The persistent CTAs take the work items (numbered longest first) in rounds
// of gridDim.x, each round in the opposite CTA order to the one before: the
// CTA given a round's longest item gets the next round's shortest, which
// evens out the CTAs' total work.  Every role of a CTA walks the same list.
__device__ __forceinline__ int64_t snake_item(int64_t r) {
  const int64_t g = gridDim.x;
  return r * g + ((r & 1) ? g - 1 - (int64_t)blockIdx.x : (int64_t)blockIdx.x);
}

__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
}

// All three kernels are persistent: the CTAs take the work items in longest-first
// order, in rounds (snake_item), and the producer loads the next item's tiles while
// the current one finishes (phase counters run across items).

// ------------------------------------------------------------------ forward
// One pass with an online softmax over two query tiles at once (slots 0 and
// 1: query tiles 2k and 2k+1 of one (batch, head); item w = (k, z) with the
// longest k first).  Both slots share every K and V tile.
//
// Softmax rows (one thread per query row, four warps per slot): each key
// tile's scores are read from TMEM, the row maximum updated, and
// P = 2^(S log2e / sqrt d - m) (bf16, unnormalised) written back into tensor
// memory over the tile's own scores, together with the running row sum l.
// Each tile takes two passes over its scores in TMEM (the maximum, then P),
// with the 32-column chunk loops rolled: an unrolled one-pass form (P held in
// registers against the current base) was faster per tile once warm, but its
// larger code cost each CTA more in instruction fetches on its first tiles
// than it saved.
// The exponent base m only moves when the row maximum exceeds it by more than
// 8 (2^8: P and l stay far from overflow); then l and the row of O already
// accumulated in TMEM are scaled by 2^(m_old - m_new) before the next product
// adds to it.  At the end O / l is stored and the row's log-sum-exp
// (m + log2 l) ln 2 saved.
//
// P stays in tensor memory: O += P V takes its A operand from there (P as
// bf16 pairs in the upper 64 columns of the slot's 128 score columns), so P
// costs neither shared memory nor its bandwidth, and shared memory holds the
// two query tiles and a ring of five K / V tiles.  P overwrites the scores,
// so the issuer starts a slot's next S = Q K^T only once that slot's P V has
// finished: PV0(j) S0(j+1) PV1(j) S1(j+1) per key tile, each S issued after
// its slot's PV completes (the other slot's work keeps the tensor pipe busy
// meanwhile).  A slot's new scores therefore imply its previous product is
// done: the softmax warps may rescale O and overwrite the scores with P
// without waiting for it.  The P chunks are written in descending column
// order into the upper half, so every write lands on scores already read.
//
// warps: 0 TMA producer, 1 MMA issuer + TMEM owner, 2-3 idle (warpgroup 0);
// 4-7 slot 0 rows (warpgroup 1); 8-11 slot 1 rows (warpgroup 2).  Warpgroup 0
// gives registers to the two row warpgroups (setmaxnreg).
// smem: Q0 | Q1 | R0 .. R4 (a ring of K_0 V_0 K_1 V_1 ...), 32 KiB each
// TMEM: S0 [0,128) (P0 in [64,128)) S1 [128,256) (P1 in [192,256))
//       O0 [256, 256+d) O1 [256+d, 256+2d)
constexpr int kFwdThreads = 384;
constexpr int kFwdRegsLow = 64, kFwdRegsHigh = 216;  // 128 x 64 + 256 x 216 <= 384 x 168
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kFwdRing = 5;

__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mqkv, const AttnProblem A, bf16* __restrict__ O,
                    float* __restrict__ lse) {
  extern __shared__ uint8_t smem_raw[];
  const Ctx c = setup_smem(smem_raw);
  auto sQ = [&](int sl) { return c.base + (uint32_t)sl * kTile; };
  auto sR = [&](uint32_t i) { return c.base + (2u + i) * kTile; };
  auto bar = [&](int k) { return c.bar0 + 8u * k; };
  const uint32_t q_full = bar(0), q_empty = bar(1);
  auto r_full = [&](uint32_t i) { return bar(2 + (int)i); };
  auto r_empty = [&](uint32_t i) { return bar(2 + (int)kFwdRing + (int)i); };
  auto s_full = [&](int sl) { return bar(12 + sl); };
  auto p_full = [&](int sl) { return bar(14 + sl); };
  auto p_empty = [&](int sl) { return bar(16 + sl); };
  auto o_full = [&](int sl) { return bar(18 + sl); };
  auto o_empty = [&](int sl) { return bar(20 + sl); };
  const uint32_t final_bar = bar(22);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nq = A.s / TR, npair = (nq + 1) / 2, items = A.Z * npair;
  const int nch = (int)(A.d / 64);
  const uint32_t dbytes = (uint32_t)(A.d * TR * 2);

  if (threadIdx.x == 0) {
    for (int k = 0; k < 23; ++k) {
      const bool four = k == 14 || k == 15 || k == 20 || k == 21;  // p_full, o_empty: one arrival per row warp
      mbar_init(bar(k), four ? kComputeWarps : 1);
    }
    *c.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_map(&mqkv);
  if (warp == 1) {
    tmem_alloc(smem_u32(c.tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *c.tmem_holder;
  if (warp < 4) {
    // ---------------------------------------------------------- warpgroup 0
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kFwdRegsLow));
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t n = 0, ic = 0;
      bool ok = true;
      for (int64_t rd = 0, w = snake_item(0); w < items && ok; w = snake_item(++rd), ++ic) {
        const int64_t k = npair - 1 - w / A.Z, z = w % A.Z, b = z / A.H, t = z % A.H;
        const int64_t iq0 = 2 * k;
        const bool two = iq0 + 1 < nq;
        const int nmax = (int)iq0 + (two ? 2 : 1);
        if (!(ok = mbar_wait(q_empty, (ic & 1) ^ 1, c.abort_flag, A.err))) break;
        mbar_arrive_expect_tx(q_full, dbytes * (two ? 2u : 1u));
        load_tile(&mqkv, A.qkv, b * A.s + iq0 * TR, t * A.d, nch, sQ(0), q_full);
        if (two) load_tile(&mqkv, A.qkv, b * A.s + (iq0 + 1) * TR, t * A.d, nch, sQ(1), q_full);
        for (int j = 0; j < nmax && ok; ++j) {
          for (int kv = 0; kv < 2; ++kv, ++n) {
            const uint32_t slot = n % kFwdRing;
            if (!(ok = mbar_wait(r_empty(slot), ((n / kFwdRing) & 1) ^ 1, c.abort_flag, A.err))) break;
            mbar_arrive_expect_tx(r_full(slot), dbytes);
            load_tile(&mqkv, A.qkv, b * A.s + (int64_t)j * TR, (kv == 0 ? A.h : 2 * A.h) + t * A.d, nch, sR(slot),
                      r_full(slot));
          }
        }
      }
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t id_s = idesc_f16_f32(TR, TR, 0, 0);         // S = Q K^T, fp16
      const uint32_t id_o = idesc_bf16_f32(TR, (int)A.d, 0, 1);  // O += P V, bf16 (P from TMEM, V MN-major)
      const int ks_d = (int)(A.d / 16);
      uint32_t n = 0, ic = 0;
      uint32_t pc[2] = {0, 0}, oc[2] = {0, 0};  // P V products issued, items finished, per slot
      bool ok = true;
      auto ring = [&](uint32_t idx, uint32_t& slot) -> bool {
        slot = idx % kFwdRing;
        return mbar_wait(r_full(slot), (idx / kFwdRing) & 1, c.abort_flag, A.err);
      };
      // S_sl = Q_sl K^T, once the slot's previous P V has read its P
      auto issue_s = [&](int sl, uint32_t kslot) -> bool {
        if (pc[sl] > 0 && !mbar_wait(p_empty(sl), (pc[sl] - 1) & 1, c.abort_flag, A.err)) return false;
        tc_fence_after();
        mma_tile(tmem + (uint32_t)(sl * TR), sQ(sl), false, sR(kslot), false, ks_d, id_s, false);
        umma_commit(s_full(sl));
        return true;
      };
      // O_sl += P_sl V, P from tensor memory
      auto issue_pv = [&](int sl, uint32_t vslot, bool first) -> bool {
        if (!mbar_wait(p_full(sl), pc[sl] & 1, c.abort_flag, A.err)) return false;
        if (first && !mbar_wait(o_empty(sl), (oc[sl] & 1) ^ 1, c.abort_flag, A.err)) return false;
        tc_fence_after();
        const uint32_t pt = tmem + (uint32_t)(sl * TR + 64), ot = tmem + 256u + (uint32_t)(sl * A.d);
        for (int k = 0; k < TR / 16; ++k)
          umma_ts(ot, pt + 8u * (uint32_t)k, desc_mnmajor(sR(vslot), k), id_o, (!first || k > 0) ? 1u : 0u);
        umma_commit(p_empty(sl));
        ++pc[sl];
        return true;
      };
      for (int64_t rd = 0, w = snake_item(0); w < items && ok; w = snake_item(++rd), ++ic) {
        const int64_t iq0 = 2 * (npair - 1 - w / A.Z);
        const bool two = iq0 + 1 < nq;
        const int nkv0 = (int)iq0 + 1, nkv1 = two ? nkv0 + 1 : 0, nmax = two ? nkv1 : nkv0;
        if (!(ok = mbar_wait(q_full, ic & 1, c.abort_flag, A.err))) break;
        const uint32_t n0 = n;  // ring index of K_0; K_j = n0 + 2j, V_j = n0 + 2j + 1
        uint32_t ks = 0;
        if (!(ok = ring(n0, ks) && issue_s(0, ks) && (!two || issue_s(1, ks)))) break;
        if (nmax == 1) umma_commit(q_empty);
        umma_commit(r_empty(ks));
        for (int j = 0; j < nmax && ok; ++j) {
          uint32_t vs = 0, kn = 0;
          const bool more = j + 1 < nmax;
          if (!(ok = ring(n0 + 2 * j + 1, vs))) break;
          if (more && !(ok = ring(n0 + 2 * j + 2, kn))) break;
          if (j < nkv0) {
            if (!(ok = issue_pv(0, vs, j == 0))) break;
            if (j + 1 < nkv0 && !(ok = issue_s(0, kn))) break;
          }
          if (j < nkv1) {
            if (!(ok = issue_pv(1, vs, j == 0))) break;
            if (j + 1 < nkv1 && !(ok = issue_s(1, kn))) break;
          }
          umma_commit(r_empty(vs));
          if (more) {
            if (j + 2 == nmax) umma_commit(q_empty);  // the item's last product with Q issued
            umma_commit(r_empty(kn));
          }
        }
        if (!ok) break;
        umma_commit(o_full(0));
        ++oc[0];
        if (two) {
          umma_commit(o_full(1));
          ++oc[1];
        }
        n = n0 + 2 * (uint32_t)nmax;
      }
      umma_commit(final_bar);
      drain(final_bar, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax rows (warpgroups 1, 2)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kFwdRegsHigh));
    const int sl = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const float sl2 = A.scale * kLog2e;
    const uint32_t s_col = (uint32_t)(sl * TR), p_col = s_col + 64u, o_col = 256u + (uint32_t)(sl * A.d);
    uint32_t sc = 0, oc = 0;
    bool ok = true;
    for (int64_t rd = 0, w = snake_item(0); w < items && ok; w = snake_item(++rd)) {
      const int64_t k = npair - 1 - w / A.Z, z = w % A.Z, b = z / A.H, t = z % A.H;
      const int64_t iq = 2 * k + sl;
      if (iq >= nq) continue;  // an odd tile count leaves the last item's slot 1 empty
      const int nkv = (int)iq + 1;
      float m = -INFINITY, l = 0.0f;
      for (int j = 0; j < nkv && ok; ++j) {
        // new scores; they also mean the slot's previous P V has finished
        if (!(ok = warp_wait(s_full(sl), sc & 1, c, A.err, lane))) break;
        ++sc;
        tc_fence_after();
        const bool diag = j == nkv - 1;
        float ps[8];  // eight partial row sums
#pragma unroll
        for (int i = 0; i < 8; ++i) ps[i] = 0.0f;
        {
          // the row maximum, one 32-column chunk at a time (the smallest code)
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll 1
          for (int cc = 0; cc < TR / 32; ++cc) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem_row(tmem, quarter, s_col + (uint32_t)(cc * 32)), v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (!diag || cc * 32 + e <= r) mx[e & 7] = fmaxf(mx[e & 7], __uint_as_float(v[e]));
          }
          float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
          mt *= sl2;
          // the TMEM accesses are warp-collective (.sync.aligned): the warp
          // rescales when any of its rows needs it, each row by its own factor
          const bool move = mt > m + kRescaleLog2;
          if (j > 0 && __any_sync(0xffffffffu, move)) {
            const float f = move ? ex2_approx(m - mt) : 1.0f;
            l *= f;
            for (int cc = 0; cc < (int)(A.d / 32); ++cc) {
              uint32_t ov[32];
              tmem_ld_32x32b_x32(tmem_row(tmem, quarter, o_col + (uint32_t)(cc * 32)), ov);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
              tmem_st_32x32b_x32(tmem_row(tmem, quarter, o_col + (uint32_t)(cc * 32)), ov);
            }
          }
          if (move) m = mt;
          // P, chunk by chunk from the highest columns down: chunk cc's 32
          // scores become 16 columns of bf16 pairs at p_col + 16 cc, over
          // scores read before
#pragma unroll 1
          for (int cc = TR / 32 - 1; cc >= 0; --cc) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem_row(tmem, quarter, s_col + (uint32_t)(cc * 32)), v);
            tmem_ld_wait();
            uint32_t pk[16];
#pragma unroll
            for (int e2 = 0; e2 < 16; ++e2) {
              const int col = cc * 32 + 2 * e2;
              const float f0 = (!diag || col <= r) ? ex2_approx(fmaf(__uint_as_float(v[2 * e2]), sl2, -m)) : 0.0f;
              const float f1 = (!diag || col + 1 <= r) ? ex2_approx(fmaf(__uint_as_float(v[2 * e2 + 1]), sl2, -m)) : 0.0f;
              ps[(2 * e2) & 7] += f0;
              ps[(2 * e2 + 1) & 7] += f1;
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(f0, f1);
              pk[e2] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            tmem_st_32x32b_x16(tmem_row(tmem, quarter, p_col + (uint32_t)(cc * 16)), pk);
          }
        }
        tmem_st_wait();
        l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
        tc_fence_before();
        warp_arrive(p_full(sl), lane);
      }
      if (!ok || !(ok = warp_wait(o_full(sl), oc & 1, c, A.err, lane))) break;
      tc_fence_after();
      const float inv_l = 1.0f / l;
      const int64_t grow = b * A.s + iq * TR + r;
      const int64_t gcol = t * A.d;
      const int64_t br = grow / A.o.bh, bc = gcol / A.o.bw;
      bf16* dst = O + A.o.block_base((int32_t)br, (int32_t)bc) + (grow - br * A.o.bh) * A.o.bw + (gcol - bc * A.o.bw);
      for (int cc = 0; cc < (int)(A.d / 32); ++cc) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(tmem_row(tmem, quarter, o_col + (uint32_t)(cc * 32)), ov);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * inv_l);
        store_row32(dst + cc * 32, ov);
      }
      tc_fence_before();
      warp_arrive(o_empty(sl), lane);
      ++oc;
      lse[z * A.s + iq * TR + r] = (m + log2f(l)) * kLn2;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ backward: dK, dV
// item w: key tile w / Z of (batch, head) w % Z (the most query tiles first)
// The key tile's rows are the TMEM lanes: S^T = K Q^T and dP^T = V dO^T, so
// P^T and dS^T come out laid out as the A operand of dV += P^T dO and
// dK += dS^T Q and stay in tensor memory: the bf16 (fp16) pairs of a
// 32-query chunk go to the upper 16 columns of the chunk they were computed
// from, which the same warp has already read.  A query tile's log-sum-exp and
// delta arrive with its Q and dO (one 512-byte bulk copy each) and are read
// per column from shared memory.
// The issuer starts S^T(j+1) once dV(j) has read P^T(j), and dP^T(j+1) once
// dK(j) has read dS^T(j): per query tile the tensor pipe sees S^T, dP^T, dV, dK,
// and the element-wise warps form P^T while dP^T is computed.
// smem: K | V | Q0 dO0 | Q1 dO1 (32 KiB each) | lse0 delta0 lse1 delta1 (512 B each)
// TMEM (lanes = keys): S^T [0,128), dP^T [128,256), dV [256,256+d), dK [256+d, 256+2d)
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap mqkv, const __grid_constant__ CUtensorMap mo,
                         const AttnProblem A, const float* __restrict__ lse, const float* __restrict__ delta,
                         const unsigned* __restrict__ dmax, bf16* __restrict__ dqkv) {
  extern __shared__ uint8_t smem_raw[];
  const Ctx c = setup_smem(smem_raw);
  const uint32_t sK = c.base, sV = c.base + kTile;
  const uint32_t sQ[2] = {c.base + 2 * kTile, c.base + 4 * kTile}, sdO[2] = {c.base + 3 * kTile, c.base + 5 * kTile};
  const uint32_t sStat = c.base + 6 * kTile;  // per slot: lse [0,128), delta [128,256) as floats
  const float* pStat = reinterpret_cast<const float*>(c.base_ptr + 6 * kTile);
  auto bar = [&](int k) { return c.bar0 + 8u * k; };
  const uint32_t kv_full = bar(0), kv_empty = bar(1), s_full = bar(2), dp_full = bar(3), p_full = bar(4),
                 ds_full = bar(5), s_free = bar(6), dp_free = bar(7), acc_full = bar(8), acc_empty = bar(9),
                 final_bar = bar(10);
  auto r_full = [&](int s) { return bar(11 + s); };
  auto r_empty = [&](int s) { return bar(13 + s); };
  constexpr int kBars = 15;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nq = A.s / TR, items = A.Z * nq;
  const int nch = (int)(A.d / 64);
  const uint32_t dbytes = (uint32_t)(A.d * TR * 2);

  if (threadIdx.x == 0) {
    for (int k = 0; k < kBars; ++k) {
      // p_full, ds_full, acc_empty: one arrival per element-wise warp
      const bool ew = k == 4 || k == 5 || k == 9;
      mbar_init(bar(k), ew ? kBwdComputeWarps : 1);
    }
    *c.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(c.tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *c.tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t n = 0, ic = 0;
      bool ok = true;
      for (int64_t rd = 0, w = snake_item(0); w < items && ok; w = snake_item(++rd), ++ic) {
        const int64_t jk = w / A.Z, z = w % A.Z, b = z / A.H, t = z % A.H;
        const int niter = (int)(nq - jk);
        if (!(ok = mbar_wait(kv_empty, (ic & 1) ^ 1, c.abort_flag, A.err))) break;
        const int64_t row_k = b * A.s + jk * TR;
        mbar_arrive_expect_tx(kv_full, 2 * dbytes);
        load_tile(&mqkv, A.qkv, row_k, A.h + t * A.d, nch, sK, kv_full);
        load_tile(&mqkv, A.qkv, row_k, 2 * A.h + t * A.d, nch, sV, kv_full);
        for (int it = 0; it < niter; ++it, ++n) {
          const int s = n & 1;
          if (!(ok = mbar_wait(r_empty(s), ((n >> 1) & 1) ^ 1, c.abort_flag, A.err))) break;
          mbar_arrive_expect_tx(r_full(s), 2 * dbytes + 2 * TR * 4);
          const int64_t row_q = b * A.s + (jk + it) * TR;
          load_tile(&mqkv, A.qkv, row_q, t * A.d, nch, sQ[s], r_full(s));
          load_tile(&mo, A.o, row_q, t * A.d, nch, sdO[s], r_full(s));
          const int64_t q0 = z * A.s + (jk + it) * TR;  // the tile's first row of lse and delta
          bulk_load(sStat + (uint32_t)s * 1024u, lse + q0, TR * 4, r_full(s));
          bulk_load(sStat + (uint32_t)s * 1024u + 512u, delta + q0, TR * 4, r_full(s));
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = idesc_f16_f32(TR, TR, 0, 0);           // S^T = K Q^T, fp16
      const uint32_t id_dp = idesc_bf16_f32(TR, TR, 0, 0);          // dP^T = V dO^T, bf16
      const uint32_t id_dv = idesc_bf16_f32(TR, (int)A.d, 0, 1);    // dV += P^T dO, bf16 (P^T from TMEM, dO MN-major)
      const uint32_t id_dk = idesc_f16_f32(TR, (int)A.d, 0, 1);     // dK += dS^T Q, fp16 (dS^T from TMEM, Q MN-major)
      const int ks_d = (int)(A.d / 16);
      // TMEM column of the A operand's 16 queries [16 k, +16): the upper half
      // of their 32-query chunk
      auto a_col = [](uint32_t base, int k) { return base + 32u * (uint32_t)(k >> 1) + 16u + 8u * (uint32_t)(k & 1); };
      uint32_t n = 0, ic = 0;
      bool ok = true;
      for (int64_t rd = 0, w = snake_item(0); w < items && ok; w = snake_item(++rd), ++ic) {
        const int niter = (int)(nq - w / A.Z);
        if (!(ok = mbar_wait(kv_full, ic & 1, c.abort_flag, A.err))) break;
        for (int it = 0; it < niter && ok; ++it, ++n) {
          const int s = n & 1;
          if (!(ok = mbar_wait(r_full(s), (n >> 1) & 1, c.abort_flag, A.err))) break;
          if (!(ok = mbar_wait(s_free, (n & 1) ^ 1, c.abort_flag, A.err))) break;  // dV(j-1) has read P^T
          tc_fence_after();
          mma_tile(tmem, sK, false, sQ[s], false, ks_d, id_s, false);  // S^T = K Q^T
          umma_commit(s_full);
          if (!(ok = mbar_wait(dp_free, (n & 1) ^ 1, c.abort_flag, A.err))) break;  // dK(j-1) has read dS^T
          tc_fence_after();
          mma_tile(tmem + 128u, sV, false, sdO[s], false, ks_d, id_dp, false);  // dP^T = V dO^T
          if (it == niter - 1) umma_commit(kv_empty);  // the item's K and V are no longer read
          umma_commit(dp_full);
          if (!(ok = mbar_wait(p_full, n & 1, c.abort_flag, A.err))) break;
          if (it == 0 && !(ok = mbar_wait(acc_empty, (ic & 1) ^ 1, c.abort_flag, A.err))) break;
          tc_fence_after();
          for (int k = 0; k < TR / 16; ++k)  // dV += P^T dO
            umma_ts(tmem + 256u, tmem + a_col(0u, k), desc_mnmajor(sdO[s], k), id_dv, (it > 0 || k > 0) ? 1u : 0u);
          umma_commit(s_free);
          if (!(ok = mbar_wait(ds_full, n & 1, c.abort_flag, A.err))) break;
          tc_fence_after();
          for (int k = 0; k < TR / 16; ++k)  // dK += dS^T Q
            umma_ts(tmem + 256u + (uint32_t)A.d, tmem + a_col(128u, k), desc_mnmajor(sQ[s], k), id_dk,
                    (it > 0 || k > 0) ? 1u : 0u);
          umma_commit(dp_free);
          umma_commit(r_empty(s));
        }
        if (ok) umma_commit(acc_full);
      }
      umma_commit(final_bar);
      drain(final_bar, 0);
    }
  } else {
    // ---------------------------------------- key rows of S^T and dP^T (then of dV, dK)
    const int quarter = warp & 3;
    const int cgp = (warp - 2) >> 2;  // query columns [32 kBwdCpw cgp, +32 kBwdCpw) of the tile
    const int r = quarter * 32 + lane;
    const float sl2 = A.scale * kLog2e;
    const float sigma = ds_sigma(dmax, A.scale, A.d), dscale = A.scale * sigma;
    uint32_t n = 0, ic = 0;
    bool ok = true;
    for (int64_t rd = 0, w = snake_item(0); w < items && ok; w = snake_item(++rd), ++ic) {
      const int64_t jk = w / A.Z, z = w % A.Z, b = z / A.H, t = z % A.H;
      const int niter = (int)(nq - jk);
      for (int it = 0; it < niter && ok; ++it, ++n) {
        const int s = n & 1;
        const float* st = pStat + s * 256;  // lse [0,128), delta [128,256) of the query tile
        if (!(ok = warp_wait(r_full(s), (n >> 1) & 1, c, A.err, lane))) break;
        __syncwarp();  // lane 0 observed the copies of lse and delta: order the other lanes' reads after it
        if (!(ok = warp_wait(s_full, n & 1, c, A.err, lane))) break;
        tc_fence_after();
        const bool diag = it == 0;
        // P^T = exp2(S^T sl2 - lse log2 e), zero where the key follows the query
        float pf[kBwdCpw][32];
#pragma unroll
        for (int i = 0; i < kBwdCpw; ++i) {
          const int ch = kBwdCpw * cgp + i;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem_row(tmem, quarter, (uint32_t)(ch * 32)), v);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 l4 = *reinterpret_cast<const float4*>(st + ch * 32 + 4 * e4);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = ch * 32 + 4 * e4 + e;
              pf[i][4 * e4 + e] =
                  (!diag || j >= r) ? ex2_approx(fmaf(__uint_as_float(v[4 * e4 + e]), sl2, -lv[e] * kLog2e)) : 0.0f;
            }
          }
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(pf[i][2 * e2], pf[i][2 * e2 + 1]);
            pk[e2] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          tmem_st_32x32b_x16(tmem_row(tmem, quarter, (uint32_t)(ch * 32 + 16)), pk);
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(p_full, lane);
        // sigma dS^T = P^T (dP^T - delta) * scale * sigma, as fp16 pairs
        if (!(ok = warp_wait(dp_full, n & 1, c, A.err, lane))) break;
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < kBwdCpw; ++i) {
          const int ch = kBwdCpw * cgp + i;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem_row(tmem, quarter, (uint32_t)(128 + ch * 32)), v);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 d4 = *reinterpret_cast<const float4*>(st + 128 + ch * 32 + 4 * e4);
            const float d0 = pf[i][4 * e4] * (__uint_as_float(v[4 * e4]) - d4.x) * dscale;
            const float d1 = pf[i][4 * e4 + 1] * (__uint_as_float(v[4 * e4 + 1]) - d4.y) * dscale;
            const float d2 = pf[i][4 * e4 + 2] * (__uint_as_float(v[4 * e4 + 2]) - d4.z) * dscale;
            const float d3 = pf[i][4 * e4 + 3] * (__uint_as_float(v[4 * e4 + 3]) - d4.w) * dscale;
            const __half2 h01 = __floats2half2_rn(d0, d1), h23 = __floats2half2_rn(d2, d3);
            pk[2 * e4] = *reinterpret_cast<const uint32_t*>(&h01);
            pk[2 * e4 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
          }
          tmem_st_32x32b_x16(tmem_row(tmem, quarter, (uint32_t)(128 + ch * 32 + 16)), pk);
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(ds_full, lane);
      }
      if (!ok || !(ok = warp_wait(acc_full, ic & 1, c, A.err, lane))) break;
      tc_fence_after();
      const int64_t grow = b * A.s + jk * TR + r;
      for (int which = 0; which < 2; ++which) {  // 0: dV at 2h + t d, 1: dK at h + t d
        const int64_t gcol = (which == 0 ? 2 * A.h : A.h) + t * A.d;
        const int64_t br = grow / A.qkv.bh, bc = gcol / A.qkv.bw;
        bf16* dst = dqkv + A.qkv.block_base((int32_t)br, (int32_t)bc) + (grow - br * A.qkv.bh) * A.qkv.bw +
                    (gcol - bc * A.qkv.bw);
        const float mul = which == 0 ? 1.0f : 1.0f / sigma;  // dK was accumulated from sigma dS
        for (int cc = cgp; cc < (int)(A.d / 32); cc += kBwdWpq) {  // this warp's 32-column chunks of d
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem_row(tmem, quarter, 256u + (uint32_t)(which * A.d) + cc * 32), v);
          tmem_ld_wait();
          store_row32(dst + cc * 32, v, mul);
        }
      }
      tc_fence_before();
      warp_arrive(acc_empty, lane);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ backward: dQ
// item w: query tile nq-1-(w / Z) of (batch, head) w % Z
// smem: Q | dO | K0 K1 K2 | V0 V1 (32 KiB each): K in a ring of three (read by
// S and by dQ), V in a ring of two (read by dP only)
// TMEM: S [0,128) dP [128,256) dQ [256,256+d), sigma dS as fp16 pairs in two
// buffers of 64 columns at 384 and 448 (the A operand of dQ += dS K)
// The element-wise warps copy a tile's S and dP into registers and release
// them at once, so the issuer runs the next key tile's S and dP while they
// form dS: per key tile the tensor pipe sees S(j+1), dP(j+1), dQ(j).
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap mqkv, const __grid_constant__ CUtensorMap mo,
                       const AttnProblem A, const float* __restrict__ lse, const float* __restrict__ delta,
                       const unsigned* __restrict__ dmax, bf16* __restrict__ dqkv) {
  extern __shared__ uint8_t smem_raw[];
  const Ctx c = setup_smem(smem_raw);
  const uint32_t sQ = c.base, sdO = c.base + kTile;
  auto sK = [&](uint32_t i) { return c.base + (2u + i) * kTile; };
  auto sV = [&](uint32_t i) { return c.base + (5u + i) * kTile; };
  auto bar = [&](int k) { return c.bar0 + 8u * k; };
  const uint32_t qo_full = bar(0), qo_empty = bar(1), s_full = bar(2), s_empty = bar(3), acc_full = bar(4),
                 acc_empty = bar(5), final_bar = bar(6);
  auto ds_full = [&](uint32_t b) { return bar(7 + (int)b); };    // 2
  auto ds_empty = [&](uint32_t b) { return bar(9 + (int)b); };   // 2
  auto k_full = [&](uint32_t i) { return bar(11 + (int)i); };    // 3
  auto k_empty = [&](uint32_t i) { return bar(14 + (int)i); };   // 3
  auto v_full = [&](uint32_t i) { return bar(17 + (int)i); };    // 2
  auto v_empty = [&](uint32_t i) { return bar(19 + (int)i); };   // 2
  constexpr int kBars = 21;
  constexpr uint32_t kDs = 384;  // first dS buffer column

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nq = A.s / TR, items = A.Z * nq;
  const int nch = (int)(A.d / 64);
  const uint32_t dbytes = (uint32_t)(A.d * TR * 2);

  if (threadIdx.x == 0) {
    for (int k = 0; k < kBars; ++k) {
      // s_empty, acc_empty, ds_full: one arrival per element-wise warp
      const bool ew = k == 3 || k == 5 || k == 7 || k == 8;
      mbar_init(bar(k), ew ? kBwdComputeWarps : 1);
    }
    *c.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(c.tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *c.tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t n = 0, ic = 0;
      bool ok = true;
      for (int64_t rd = 0, w = snake_item(0); w < items && ok; w = snake_item(++rd), ++ic) {
        const int64_t iq = nq - 1 - w / A.Z, z = w % A.Z, b = z / A.H, t = z % A.H;
        const int niter = (int)iq + 1;
        if (!(ok = mbar_wait(qo_empty, (ic & 1) ^ 1, c.abort_flag, A.err))) break;
        const int64_t row_q = b * A.s + iq * TR;
        mbar_arrive_expect_tx(qo_full, 2 * dbytes);
        load_tile(&mqkv, A.qkv, row_q, t * A.d, nch, sQ, qo_full);
        load_tile(&mo, A.o, row_q, t * A.d, nch, sdO, qo_full);
        for (int it = 0; it < niter; ++it, ++n) {
          const uint32_t ks = n % 3, vs = n & 1;
          const int64_t row_k = b * A.s + (int64_t)it * TR;
          // V first: its slot frees when dP(j-2) completes, K's only when dQ(j-3) does
          if (!(ok = mbar_wait(v_empty(vs), ((n >> 1) & 1) ^ 1, c.abort_flag, A.err))) break;
          mbar_arrive_expect_tx(v_full(vs), dbytes);
          load_tile(&mqkv, A.qkv, row_k, 2 * A.h + t * A.d, nch, sV(vs), v_full(vs));
          if (!(ok = mbar_wait(k_empty(ks), ((n / 3) & 1) ^ 1, c.abort_flag, A.err))) break;
          mbar_arrive_expect_tx(k_full(ks), dbytes);
          load_tile(&mqkv, A.qkv, row_k, A.h + t * A.d, nch, sK(ks), k_full(ks));
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = idesc_f16_f32(TR, TR, 0, 0);           // S = Q K^T, fp16
      const uint32_t id_dp = idesc_bf16_f32(TR, TR, 0, 0);          // dP = dO V^T, bf16
      const uint32_t id_acc = idesc_f16_f32(TR, (int)A.d, 0, 1);    // dQ += dS K, fp16 (dS from TMEM, K MN-major)
      const int ks_d = (int)(A.d / 16);
      uint32_t n = 0, ic = 0;
      bool ok = true;
      // S and dP of global key-tile iteration m, once the element-wise warps
      // hold iteration m-1's; V's slot is free again when dP completes
      auto issue_sdp = [&](uint32_t m, bool last) -> bool {
        if (!mbar_wait(k_full(m % 3), (m / 3) & 1, c.abort_flag, A.err)) return false;
        if (!mbar_wait(v_full(m & 1), (m >> 1) & 1, c.abort_flag, A.err)) return false;
        if (!mbar_wait(s_empty, (m & 1) ^ 1, c.abort_flag, A.err)) return false;
        tc_fence_after();
        mma_tile(tmem, sQ, false, sK(m % 3), false, ks_d, id_s, false);          // S = Q K^T
        mma_tile(tmem + 128u, sdO, false, sV(m & 1), false, ks_d, id_dp, false);  // dP = dO V^T
        umma_commit(v_empty(m & 1));
        if (last) umma_commit(qo_empty);  // the item's Q and dO are no longer read
        umma_commit(s_full);
        return true;
      };
      for (int64_t rd = 0, w = snake_item(0); w < items && ok; w = snake_item(++rd), ++ic) {
        const int niter = (int)(nq - 1 - w / A.Z) + 1;
        if (!(ok = mbar_wait(qo_full, ic & 1, c.abort_flag, A.err))) break;
        if (!(ok = issue_sdp(n, niter == 1))) break;
        for (int it = 0; it < niter && ok; ++it, ++n) {
          if (it + 1 < niter && !(ok = issue_sdp(n + 1, it + 2 == niter))) break;
          const uint32_t db = n & 1;
          if (!(ok = mbar_wait(ds_full(db), (n >> 1) & 1, c.abort_flag, A.err))) break;
          if (it == 0 && !(ok = mbar_wait(acc_empty, (ic & 1) ^ 1, c.abort_flag, A.err))) break;
          tc_fence_after();
          const uint32_t dst = tmem + kDs + 64u * db;
          for (int k = 0; k < TR / 16; ++k)  // dQ += dS K
            umma_ts(tmem + 256u, dst + 8u * (uint32_t)k, desc_mnmajor(sK(n % 3), k), id_acc,
                    (it > 0 || k > 0) ? 1u : 0u);
          umma_commit(ds_empty(db));
          umma_commit(k_empty(n % 3));
        }
        if (ok) umma_commit(acc_full);
      }
      umma_commit(final_bar);
      drain(final_bar, 0);
    }
  } else {
    // ------------------------------------------------------------ query rows
    const int quarter = warp & 3;
    const int cgp = (warp - 2) >> 2;  // key columns [32 kBwdCpw cgp, +32 kBwdCpw) of the tile
    const int r = quarter * 32 + lane;
    const float sl2 = A.scale * kLog2e;
    const float sigma = ds_sigma(dmax, A.scale, A.d), dscale = A.scale * sigma;
    uint32_t n = 0, ic = 0;
    bool ok = true;
    for (int64_t rd = 0, w = snake_item(0); w < items && ok; w = snake_item(++rd), ++ic) {
      const int64_t iq = nq - 1 - w / A.Z, z = w % A.Z, b = z / A.H, t = z % A.H;
      const int niter = (int)iq + 1;
      const int64_t qrow = z * A.s + iq * TR + r;
      const float l2 = lse[qrow] * kLog2e, dr = delta[qrow];
      for (int it = 0; it < niter && ok; ++it, ++n) {
        if (!(ok = warp_wait(s_full, n & 1, c, A.err, lane))) break;
        tc_fence_after();
        const bool diag = it == niter - 1;
        uint32_t v[kBwdCpw][32], wv[kBwdCpw][32];
#pragma unroll
        for (int i = 0; i < kBwdCpw; ++i) {
          tmem_ld_32x32b_x32(tmem_row(tmem, quarter, (uint32_t)((kBwdCpw * cgp + i) * 32)), v[i]);
          tmem_ld_32x32b_x32(tmem_row(tmem, quarter, (uint32_t)(128 + (kBwdCpw * cgp + i) * 32)), wv[i]);
        }
        tmem_ld_wait();
        tc_fence_before();
        warp_arrive(s_empty, lane);  // S and dP are in registers: the next key tile's may overwrite them
        // sigma dS = P (dP - delta) * scale * sigma, P = exp2(S sl2 - lse), zero where the key follows the query
        uint32_t pk[kBwdCpw][16];
#pragma unroll
        for (int i = 0; i < kBwdCpw; ++i) {
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            const int k = (kBwdCpw * cgp + i) * 32 + 2 * e2;
            const float p0 = (!diag || k <= r) ? ex2_approx(fmaf(__uint_as_float(v[i][2 * e2]), sl2, -l2)) : 0.0f;
            const float p1 = (!diag || k + 1 <= r) ? ex2_approx(fmaf(__uint_as_float(v[i][2 * e2 + 1]), sl2, -l2)) : 0.0f;
            const __half2 h2 = __floats2half2_rn(p0 * (__uint_as_float(wv[i][2 * e2]) - dr) * dscale,
                                                 p1 * (__uint_as_float(wv[i][2 * e2 + 1]) - dr) * dscale);
            pk[i][e2] = *reinterpret_cast<const uint32_t*>(&h2);
          }
        }
        const uint32_t db = n & 1;
        if (!(ok = warp_wait(ds_empty(db), ((n >> 1) & 1) ^ 1, c, A.err, lane))) break;  // dQ(j-2) has read it
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < kBwdCpw; ++i)
          tmem_st_32x32b_x16(tmem_row(tmem, quarter, kDs + 64u * db + (uint32_t)((kBwdCpw * cgp + i) * 16)), pk[i]);
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(ds_full(db), lane);
      }
      if (!ok || !(ok = warp_wait(acc_full, ic & 1, c, A.err, lane))) break;
      tc_fence_after();
      const int64_t grow = b * A.s + iq * TR + r;
      const int64_t gcol = t * A.d;
      const int64_t br = grow / A.qkv.bh, bc = gcol / A.qkv.bw;
      bf16* dst = dqkv + A.qkv.block_base((int32_t)br, (int32_t)bc) + (grow - br * A.qkv.bh) * A.qkv.bw +
                  (gcol - bc * A.qkv.bw);
      const float inv_sigma = 1.0f / sigma;  // dQ was accumulated from sigma dS
      for (int cc = cgp; cc < (int)(A.d / 32); cc += kBwdWpq) {  // this warp's 32-column chunks of d
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_row(tmem, quarter, 256u + cc * 32), v);
        tmem_ld_wait();
        store_row32(dst + cc * 32, v, inv_sigma);
      }
      tc_fence_before();
      warp_arrive(acc_empty, lane);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// delta[z*s + r] = sum over the head's d columns of dO * O.  One warp per
// token row: 16-byte loads, 256 columns (every head in them) per step, four
// steps in flight; the G = d/8 lanes that hold one head reduce with shuffles.
// 64 registers let four CTAs share an SM, so a grid of one row per warp is
// resident at once.  Index arithmetic in 32 bits (the launcher checks that
// the extents fit).
// The same pass takes dmax0 = max over rows and heads of |dO_r|^2 for the
// bound that scales the score gradients (ds_sigma): each warp keeps a
// running maximum, the CTA combines its warps' in shared memory and takes
// one atomic max (non-negative floats order as their bits; zero on entry).
template <int G>
__global__ void __launch_bounds__(256, 4) attn_delta_kernel(const AttnProblem A, const bf16* __restrict__ O,
                                                            const bf16* __restrict__ dO, float* __restrict__ delta,
                                                            unsigned* __restrict__ dmax0) {
  constexpr int U = 4;
  __shared__ float red[8];
  const int lane = threadIdx.x & 31;
  const uint32_t M = (uint32_t)(A.Z / A.H * A.s);  // token rows
  const uint32_t s_len = (uint32_t)A.s, bh = (uint32_t)A.o.bh, bw = (uint32_t)A.o.bw, h = (uint32_t)A.h;
  const uint32_t nw = gridDim.x * 8u;
  float mdo = 0.0f;
  for (uint32_t tok = blockIdx.x * 8u + (threadIdx.x >> 5); tok < M; tok += nw) {
    const uint32_t b = tok / s_len, rr = tok - b * s_len;
    const uint32_t br = tok / bh, rin = tok - br * bh;
#pragma unroll 1
    for (uint32_t c0 = 0; c0 < h; c0 += 256u * U) {
      uint4 a[U], g[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t col = c0 + u * 256u + lane * 8u;
        if (col < h) {
          const uint32_t bc = col / bw;
          const int64_t off = A.o.block_base((int32_t)br, (int32_t)bc) + (int64_t)rin * bw + (col - bc * bw);
          a[u] = __ldg(reinterpret_cast<const uint4*>(O + off));
          g[u] = __ldg(reinterpret_cast<const uint4*>(dO + off));
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t col = c0 + u * 256u + lane * 8u;
        float acc = 0.0f, sg = 0.0f;
        if (col < h) {
          const __nv_bfloat162* ah = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
          const __nv_bfloat162* gh = reinterpret_cast<const __nv_bfloat162*>(&g[u]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(ah[e]), y = __bfloat1622float2(gh[e]);
            acc += x.x * y.x + x.y * y.y;
            sg += y.x * y.x + y.y * y.y;
          }
        }
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) {
          acc += __shfl_xor_sync(0xffffffffu, acc, o);
          sg += __shfl_xor_sync(0xffffffffu, sg, o);
        }
        if ((lane & (G - 1)) == 0 && col < h)
          delta[((int64_t)b * A.H + col / (uint32_t)A.d) * s_len + rr] = acc;
        mdo = fmaxf(mdo, sg);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mdo = fmaxf(mdo, __shfl_xor_sync(0xffffffffu, mdo, o));
  if (lane == 0) red[threadIdx.x >> 5] = mdo;
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 1; k < 8; ++k) mdo = fmaxf(mdo, red[k]);
    atomicMax(dmax0, __float_as_uint(mdo));
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// box of 64 columns x 128 rows over a bf16 matrix grid
tp3d_status tile_map(CUtensorMap* m, const Grid& g, const void* ptr) {
  auto fn = encode();
  if (!fn) return TP3D_ECUDA;
  cuuint64_t dims[3] = {(cuuint64_t)g.bw, (cuuint64_t)g.bh, (cuuint64_t)g.nshards()};
  cuuint64_t strides[2] = {(cuuint64_t)g.bw * 2, (cuuint64_t)(g.bh * g.bw * 2)};
  cuuint32_t box[3] = {64, TR, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TP3D_OK : TP3D_ECUDA;
}

tp3d_status check(const AttnProblem& A) {
  if (A.d != 64 && A.d != 128) return TP3D_EUNSUPPORTED;
  if (A.qkv.R > INT32_MAX || A.qkv.C > INT32_MAX || A.o.R > INT32_MAX || A.o.C > INT32_MAX) return TP3D_EUNSUPPORTED;
  if (A.s % TR || A.qkv.bh % TR || A.o.bh % TR || A.qkv.bw % A.d || A.o.bw % A.d) return TP3D_EUNSUPPORTED;
  if (A.Z * (A.s / TR) > 0x7fffffff) return TP3D_EUNSUPPORTED;
  return TP3D_OK;
}

}  // namespace

tp3d_status launch_attn_fwd(const tp3d_ctx* ctx, const AttnProblem& A, const void* qkv, void* o, float* lse,
                            cudaStream_t s) {
  TP3D_TRY(check(A));
  CUtensorMap mq;
  TP3D_TRY(tile_map(&mq, A.qkv, qkv));
  TP3D_CUDA_TRY(cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
  // setmaxnreg.inc waits until the block's launch registers cover the split
  cudaFuncAttributes fa;
  TP3D_CUDA_TRY(cudaFuncGetAttributes(&fa, attn_fwd_kernel));
  if (fa.numRegs * kFwdThreads < 128 * kFwdRegsLow + 256 * kFwdRegsHigh) return TP3D_EUNSUPPORTED;
  const int64_t items = A.Z * ((A.s / TR + 1) / 2);  // pairs of query tiles
  const unsigned grid = (unsigned)(items < ctx->num_sms ? items : ctx->num_sms);
  attn_fwd_kernel<<<grid, kFwdThreads, kSmem, s>>>(mq, A, static_cast<bf16*>(o), lse);
  return cudaGetLastError() == cudaSuccess ? TP3D_OK : TP3D_ECUDA;
}

tp3d_status launch_attn_bwd(const tp3d_ctx* ctx, const AttnProblem& A, const void* qkv, const void* o,
                            const void* dO, const float* lse, float* delta, unsigned* dmax, void* dqkv,
                            cudaStream_t s) {
  TP3D_TRY(check(A));
  // the dK/dV kernel copies 128-row runs of lse and delta with bulk copies
  if ((reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(delta)) & 15u) return TP3D_EALIGN;
  CUtensorMap mq, mo;
  TP3D_TRY(tile_map(&mq, A.qkv, qkv));
  TP3D_TRY(tile_map(&mo, A.o, dO));
  const int64_t tokens = A.Z / A.H * A.s;
  int64_t dgrid = (tokens + 7) / 8;
  if (dgrid > (int64_t)ctx->num_sms * 8) dgrid = (int64_t)ctx->num_sms * 8;
  TP3D_CUDA_TRY(cudaMemsetAsync(dmax, 0, sizeof(unsigned), s));  // dmax[0]; dmax[1] came with Q, K, V
  const bf16 *ob = static_cast<const bf16*>(o), *gb = static_cast<const bf16*>(dO);
  if (A.d == 128)
    attn_delta_kernel<16><<<(unsigned)dgrid, 256, 0, s>>>(A, ob, gb, delta, dmax);
  else
    attn_delta_kernel<8><<<(unsigned)dgrid, 256, 0, s>>>(A, ob, gb, delta, dmax);
  TP3D_CUDA_TRY(cudaGetLastError());
  TP3D_CUDA_TRY(cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
  TP3D_CUDA_TRY(cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
  const int64_t items = A.Z * (A.s / TR);
  const unsigned grid = (unsigned)(items < ctx->num_sms ? items : ctx->num_sms);
  attn_bwd_dkdv_kernel<<<grid, kBwdThreads, kSmem, s>>>(mq, mo, A, lse, delta, dmax, static_cast<bf16*>(dqkv));
  TP3D_CUDA_TRY(cudaGetLastError());
  attn_bwd_dq_kernel<<<grid, kBwdThreads, kSmem, s>>>(mq, mo, A, lse, delta, dmax, static_cast<bf16*>(dqkv));
  return cudaGetLastError() == cudaSuccess ? TP3D_OK : TP3D_ECUDA;
}

}  // namespace tp3d
