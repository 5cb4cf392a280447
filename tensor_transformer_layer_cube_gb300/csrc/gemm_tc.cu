// gemm_tc.cu - the sharded, batched bf16 GEMM on the sm_103a tensor cores.
//
// Persistent, warp-specialised kernel, one CTA per SM:
//   warp 0      TMA producer: 3-D tensor maps (shard column, shard row,
//               shard number) read each operand tile straight out of the shard
//               that holds it - the all-gathers of "Maximizing Parallelism in
//               Distributed Training for Huge Neural Networks", Algorithm 1,
//               become coordinates.  128-byte swizzle, STAGES-deep ring.
//   warp 1      MMA issuer: tcgen05.mma kind::f16 (bf16 x bf16 -> fp32) with
//               the accumulator in tensor memory; the contraction loop runs
//               over every depth index l in ascending order into the same
//               accumulator (the reduce-scatter over z of Algorithm 1).
//               Two accumulators alternate so the epilogue of one tile
//               overlaps the products of the next.  Also owns TMEM alloc.
//   warps 2-9   epilogue: tcgen05.ld of the 128 x BN fp32 tile, scale, bias
//               (Algorithm 7's b_j), GELU / GELU-backward, residual, bf16 or
//               fp32 stores into the output's shards.
// Every mbarrier wait is bounded (see common.cuh); a wait that runs out sets
// the context's error word, the CTA drains what it issued and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm.cuh"

namespace tp3d {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kEpiWarps = 8;                      // two per TMEM lane quarter
constexpr int kThreads = 32 * (2 + kEpiWarps);

template <int BN>
struct TcCfg {
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int STAGE_OUT = 4096;  // per epilogue warp: 32 rows x 128 bytes of output staging
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = STAGES * STAGE_BYTES + kEpiWarps * STAGE_OUT + BAR_BYTES + 1024;
};

struct TileInfo {
  int32_t z;
  int64_t m0, n0, m_end, n_end;  // per-batch logical coordinates; *_end = segment end
};

__device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <int BN>
__device__ __forceinline__ void decode_tile(const GemmProblem& P, int64_t t, TileInfo& T) {
  const int64_t tpsM = ceil_div(P.segM, BM), tpsN = ceil_div(P.segN, BN);
  const int64_t tiles_m = (P.M / P.segM) * tpsM, tiles_n = (P.N / P.segN) * tpsN;
  const int64_t per_z = tiles_m * tiles_n;
  T.z = (int32_t)(t / per_z);
  const int64_t r = t - (int64_t)T.z * per_z;
  const int64_t tn = r / tiles_m, tm = r - tn * tiles_m;
  const int64_t sm = tm / tpsM, sn = tn / tpsN;
  T.m0 = sm * P.segM + (tm - sm * tpsM) * BM;
  T.n0 = sn * P.segN + (tn - sn * tpsN) * BN;
  T.m_end = sm * P.segM + P.segM;
  T.n_end = sn * P.segN + P.segN;
}

template <int BN>
__device__ __forceinline__ int64_t total_tiles(const GemmProblem& P) {
  return (int64_t)P.Z * (P.M / P.segM) * ceil_div(P.segM, BM) * (P.N / P.segN) * ceil_div(P.segN, BN);
}

template <int BN>
__device__ __forceinline__ bool tile_skipped(const GemmProblem& P, const TileInfo& T) {
  return P.causal == CAUSAL_SKIP_UPPER && T.n0 > T.m0 + BM - 1;
}

// Contraction tiles start at k0 = segment * segK + kt * BK (kt < ceil(segK / BK)).
// A tile needs the k0 in [klo, khi): all of them, or the causal part.
__device__ __forceinline__ void k_bounds(const GemmProblem& P, const TileInfo& T, int64_t& klo, int64_t& khi) {
  klo = 0;
  khi = P.K;
  if (P.causal == CAUSAL_K_LE_M) khi = T.m0 + BM < P.K ? T.m0 + BM : P.K;
  if (P.causal == CAUSAL_K_GE_M) klo = T.m0 - BK + 1;
}

__device__ __forceinline__ bool tile_has_k(const GemmProblem& P, int64_t klo, int64_t khi, int32_t nsegK,
                                           int32_t tpsK) {
  for (int32_t sg = 0; sg < nsegK; ++sg) {
    const int64_t ks = (int64_t)sg * P.segK;
    const int64_t kt0 = klo > ks ? (klo - ks + BK - 1) / BK : 0;
    if (kt0 < tpsK && ks + kt0 * BK < khi) return true;
  }
  return false;
}

// block (br, bc) of an operand -> shard number, or one past the last shard
// (a TMA coordinate that reads zeros) when the block lies outside the matrix
__device__ __forceinline__ int shard_or_oob(const Grid& g, int64_t br, int64_t bc) {
  return (br < g.rb && bc < g.cb) ? g.shard((int32_t)br, (int32_t)bc) : g.nshards();
}
// The same with shifts where the cube edge q is a power of two (qs = log2 q;
// qs < 0: Grid::shard's divisions)
__device__ __forceinline__ int shard_or_oob_q(const Grid& g, int32_t br, int32_t bc, int qs) {
  if (br >= g.rb || bc >= g.cb) return g.nshards();
  if (qs < 0) return g.shard(br, bc);
  const int32_t qm = (1 << qs) - 1;
  switch (g.kind) {
    case TP3D_CUBE_A: return (br << qs) + bc;
    case TP3D_CUBE_B: return ((((bc & qm) << qs) + (bc >> qs)) << qs) + br;
    case TP3D_CUBE_C: return ((((br >> qs) << qs) + bc) << qs) + (br & qm);
    case TP3D_CUBE_B_SWAP: return ((((bc & qm) << qs) + br) << qs) + (bc >> qs);
    default: return g.shard(br, bc);
  }
}
__device__ __forceinline__ int log2_if_pow2(int q) { return (q > 0 && (q & (q - 1)) == 0) ? __ffs(q) - 1 : -1; }

__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// GELU(x) = x Phi(x), Phi(x) = (1 + erf(x / sqrt 2)) / 2, with erf from
// Abramowitz and Stegun, "Handbook of Mathematical Functions", formula
// 7.1.26 (Hastings' rational approximation, |error| <= 1.5e-7 for z >= 0):
//   erf(z) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2),
//   t = 1 / (1 + p z),
// extended to z < 0 by odd symmetry.  The lower tail Phi(x) = erfc(|x| / sqrt 2) / 2
// (x < 0) is taken directly, without the cancellation of 1 - erf; the 1/2
// rides in the coefficients (exact: a power of two).  exp(-z^2) is
// 2^(-z^2 log2 e) on the special-function unit, and is also the Gaussian
// density the backward needs.  Branch-free: one reciprocal and one
// exponential per element.
//
// Two forms, with the same operations in the same order (so the same bits):
// one value at a time, and two at once on the paired fp32 pipe (fma / mul
// .f32x2: one instruction for both halves), which the epilogue's fast path
// uses - GELU is bound by instruction issue there.
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
namespace gelu_c {
constexpr float kRsqrt2 = 0.70710678118654752f, kP = 0.3275911f, kNegLog2e = -1.44269504088896341f;
constexpr float kA1 = 0.5f * 0.254829592f, kA2 = 0.5f * -0.284496736f, kA3 = 0.5f * 1.421413741f,
                kA4 = 0.5f * -1.453152027f, kA5 = 0.5f * 1.061405429f;
constexpr float kRsqrt2pi = 0.39894228040143268f;
}  // namespace gelu_c
__device__ __forceinline__ float gauss_cdf(float x, float& e) {
  using namespace gelu_c;
  const float z = fabsf(x) * kRsqrt2;
  const float t = rcp_approx(fmaf(z, kP, 1.0f));
  float p = fmaf(t, kA5, kA4);
  p = fmaf(t, p, kA3);
  p = fmaf(t, p, kA2);
  p = fmaf(t, p, kA1);
  e = ex2_approx(z * (z * kNegLog2e));
  const float tail = (p * t) * e;  // erfc(|x| / sqrt 2) / 2
  return x < 0.0f ? tail : fmaf(tail, -1.0f, 1.0f);
}
__device__ __forceinline__ float gelu_f(float x) {
  float e;
  return x * gauss_cdf(x, e);
}
__device__ __forceinline__ float gelu_grad_f(float x) {
  float e;
  const float cdf = gauss_cdf(x, e);
  return fmaf(x * gelu_c::kRsqrt2pi, e, cdf);  // Phi(x) + x phi(x)
}

// two fp32 values in one 64-bit register pair
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk2(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(f32x2 v, float& a, float& b) { asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v)); }
__device__ __forceinline__ f32x2 splat2(float a) { return pk2(a, a); }
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// gauss_cdf of both halves of X: the cdfs and exp(-x^2 / 2)
__device__ __forceinline__ void gauss_cdf2(f32x2 X, f32x2& C, f32x2& E) {
  using namespace gelu_c;
  const f32x2 Z = mul2(X & 0x7fffffff7fffffffull, splat2(kRsqrt2));
  float d0, d1;
  upk2(fma2(Z, splat2(kP), splat2(1.0f)), d0, d1);
  const f32x2 T = pk2(rcp_approx(d0), rcp_approx(d1));
  f32x2 Pp = fma2(T, splat2(kA5), splat2(kA4));
  Pp = fma2(T, Pp, splat2(kA3));
  Pp = fma2(T, Pp, splat2(kA2));
  Pp = fma2(T, Pp, splat2(kA1));
  float q0, q1;
  upk2(mul2(Z, mul2(Z, splat2(kNegLog2e))), q0, q1);
  E = pk2(ex2_approx(q0), ex2_approx(q1));
  const f32x2 TL = mul2(mul2(Pp, T), E);
  float t0, t1, o0, o1, x0, x1;
  upk2(TL, t0, t1);
  upk2(fma2(TL, splat2(-1.0f), splat2(1.0f)), o0, o1);
  upk2(X, x0, x1);
  C = pk2(x0 < 0.0f ? t0 : o0, x1 < 0.0f ? t1 : o1);
}
// x[e], x[e + 1] = GELU of themselves
__device__ __forceinline__ void gelu_pair(float& a, float& b) {
  const f32x2 X = pk2(a, b);
  f32x2 C, E;
  gauss_cdf2(X, C, E);
  upk2(mul2(X, C), a, b);
}
// a, b *= GELU'(za), GELU'(zb)
__device__ __forceinline__ void gelu_grad_mul_pair(float za, float zb, float& a, float& b) {
  const f32x2 Zv = pk2(za, zb);
  f32x2 C, E;
  gauss_cdf2(Zv, C, E);
  const f32x2 G = fma2(mul2(Zv, splat2(gelu_c::kRsqrt2pi)), E, C);
  upk2(mul2(pk2(a, b), G), a, b);
}
// x[0..7] (+)= and *= on pairs
__device__ __forceinline__ void add8_pairs(float* x, const float* y) {
#pragma unroll
  for (int e = 0; e < 8; e += 2) upk2(add2(pk2(x[e], x[e + 1]), pk2(y[e], y[e + 1])), x[e], x[e + 1]);
}
__device__ __forceinline__ void scale8_pairs(float* x, float s) {
#pragma unroll
  for (int e = 0; e < 8; e += 2) upk2(mul2(pk2(x[e], x[e + 1]), splat2(s)), x[e], x[e + 1]);
}

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float* f) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return v;
}
// max over the warp, then one atomic max (non-negative floats order as their bits)
__device__ __forceinline__ void warp_amax(float m, unsigned* out, int lane) {
  if (!out) return;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) atomicMax(out, __float_as_uint(m));
}
// fp16 form; a value beyond fp16's finite range raises TP3D_ERANGE
__device__ __forceinline__ uint4 pack8h(const float* f, int* err) {
  uint4 v;
  __half2* h = reinterpret_cast<__half2*>(&v);
  float mx = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
    mx = fmaxf(mx, fmaxf(fabsf(f[2 * i]), fabsf(f[2 * i + 1])));
  }
  if (mx > kHalfMax) raise_error(err, TP3D_ERANGE);
  return v;
}


// arrive on a peer's mbarrier without a memory release: what it orders is the
// warp's tensor-memory reads, which tcgen05.fence::before_thread_sync covers
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// One tile's epilogue for the calling epilogue warp (32 rows x BN/2 columns
// of the tile's TMEM accumulator `buf`).  Warp w may read TMEM lanes
// 32*(w%4) .. +31 only: two warps share each lane quarter (= 32 rows of the
// tile) and split its columns in halves, 32 columns per chunk.
// A chunk inside the tile's segment (the common case) takes the fast path:
//  - the residual or GELU input comes by TMA into the second half of the
//    warp's staging buffer; the next chunk's load is issued as soon as this
//    one has been read, so its latency hides behind the arithmetic;
//  - the results are computed into registers first, then (once the previous
//    TMA store has finished reading the staging buffer) written there with
//    the 64-byte (bf16) or 128-byte (fp32) swizzle and sent out by one TMA
//    store per output.
// A chunk crossing the segment's edge is written element-wise under a mask.
// After its last TMEM load the warp arrives on `tempty` (in the peer CTA when
// `tempty_remote`, a shared::cluster address).
// H16: the problem has fp16 output columns or a device-resident scale
// (instantiated apart, so the plain epilogue's code is left as it is: its
// speed answers to code layout).
// The TMA load of the auxiliary input's first chunk for this warp (the
// coordinates epilogue_tile computes for it), issued before the tile's
// accumulator is ready so that its latency hides behind the contraction.
// Returns whether it was issued: the problem has an auxiliary input and the
// chunk takes the fast path.  The staging half it fills is free: the warp
// read the previous tile's last chunk from it before leaving that tile.
template <int BN>
__device__ __forceinline__ bool aux_prefetch(const GemmProblem& P, const TileInfo& T, int warp, int lane,
                                             uint8_t* stg, const CUtensorMap* mapX, uint32_t aux_bar) {
  const void* aux = P.epi.resid ? P.epi.resid : P.epi.gin;
  if (aux == nullptr || P.epi.zsave != nullptr || P.epi.out_f32) return false;
  constexpr int CH = BN / 64;
  const int quarter = warp & 3, half = (warp - 2) >> 2;
  const int64_t n = T.n0 + (int64_t)(half * CH) * 32;
  if (!(T.m0 + quarter * 32 + 31 < T.m_end && n + 32 <= T.n_end)) return false;
  const Grid& cg = P.c.g;
  const int64_t gm = T.m0 + quarter * 32 + lane + op_off(P.c.hi1, P.c.lo1, P.c.base1, T.z, P.Hz);
  const int64_t gn0 = T.n0 + op_off(P.c.hi2, P.c.lo2, P.c.base2, T.z, P.Hz);
  const int64_t cbr = (uint32_t)(gm - lane) / (uint32_t)cg.bh, cbc = (uint32_t)gn0 / (uint32_t)cg.bw;
  if (lane == 0) {
    mbar_arrive_expect_tx(aux_bar, 2048u);
    tma_load_3d(smem_u32(stg) + 2048u, mapX, aux_bar, (int)(gn0 + (n - T.n0) - cbc * cg.bw),
                (int)(gm - lane - cbr * cg.bh), cg.shard((int32_t)cbr, (int32_t)cbc));
  }
  return true;
}

template <int BN, bool H16>
__device__ __forceinline__ void epilogue_tile(const GemmProblem& P, const TileInfo& T, bool any_k, int buf,
                                              uint32_t tmem_base, int warp, int lane, uint8_t* stg,
                                              const CUtensorMap* mapC, const CUtensorMap* mapZ,
                                              const CUtensorMap* mapX, uint32_t aux_bar, uint32_t& aux_phase,
                                              volatile int* abort_flag, uint32_t tempty, bool tempty_remote,
                                              uint32_t& stores, float& cmax, bool aux0_issued = false) {
  const void* aux = P.epi.resid ? P.epi.resid : P.epi.gin;
  const bool aux_ok = aux != nullptr && P.epi.zsave == nullptr && !P.epi.out_f32;
  const int quarter = warp & 3;
  const int half = (warp - 2) >> 2;
  const int row = quarter * 32 + lane;
  constexpr int CH = BN / 64;  // 32-column chunks per warp
  const Grid& cg = P.c.g;
  const bool f32 = P.epi.out_f32 != 0;
  const uint32_t stg_y = smem_u32(stg), stg_z = stg_y + 2048u;
  const int64_t m = T.m0 + row;
  const bool row_ok = m < T.m_end;
  const bool rows_full = T.m0 + quarter * 32 + 31 < T.m_end;
  const int64_t gm = m + op_off(P.c.hi1, P.c.lo1, P.c.base1, T.z, P.Hz);
  const int64_t gn0 = T.n0 + op_off(P.c.hi2, P.c.lo2, P.c.base2, T.z, P.Hz);
  // 32-bit divisions (every launcher checks the extents)
  const int64_t cbr = (uint32_t)(gm - lane) / (uint32_t)cg.bh, cbc = (uint32_t)gn0 / (uint32_t)cg.bw;  // C block of the warp's rows
  const int c1 = (int)(gm - lane - cbr * cg.bh);
  const int c2 = cg.shard((int32_t)cbr, (int32_t)cbc);
  int64_t row_base = 0;
  if (row_ok) {
    const int64_t br = (uint32_t)gm / (uint32_t)cg.bh;
    row_base = cg.block_base((int32_t)br, (int32_t)cbc) + (gm - br * cg.bh) * cg.bw + (gn0 - cbc * cg.bw);
  }
  auto chunk_n = [&](int cc) { return T.n0 + (half * CH + cc) * 32; };
  auto fast = [&](int cc) { return rows_full && chunk_n(cc) + 32 <= T.n_end; };
  auto chunk_c0 = [&](int cc) { return (int)(gn0 + (chunk_n(cc) - T.n0) - cbc * cg.bw); };
  auto aux_issue = [&](int cc) {
    if (lane == 0) {
      mbar_arrive_expect_tx(aux_bar, 2048u);
      tma_load_3d(stg_z, mapX, aux_bar, chunk_c0(cc), c1, c2);
    }
  };
  if (aux_ok && fast(0) && !aux0_issued) aux_issue(0);  // else issued before the accumulator wait
  const __nv_bfloat16* bias = static_cast<const __nv_bfloat16*>(P.epi.bias);
  const float alpha = H16 && P.epi.alpha_dev ? P.epi.alpha * *P.epi.alpha_dev : P.epi.alpha;
  const bool scaled = alpha != 1.0f;
#pragma unroll 1
  for (int cc = 0; cc < CH; ++cc) {
    const int ch = half * CH + cc;
    uint32_t r[32];
    tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * BN + ch * 32), r);
    // the chunk's 32 bias values (the same for every lane) load under the TMEM read
    uint4 bv[4];
    if (bias && chunk_n(cc) + 32 <= T.n_end) {
#pragma unroll
      for (int v = 0; v < 4; ++v) bv[v] = *reinterpret_cast<const uint4*>(bias + (gn0 + (chunk_n(cc) - T.n0) + v * 8));
    }
    tmem_ld_wait();
    if (cc == CH - 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (tempty_remote)
          mbar_arrive_remote_relaxed(tempty);
        else
          mbar_arrive(tempty);
      }
    }
    const int64_t n = chunk_n(cc);
    if (n >= T.n_end) continue;
    // fp16 output for the chunk's 32 columns (the bound is a multiple of 32)
    const bool h16 = H16 && gn0 + (n - T.n0) < P.epi.f16_cols;
    if (fast(cc)) {
      // ---------------------------------------------------------- fast path
      // sv: the auxiliary input read from staging, or the pre-activation to
      // save (a problem never has both)
      uint4 sv[4];
      if (aux_ok) {
        bool ok = lane == 0 ? mbar_wait(aux_bar, aux_phase & 1u, abort_flag, P.err) : false;
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) {
          // the load into the staging buffer may still be in flight: let it land first
          if (lane == 0) mbar_wait_drain(aux_bar, aux_phase & 1u);
          __syncwarp();
          return;
        }
        ++aux_phase;
#pragma unroll
        for (int v = 0; v < 4; ++v)
          sv[v] = *reinterpret_cast<const uint4*>(stg + 2048 + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4));
        __syncwarp();
        if (cc + 1 < CH && fast(cc + 1)) aux_issue(cc + 1);
      }
      // bf16 output without an auxiliary input or saved pre-activation uses
      // both 2 KiB halves of the staging buffer in turn
      const bool dbl = !aux_ok && P.epi.zsave == nullptr && !f32;
      uint8_t* ybuf = stg + (dbl ? (stores & 1u) * 2048u : 0u);
      uint4 yv[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = any_k ? __uint_as_float(r[v * 8 + e]) : 0.0f;
        // the arithmetic on pairs of columns (the paired fp32 pipe)
        if (scaled) scale8_pairs(x, alpha);
        if (bias) {
          float bb[8];
          unpack8(bv[v], bb);
          add8_pairs(x, bb);
        }
        if (P.epi.zsave) sv[v] = pack8(x);
        if (P.epi.act == EPI_GELU) {
#pragma unroll
          for (int e = 0; e < 8; e += 2) gelu_pair(x[e], x[e + 1]);
        } else if (P.epi.act == EPI_GELU_BWD) {
          float zz[8];
          unpack8(sv[v], zz);
#pragma unroll
          for (int e = 0; e < 8; e += 2) gelu_grad_mul_pair(zz[e], zz[e + 1], x[e], x[e + 1]);
        }
        if (P.epi.resid) {
          float rr[8];
          unpack8(sv[v], rr);
          add8_pairs(x, rr);
        }
        if (!f32) {
          yv[v] = h16 ? pack8h(x, P.err) : pack8(x);
          if (H16 && !h16) {
#pragma unroll
            for (int e = 0; e < 8; ++e) cmax = fmaxf(cmax, fabsf(x[e]));
          }
        } else {
          // fp32: each 16-column half (two groups) goes out by its own TMA
          // store from the staging half the store before last used
          if ((v & 1) == 0 && stores) {
            if (lane == 0) bulk_wait_read_1();
            __syncwarp();
          }
          uint8_t* hb = stg + (stores & 1u) * 2048u;
          const int u0 = 2 * (v & 1);
          *reinterpret_cast<float4*>(hb + lane * 64 + ((u0 ^ ((lane >> 1) & 3)) << 4)) = make_float4(x[0], x[1], x[2], x[3]);
          *reinterpret_cast<float4*>(hb + lane * 64 + (((u0 + 1) ^ ((lane >> 1) & 3)) << 4)) =
              make_float4(x[4], x[5], x[6], x[7]);
          if (v & 1) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(mapC, smem_u32(hb), chunk_c0(cc) + 16 * (v >> 1), c1, c2);
              bulk_commit();
            }
            ++stores;
          }
        }
      }
      if (f32) continue;  // stored half by half above
      if (!f32) {
        if (stores) {
          // double-buffered: the store that last used this half was issued two chunks ago
          if (lane == 0) {
            if (dbl)
              bulk_wait_read_1();
            else
              bulk_wait_read_all();
          }
          __syncwarp();
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) *reinterpret_cast<uint4*>(ybuf + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4)) = yv[v];
        if (P.epi.zsave) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            *reinterpret_cast<uint4*>(stg + 2048 + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4)) = sv[v];
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(mapC, smem_u32(ybuf), chunk_c0(cc), c1, c2);
        if (P.epi.zsave) tma_store_3d(mapZ, stg_z, chunk_c0(cc), c1, c2);
        bulk_commit();
      }
      ++stores;
    } else if (row_ok) {
      // ---------------------------------------------------------- masked path
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int64_t nv = n + v * 8;
        if (nv >= T.n_end) break;
        const int64_t off = row_base + (nv - T.n0);
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = any_k ? __uint_as_float(r[v * 8 + e]) * alpha : 0.0f;
        if (bias) {
          float bb[8];
          unpack8(*reinterpret_cast<const uint4*>(bias + (gn0 + (nv - T.n0))), bb);
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] += bb[e];
        }
        if (P.epi.zsave) *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(P.epi.zsave) + off) = pack8(x);
        if (P.epi.act == EPI_GELU) {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = gelu_f(x[e]);
        } else if (P.epi.act == EPI_GELU_BWD) {
          float zz[8];
          unpack8(*reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(P.epi.gin) + off), zz);
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] *= gelu_grad_f(zz[e]);
        }
        if (P.epi.resid) {
          float rr[8];
          unpack8(*reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(P.epi.resid) + off), rr);
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] += rr[e];
        }
        if (!f32) {
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(const_cast<void*>(P.c.ptr)) + off) =
              h16 ? pack8h(x, P.err) : pack8(x);
          if (H16 && !h16) {
#pragma unroll
            for (int e = 0; e < 8; ++e) cmax = fmaxf(cmax, fabsf(x[e]));
          }
        } else {
          float4* o = reinterpret_cast<float4*>(static_cast<float*>(const_cast<void*>(P.c.ptr)) + off);
          o[0] = make_float4(x[0], x[1], x[2], x[3]);
          o[1] = make_float4(x[4], x[5], x[6], x[7]);
        }
      }
    }
  }
}

template <int BN, bool H16>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapC, const __grid_constant__ CUtensorMap mapZ,
                   const __grid_constant__ CUtensorMap mapX, const GemmProblem P) {
  using Cfg = TcCfg<BN>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint8_t* stage_out = base_ptr + S * Cfg::STAGE_BYTES;  // kEpiWarps x 4 KiB, 1024-aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage_out + kEpiWarps * Cfg::STAGE_OUT);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * S + 5 + kEpiWarps);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t final_bar = bar0 + 8u * (2 * S + 4);
  auto aux_bar = [&](int ew) { return bar0 + 8u * (2 * S + 5 + ew); };  // one per epilogue warp
  auto a_stage = [&](int s) { return base + (uint32_t)(s * Cfg::A_BYTES); };
  auto b_stage = [&](int s) { return base + (uint32_t)(S * Cfg::A_BYTES + s * Cfg::B_BYTES); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), kEpiWarps);
    }
    mbar_init(final_bar, 1);
    for (int e = 0; e < kEpiWarps; ++e) mbar_init(aux_bar(e), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&mapA);
    tma_prefetch_map(&mapB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int64_t ntiles = total_tiles<BN>(P);
  const int32_t segK = (int32_t)P.segK;
  const int32_t tpsK = (segK + BK - 1) / BK;
  const int32_t nsegK = (int32_t)(P.K / P.segK);
  const bool a_mn = P.a.mn_major != 0, b_mn = P.b.mn_major != 0;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      // Shard coordinates change only at contraction-segment boundaries, so
      // they are computed once per tile (the M / N side) and once per
      // segment (the K side); the inner loop only adds BK.
      uint32_t it = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        TileInfo T;
        decode_tile<BN>(P, t, T);
        if (tile_skipped<BN>(P, T)) continue;
        int64_t klo, khi;
        k_bounds(P, T, klo, khi);
        const int64_t am = T.m0 + op_off(P.a.hi1, P.a.lo1, P.a.base1, T.z, P.Hz);
        const int64_t ak = op_off(P.a.hi2, P.a.lo2, P.a.base2, T.z, P.Hz);
        const int64_t bk = op_off(P.b.hi1, P.b.lo1, P.b.base1, T.z, P.Hz);
        const int64_t bn = T.n0 + op_off(P.b.hi2, P.b.lo2, P.b.base2, T.z, P.Hz);
        // M / N side, fixed for the tile
        int64_t a_br = 0, b_br = 0;
        int a_c1 = 0, b_c1 = 0;
        int64_t a_bc[BM / 64], b_bc[BN / 64];
        int a_c0[BM / 64], b_c0[BN / 64];
        if (!a_mn) {
          a_br = am / P.a.g.bh;
          a_c1 = (int)(am - a_br * P.a.g.bh);
        } else {
#pragma unroll
          for (int h = 0; h < BM / 64; ++h) {
            a_bc[h] = (am + 64 * h) / P.a.g.bw;
            a_c0[h] = (int)(am + 64 * h - a_bc[h] * P.a.g.bw);
          }
        }
        if (!b_mn) {
          b_br = bn / P.b.g.bh;
          b_c1 = (int)(bn - b_br * P.b.g.bh);
        } else {
#pragma unroll
          for (int h = 0; h < BN / 64; ++h) {
            b_bc[h] = (bn + 64 * h) / P.b.g.bw;
            b_c0[h] = (int)(bn + 64 * h - b_bc[h] * P.b.g.bw);
          }
        }
        for (int32_t sg = 0; sg < nsegK && ok; ++sg) {
          const int64_t ks = (int64_t)sg * segK;
          if (ks >= khi) break;
          if (ks + segK <= klo) continue;
          // K side, fixed for the segment
          int a_k = 0, b_k = 0, a_sh = 0, b_sh = 0;
          int a_shh[BM / 64], b_shh[BN / 64];
          if (!a_mn) {
            const int64_t bc = (ak + ks) / P.a.g.bw;
            a_k = (int)(ak + ks - bc * P.a.g.bw);
            a_sh = shard_or_oob(P.a.g, a_br, bc);
          } else {
            const int64_t br = (ak + ks) / P.a.g.bh;
            a_k = (int)(ak + ks - br * P.a.g.bh);
#pragma unroll
            for (int h = 0; h < BM / 64; ++h) a_shh[h] = shard_or_oob(P.a.g, br, a_bc[h]);
          }
          if (!b_mn) {
            const int64_t bc = (bk + ks) / P.b.g.bw;
            b_k = (int)(bk + ks - bc * P.b.g.bw);
            b_sh = shard_or_oob(P.b.g, b_br, bc);
          } else {
            const int64_t br = (bk + ks) / P.b.g.bh;
            b_k = (int)(bk + ks - br * P.b.g.bh);
#pragma unroll
            for (int h = 0; h < BN / 64; ++h) b_shh[h] = shard_or_oob(P.b.g, br, b_bc[h]);
          }
          for (int32_t kt = 0; kt < tpsK; ++kt) {
            const int64_t k0 = ks + (int64_t)kt * BK;
            if (k0 < klo || k0 >= khi) continue;
            const int s = (int)(it % S);
            const uint32_t ph = (it / S) & 1u;
            // test hook: stop loading (and drain what is in flight, below)
            if (P.stall_after >= 0 && (int64_t)it >= P.stall_after) {
              ok = false;
              break;
            }
            if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, P.err)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(full_bar(s), Cfg::STAGE_BYTES);
            const int kofs = kt * BK;
            if (!a_mn) {
              tma_load_3d(a_stage(s), &mapA, full_bar(s), a_k + kofs, a_c1, a_sh);
            } else {
#pragma unroll
              for (int h = 0; h < BM / 64; ++h)
                tma_load_3d(a_stage(s) + h * 8192u, &mapA, full_bar(s), a_c0[h], a_k + kofs, a_shh[h]);
            }
            if (!b_mn) {
              tma_load_3d(b_stage(s), &mapB, full_bar(s), b_k + kofs, b_c1, b_sh);
            } else {
#pragma unroll
              for (int h = 0; h < BN / 64; ++h)
                tma_load_3d(b_stage(s) + h * 8192u, &mapB, full_bar(s), b_c0[h], b_k + kofs, b_shh[h]);
            }
            ++it;
          }
        }
      }
      if (!ok) {
        // drain: let every load this thread issued land before the CTA exits
        const uint32_t first = it > (uint32_t)S ? it - S : 0u;
        for (uint32_t j = first; j < it; ++j) mbar_wait_drain(full_bar((int)(j % S)), (j / S) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc = P.in_f16 ? idesc_f16_f32(BM, BN, a_mn ? 1 : 0, b_mn ? 1 : 0)
                                      : idesc_bf16_f32(BM, BN, a_mn ? 1 : 0, b_mn ? 1 : 0);
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        TileInfo T;
        decode_tile<BN>(P, t, T);
        if (tile_skipped<BN>(P, T)) continue;
        int64_t klo, khi;
        k_bounds(P, T, klo, khi);
        const int buf = (int)(tc & 1u);
        const uint32_t tph = (tc >> 1) & 1u;
        if (!mbar_wait(tempty_bar(buf), tph ^ 1u, abort_flag, P.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
        bool first = true;
        for (int32_t sg = 0; sg < nsegK && ok; ++sg) {
          const int64_t ks = (int64_t)sg * segK;
          if (ks >= khi) break;
          if (ks + segK <= klo) continue;
          for (int32_t kt = 0; kt < tpsK; ++kt) {
            const int64_t k0 = ks + (int64_t)kt * BK;
            if (k0 < klo || k0 >= khi) continue;
            const int s = (int)(it % S);
            const uint32_t ph = (it / S) & 1u;
            if (!mbar_wait(full_bar(s), ph, abort_flag, P.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int k16 = 0; k16 < BK / 16; ++k16) {
              const uint64_t ad = a_mn ? smem_desc_sw128(a_stage(s) + k16 * 2048u, 8192u, 1024u)
                                       : smem_desc_sw128(a_stage(s) + k16 * 32u, 16u, 1024u);
              const uint64_t bd = b_mn ? smem_desc_sw128(b_stage(s) + k16 * 2048u, 8192u, 1024u)
                                       : smem_desc_sw128(b_stage(s) + k16 * 32u, 16u, 1024u);
              umma_bf16(d_tmem, ad, bd, idesc, (first && k16 == 0) ? 0u : 1u);
            }
            first = false;
            umma_commit(empty_bar(s));
            ++it;
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(buf));
        ++tc;
      }
      // wait until every product this thread issued has finished before TMEM is freed
      umma_commit(final_bar);
      mbar_wait_drain(final_bar, 0);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    uint32_t tc = 0;
    uint32_t stores = 0;  // TMA stores this warp has issued from its staging buffer
    uint32_t aux_phase = 0;
    uint8_t* stg = stage_out + (warp - 2) * Cfg::STAGE_OUT;
    float cmax = 0.0f;  // H16: the largest |C| of the bf16 columns this warp stored
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
      TileInfo T;
      decode_tile<BN>(P, t, T);
      if (tile_skipped<BN>(P, T)) continue;
      int64_t klo, khi;
      k_bounds(P, T, klo, khi);
      const bool any_k = tile_has_k(P, klo, khi, nsegK, tpsK);
      const int buf = (int)(tc & 1u);
      const uint32_t tph = (tc >> 1) & 1u;
      const bool aux0 = aux_prefetch<BN>(P, T, warp, lane, stg, &mapX, aux_bar(warp - 2));
      // one lane waits and the warp follows it, so the warp stays converged
      // for the .sync.aligned tensor-memory loads
      bool ok = lane == 0 ? mbar_wait(tfull_bar(buf), tph, abort_flag, P.err) : false;
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) {
        if (aux0 && lane == 0) mbar_wait_drain(aux_bar(warp - 2), aux_phase & 1u);  // let the load land
        __syncwarp();
        break;
      }
      tc_fence_after();
      epilogue_tile<BN, H16>(P, T, any_k, buf, tmem_base, warp, lane, stg, &mapC, &mapZ, &mapX, aux_bar(warp - 2),
                             aux_phase, abort_flag, tempty_bar(buf), false, stores, cmax, aux0);
      ++tc;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    if (H16) warp_amax(cmax, P.epi.amax_out, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ CTA pairs
// The same GEMM on clusters of two CTAs (tcgen05 cta_group::2): a pair
// computes a 256 x 256 tile; CTA r of the pair holds rows [128 r, +128) of
// the A tile and columns [128 r, +128) of the B tile, the even CTA issues
// M = 256, N = 256 products that read A from each CTA's own shared memory and
// B from both, and each CTA's tensor memory receives its 128 rows.  Per SM
// this moves 32 KiB per contraction step instead of 48 KiB (B is loaded once
// per pair) and leaves room for a 6-deep ring.  Only for problems without a
// causal mask (both CTAs of a pair run the same contraction range).
//
// Barriers: full[s] lives in the even CTA and takes the even producer's
// expect-tx arrival for both CTAs' bytes plus both CTAs' TMA completions;
// empty[s] and tfull[b] live in each CTA and are arrived on by the even CTA's
// commits (multicast to both); tempty[b] lives in the even CTA and takes the
// arrivals of both CTAs' epilogue warps.
// KD: contraction depth of a stage, 64 (six stages) or 128 (three stages of
// 16 KiB boxes: fewer, larger TMA transfers for the same bytes in flight).
template <int KD>
struct Tc2Cfg {
  static constexpr int BN = 256;
  static constexpr int BKP = KD;
  static constexpr int STAGES = KD == 64 ? 6 : 3;
  static constexpr int A_BYTES = 128 * KD * 2;
  static constexpr int B_BYTES = 128 * KD * 2;  // this CTA's half of B
  static constexpr uint32_t KCHUNK = 128 * 128;  // one 64-column K-major chunk of 128 rows
  static constexpr uint32_t MNBOX = KD * 128;    // one 64-column MN-major box of KD rows
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 512;
  static constexpr int STAGE_OUT = 4096;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = STAGES * STAGE_BYTES + kEpiWarps * STAGE_OUT + BAR_BYTES + 1024;
};

// Tile t for CTA r of the pair.  32-bit arithmetic (the launcher checks that
// every extent and the tile count fit): a 64-bit division is a long software
// sequence, and this runs at every tile change of the producer.
__device__ __forceinline__ uint32_t udiv32(int64_t a, int64_t b) { return (uint32_t)a / (uint32_t)b; }
__device__ __forceinline__ void decode_pair_tile(const GemmProblem& P, int64_t t, uint32_t r, TileInfo& T) {
  const uint32_t segM = (uint32_t)P.segM, segN = (uint32_t)P.segN;
  const uint32_t tpsM = (segM + 255u) / 256u, tpsN = (segN + 255u) / 256u;
  const uint32_t tiles_m = udiv32(P.M, segM) * tpsM;
  const uint32_t per_z = tiles_m * udiv32(P.N, segN) * tpsN;
  const uint32_t tt = (uint32_t)t;
  const uint32_t z = tt / per_z;
  const uint32_t rem = tt - z * per_z;
  const uint32_t tn = rem / tiles_m, tm = rem - tn * tiles_m;
  const uint32_t sm = tm / tpsM, sn = tn / tpsN;
  T.z = (int32_t)z;
  T.m0 = (int64_t)sm * segM + (int64_t)(tm - sm * tpsM) * 256 + 128 * (int64_t)r;
  T.n0 = (int64_t)sn * segN + (int64_t)(tn - sn * tpsN) * 256;
  T.m_end = (int64_t)sm * segM + segM;
  T.n_end = (int64_t)sn * segN + segN;
}

__device__ __forceinline__ int64_t total_pair_tiles(const GemmProblem& P) {
  return (int64_t)P.Z * (P.M / P.segM) * ceil_div(P.segM, 256) * (P.N / P.segN) * ceil_div(P.segN, 256);
}

template <int KD, bool H16>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                    const __grid_constant__ CUtensorMap mapC, const __grid_constant__ CUtensorMap mapZ,
                    const __grid_constant__ CUtensorMap mapX, const GemmProblem P, const uint32_t wide) {
  using Cfg = Tc2Cfg<KD>;
  constexpr int S = Cfg::STAGES;
  constexpr int BKP = Cfg::BKP;
  constexpr int BN = Cfg::BN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint8_t* stage_out = base_ptr + S * Cfg::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage_out + kEpiWarps * Cfg::STAGE_OUT);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * S + 5 + kEpiWarps);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t final_bar = bar0 + 8u * (2 * S + 4);
  auto aux_bar = [&](int ew) { return bar0 + 8u * (2 * S + 5 + ew); };  // one per epilogue warp
  auto a_stage = [&](int s) { return base + (uint32_t)(s * Cfg::A_BYTES); };
  auto b_stage = [&](int s) { return base + (uint32_t)(S * Cfg::A_BYTES + s * Cfg::B_BYTES); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * kEpiWarps);
    }
    mbar_init(final_bar, 1);
    for (int e = 0; e < kEpiWarps; ++e) mbar_init(aux_bar(e), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_holder), Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&mapA);
    tma_prefetch_map(&mapB);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int64_t ntiles = total_pair_tiles(P);
  const int64_t nclusters = gridDim.x >> 1, cid = blockIdx.x >> 1;
  const int32_t segK = (int32_t)P.segK;
  const int32_t tpsK = (segK + BKP - 1) / BKP;
  const int32_t nsegK = (int32_t)(P.K / P.segK);
  const bool a_mn = P.a.mn_major != 0, b_mn = P.b.mn_major != 0;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      // Where a tile's operand boxes start (block row or columns and offsets
      // inside the block).  The next tile's are worked out while the current
      // tile's first stage is in flight, so a tile change costs no arithmetic.
      struct TileLd {
        int64_t ak, bk;
        int32_t a_br, b_br, a_c1, b_c1;
        int32_t a_bc[2], b_bc[2], a_c0[2], b_c0[2];
        int32_t a_k0, a_blk0, b_k0, b_blk0;  // segment 0: contraction offset in its block, and that block
      };
      auto setup = [&](int64_t t, TileLd& L) {
        TileInfo T;
        decode_pair_tile(P, t, rank, T);
        const int64_t am = T.m0 + op_off(P.a.hi1, P.a.lo1, P.a.base1, T.z, P.Hz);
        L.ak = op_off(P.a.hi2, P.a.lo2, P.a.base2, T.z, P.Hz);
        L.bk = op_off(P.b.hi1, P.b.lo1, P.b.base1, T.z, P.Hz);
        const int64_t bn = T.n0 + 128 * (int64_t)rank + op_off(P.b.hi2, P.b.lo2, P.b.base2, T.z, P.Hz);
        if (!a_mn) {
          L.a_br = (int32_t)udiv32(am, P.a.g.bh);
          L.a_c1 = (int32_t)(am - (int64_t)L.a_br * P.a.g.bh);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            L.a_bc[h] = (int32_t)udiv32(am + 64 * h, P.a.g.bw);
            L.a_c0[h] = (int32_t)(am + 64 * h - (int64_t)L.a_bc[h] * P.a.g.bw);
          }
        }
        if (!b_mn) {
          L.b_br = (int32_t)udiv32(bn, P.b.g.bh);
          L.b_c1 = (int32_t)(bn - (int64_t)L.b_br * P.b.g.bh);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            L.b_bc[h] = (int32_t)udiv32(bn + 64 * h, P.b.g.bw);
            L.b_c0[h] = (int32_t)(bn + 64 * h - (int64_t)L.b_bc[h] * P.b.g.bw);
          }
        }
        // the contraction's first segment: later segments step from it by segK
        // (which divides every block extent along the contraction)
        const int64_t akd = a_mn ? P.a.g.bh : P.a.g.bw, bkd = b_mn ? P.b.g.bh : P.b.g.bw;
        L.a_blk0 = (int32_t)udiv32(L.ak, akd);
        L.a_k0 = (int32_t)(L.ak - (int64_t)L.a_blk0 * akd);
        L.b_blk0 = (int32_t)udiv32(L.bk, bkd);
        L.b_k0 = (int32_t)(L.bk - (int64_t)L.b_blk0 * bkd);
      };
      const int qsa = log2_if_pow2(P.a.g.q), qsb = log2_if_pow2(P.b.g.q);
      const int32_t akd = (int32_t)(a_mn ? P.a.g.bh : P.a.g.bw), bkd = (int32_t)(b_mn ? P.b.g.bh : P.b.g.bw);
      uint32_t it = 0;
      bool ok = true;
      TileLd cur = {}, nxt = {};
      if (cid < ntiles) setup(cid, cur);
      for (int64_t t = cid; t < ntiles && ok; t += nclusters) {
        const int32_t a_br = cur.a_br, b_br = cur.b_br;
        const int a_c1 = cur.a_c1, b_c1 = cur.b_c1;
        const int32_t a_bc[2] = {cur.a_bc[0], cur.a_bc[1]}, b_bc[2] = {cur.b_bc[0], cur.b_bc[1]};
        const int a_c0[2] = {cur.a_c0[0], cur.a_c0[1]}, b_c0[2] = {cur.b_c0[0], cur.b_c0[1]};
        // the running segment: offset in the contraction block, and the block
        int32_t a_k = cur.a_k0, a_blk = cur.a_blk0, b_k = cur.b_k0, b_blk = cur.b_blk0;
        bool next_ready = false;
        for (int32_t sg = 0; sg < nsegK && ok; ++sg) {
          if (sg > 0) {  // step one segment (no division: segK divides the block extent)
            a_k += segK;
            if (a_k >= akd) {
              a_k -= akd;
              ++a_blk;
            }
            b_k += segK;
            if (b_k >= bkd) {
              b_k -= bkd;
              ++b_blk;
            }
          }
          int a_sh = 0, b_sh = 0;
          int a_shh[2], b_shh[2];
          if (!a_mn) {
            a_sh = shard_or_oob_q(P.a.g, a_br, a_blk, qsa);
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) a_shh[h] = shard_or_oob_q(P.a.g, a_blk, a_bc[h], qsa);
          }
          if (!b_mn) {
            b_sh = shard_or_oob_q(P.b.g, b_br, b_blk, qsb);
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) b_shh[h] = shard_or_oob_q(P.b.g, b_blk, b_bc[h], qsb);
          }
          for (int32_t kt = 0; kt < tpsK; ++kt) {
            const int s = (int)(it % S);
            const uint32_t ph = (it / S) & 1u;
            // test hook: both CTAs stop loading after the same stage (the even
            // CTA then drains every load in flight, below)
            if (P.stall_after >= 0 && (int64_t)it >= P.stall_after) {
              ok = false;
              break;
            }
            if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, P.err)) {
              ok = false;
              break;
            }
            const uint32_t fb = map_to_cta(full_bar(s), 0);
            // the even CTA expects both CTAs' bytes; the odd CTA's loads may land first
            // (the transaction count goes negative, the phase cannot end before this arrival)
            if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * Cfg::STAGE_BYTES);
            const int kofs = kt * BKP;
            // a wide map moves an operand's whole stage in one box (its 64-column
            // chunks land KCHUNK or MNBOX apart, as the separate boxes would)
            if (wide & 1u) {
              if (!a_mn)
                tma_load_4d_pair(a_stage(s), &mapA, fb, a_c1, (a_k + kofs) >> 6, a_sh);
              else
                tma_load_4d_pair(a_stage(s), &mapA, fb, a_k + kofs, a_c0[0] >> 6, a_shh[0]);
            } else if (!a_mn) {
#pragma unroll
              for (int c = 0; c < BKP / 64; ++c)
                tma_load_3d_pair(a_stage(s) + c * Cfg::KCHUNK, &mapA, fb, a_k + kofs + 64 * c, a_c1, a_sh);
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h)
                tma_load_3d_pair(a_stage(s) + h * Cfg::MNBOX, &mapA, fb, a_c0[h], a_k + kofs, a_shh[h]);
            }
            if (wide & 2u) {
              if (!b_mn)
                tma_load_4d_pair(b_stage(s), &mapB, fb, b_c1, (b_k + kofs) >> 6, b_sh);
              else
                tma_load_4d_pair(b_stage(s), &mapB, fb, b_k + kofs, b_c0[0] >> 6, b_shh[0]);
            } else if (!b_mn) {
#pragma unroll
              for (int c = 0; c < BKP / 64; ++c)
                tma_load_3d_pair(b_stage(s) + c * Cfg::KCHUNK, &mapB, fb, b_k + kofs + 64 * c, b_c1, b_sh);
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h)
                tma_load_3d_pair(b_stage(s) + h * Cfg::MNBOX, &mapB, fb, b_c0[h], b_k + kofs, b_shh[h]);
            }
            ++it;
            if (!next_ready) {  // the first stage is in flight: prepare the next tile
              next_ready = true;
              if (t + nclusters < ntiles) setup(t + nclusters, nxt);
            }
          }
        }
        cur = nxt;
      }
      if (!ok && leader) {
        // drain: every load of both CTAs completes on the even CTA's full barriers
        const uint32_t first = it > (uint32_t)S ? it - S : 0u;
        for (uint32_t j = first; j < it; ++j) mbar_wait_drain(full_bar((int)(j % S)), (j / S) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer (even CTA)
      const uint32_t idesc = P.in_f16 ? idesc_f16_f32(256, BN, a_mn ? 1 : 0, b_mn ? 1 : 0)
                                      : idesc_bf16_f32(256, BN, a_mn ? 1 : 0, b_mn ? 1 : 0);
      // Stage 0's operand descriptors, built once: a stage, chunk or row step
      // adds its byte offset / 16 to the 14-bit address field (shared
      // addresses stay below 256 KiB, so the field never carries).  Fewer
      // instructions per stage for this warp, which shares its scheduler with
      // two epilogue warps, keep the tensor pipe fed.
      const uint64_t adesc0 =
          a_mn ? smem_desc_sw128(a_stage(0), Cfg::MNBOX, 1024u) : smem_desc_sw128(a_stage(0), 16u, 1024u);
      const uint64_t bdesc0 =
          b_mn ? smem_desc_sw128(b_stage(0), Cfg::MNBOX, 1024u) : smem_desc_sw128(b_stage(0), 16u, 1024u);
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int64_t t = cid; t < ntiles && ok; t += nclusters) {
        const int buf = (int)(tc & 1u);
        const uint32_t tph = (tc >> 1) & 1u;
        if (!mbar_wait(tempty_bar(buf), tph ^ 1u, abort_flag, P.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
        bool first = true;
        for (int32_t sg = 0; sg < nsegK && ok; ++sg) {
          for (int32_t kt = 0; kt < tpsK; ++kt) {
            const int s = (int)(it % S);
            const uint32_t ph = (it / S) & 1u;
            if (!mbar_wait(full_bar(s), ph, abort_flag, P.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t as0 = adesc0 + (uint64_t)((s * Cfg::A_BYTES) >> 4);
            const uint64_t bs0 = bdesc0 + (uint64_t)((s * Cfg::B_BYTES) >> 4);
#pragma unroll
            for (int k16 = 0; k16 < BKP / 16; ++k16) {
              // K-major: 64-column chunks of 128 rows, +32 B per 16 columns;
              // MN-major: 64-wide boxes of BKP rows, +16 rows per step
              const uint32_t kk = (uint32_t)(k16 >> 2) * Cfg::KCHUNK + (uint32_t)(k16 & 3) * 32u;
              const uint64_t ad = as0 + (uint64_t)((a_mn ? k16 * 2048u : kk) >> 4);
              const uint64_t bd = bs0 + (uint64_t)((b_mn ? k16 * 2048u : kk) >> 4);
              umma_bf16_pair(d_tmem, ad, bd, idesc, (first && k16 == 0) ? 0u : 1u);
            }
            first = false;
            umma_commit_pair_mc(empty_bar(s), 3);
            ++it;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(tfull_bar(buf), 3);
        ++tc;
      }
      // every product issued must finish before the pair frees its TMEM
      umma_commit_pair_mc(final_bar, 1);
      mbar_wait_drain(final_bar, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    uint32_t tc = 0;
    uint32_t stores = 0;
    uint32_t aux_phase = 0;
    uint8_t* stg = stage_out + (warp - 2) * Cfg::STAGE_OUT;
    float cmax = 0.0f;  // H16: the largest |C| of the bf16 columns this warp stored
    for (int64_t t = cid; t < ntiles; t += nclusters) {
      TileInfo T;
      decode_pair_tile(P, t, rank, T);
      const int buf = (int)(tc & 1u);
      const uint32_t tph = (tc >> 1) & 1u;
      const bool aux0 = aux_prefetch<BN>(P, T, warp, lane, stg, &mapX, aux_bar(warp - 2));
      bool ok = lane == 0 ? mbar_wait(tfull_bar(buf), tph, abort_flag, P.err) : false;
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) {
        if (aux0 && lane == 0) mbar_wait_drain(aux_bar(warp - 2), aux_phase & 1u);  // let the load land
        __syncwarp();
        break;
      }
      tc_fence_after();
      epilogue_tile<BN, H16>(P, T, true, buf, tmem_base, warp, lane, stg, &mapC, &mapZ, &mapX, aux_bar(warp - 2),
                             aux_phase, abort_flag, map_to_cta(tempty_bar(buf), 0), true, stores, cmax, aux0);
      ++tc;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    if (H16) warp_amax(cmax, P.epi.amax_out, lane);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA frees the pair's TMEM or barriers while the other still uses them
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- chained GEMMs
// Two GEMMs in one persistent launch of CTA pairs, the second (job 1) reading
// the first's output (job 0) as its A operand: the MLP block of "Maximizing
// Parallelism in Distributed Training for Huge Neural Networks" §3.2, Y1 =
// GELU(X W1 + b1) feeding Y = Y1 W2 + b2 (the column-then-row split of
// Megatron's "Tensor parallelism").  The launch's work units are job 0's
// tiles, then job 1's tiles (times its contraction splits), each kind with
// the row tiles slowest, dealt to the clusters round-robin; every cluster
// takes its units in increasing order.
//  - A job-1 unit needs the rows of Y1 it contracts over: job 0's epilogue
//    warps count each finished tile (after its TMA stores have completed)
//    into a counter per (row tile, contraction half), and job 1's producers
//    wait for the full count before loading (bounded waits).  Job 1's units
//    start while job 0's last tiles are still in their epilogues.
//  - With two contraction halves, each half's unit writes its raw fp32 sums
//    (the plain fp32 epilogue, TMA stores) to its own slot of a scratch.  Per
//    epilogue-warp region (32 rows x 128 columns) a counter takes one arrival
//    from each half; the warp that arrives second adds the two slots (slot 0
//    first, so the sums do not depend on which half finished first), applies
//    the bias, and writes the bf16 output, reading and writing whole rows.
// Every wait is on a lower-numbered unit, so the launch cannot deadlock while
// its clusters are resident (a cluster not yet resident starts when any
// other kernel on the device leaves an SM); a wait that runs out raises
// TP3D_ETIMEOUT like every other.  The last CTA to leave zeroes the counters
// for the next launch.
struct ChainArgs {
  int64_t units0, units1;  // job 0 tiles; job 1 tiles x splits
  int32_t splits;          // 1 or 2: job 1's contraction halves
  int32_t ready_target;    // arrivals that complete one (row tile, half) of job 0's output
  int* ready;              // [row tile][half]
  int* fix;                // [job-1 tile][CTA][epilogue warp]: arrivals of the two halves
  int* exits;              // CTAs that have left
  int32_t n_ready, n_fix;
  const float* part;       // the halves' sums: slot s holds rows s M .. s M + M - 1 (dense, N columns)
};

// The second half to finish adds both halves' sums for its warp's region
// (rows T.m0 + 32 quarter .. +31, columns T.n0 + 128 half .. +127): lane l
// takes columns 4l .. 4l + 3 of each row, so every read (512 bytes of fp32)
// and write (256 bytes of bf16) of a row is one contiguous span.  Then
// alpha, bias, GELU and residual as the tensor-memory epilogue applies them.
__device__ __noinline__ void chain_fixup(const float* __restrict__ part, int64_t M, int64_t N, const Grid cg,
                                         __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ bias,
                                         const __nv_bfloat16* __restrict__ res, float alpha, int act, int64_t m0,
                                         int64_t n0, int warp, int lane) {
  const int quarter = warp & 3, hf = (warp - 2) >> 2;
  const int64_t n = n0 + hf * 128 + lane * 4;
  const int32_t bc = (int32_t)((uint32_t)n / (uint32_t)cg.bw);  // the region lies in one block column
  float bb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (bias) {
    const __nv_bfloat162* bp = reinterpret_cast<const __nv_bfloat162*>(bias + n);
    const float2 b0 = __bfloat1622float2(bp[0]), b1 = __bfloat1622float2(bp[1]);
    bb[0] = b0.x; bb[1] = b0.y; bb[2] = b1.x; bb[3] = b1.y;
  }
  const int64_t mr = m0 + quarter * 32;
  const int32_t br = (int32_t)((uint32_t)mr / (uint32_t)cg.bh);  // 32 rows inside one block row
  const int64_t base = cg.block_base(br, bc) + (mr - (int64_t)br * cg.bh) * cg.bw + (n - (int64_t)bc * cg.bw);
#pragma unroll 1
  for (int i = 0; i < 32; i += 8) {
    float4 a[8], b[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t m = mr + i + u;
      a[u] = __ldcg(reinterpret_cast<const float4*>(part + m * N + n));
      b[u] = __ldcg(reinterpret_cast<const float4*>(part + (M + m) * N + n));
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t off = base + (int64_t)(i + u) * cg.bw;
      float x[4] = {a[u].x + b[u].x, a[u].y + b[u].y, a[u].z + b[u].z, a[u].w + b[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[e] = x[e] * alpha + bb[e];
        if (act == EPI_GELU) x[e] = gelu_f(x[e]);
      }
      if (res) {
        const __nv_bfloat162* rp = reinterpret_cast<const __nv_bfloat162*>(res + off);
        const float2 r0 = __bfloat1622float2(rp[0]), r1 = __bfloat1622float2(rp[1]);
        x[0] += r0.x; x[1] += r0.y; x[2] += r1.x; x[3] += r1.y;
      }
      __nv_bfloat162 h[2] = {__floats2bfloat162_rn(x[0], x[1]), __floats2bfloat162_rn(x[2], x[3])};
      *reinterpret_cast<uint2*>(out + off) = *reinterpret_cast<const uint2*>(h);
    }
  }
}

// tile -> coordinates, row tiles slowest; tm_out = the row tile
__device__ __forceinline__ void decode_rows_slow(const GemmProblem& P, uint32_t tile, uint32_t r, TileInfo& T,
                                                 uint32_t& tm_out) {
  const uint32_t segM = (uint32_t)P.segM, segN = (uint32_t)P.segN;
  const uint32_t tpsM = (segM + 255u) / 256u, tpsN = (segN + 255u) / 256u;
  const uint32_t tiles_n = udiv32(P.N, segN) * tpsN;
  const uint32_t tm = tile / tiles_n, tn = tile - tm * tiles_n;
  const uint32_t sm = tm / tpsM, sn = tn / tpsN;
  T.z = 0;
  T.m0 = (int64_t)sm * segM + (int64_t)(tm - sm * tpsM) * 256 + 128 * (int64_t)r;
  T.n0 = (int64_t)sn * segN + (int64_t)(tn - sn * tpsN) * 256;
  T.m_end = (int64_t)sm * segM + segM;
  T.n_end = (int64_t)sn * segN + segN;
  tm_out = tm;
}

struct ChainUnit {
  int32_t job, s;     // job; contraction half (job 1)
  uint32_t tile;      // the job's tile
  int32_t sg0, sg1;   // contraction segments [sg0, sg1)
};
__device__ __forceinline__ ChainUnit chain_unit(const GemmProblem& P0, const GemmProblem& P1, const ChainArgs& C,
                                                int64_t u) {
  ChainUnit U;
  if (u < C.units0) {
    U.job = 0;
    U.s = 0;
    U.tile = (uint32_t)u;
    U.sg0 = 0;
    U.sg1 = (int32_t)udiv32(P0.K, P0.segK);
  } else {
    const uint32_t v = (uint32_t)(u - C.units0);
    U.job = 1;
    U.tile = v / (uint32_t)C.splits;
    U.s = (int32_t)(v - U.tile * (uint32_t)C.splits);
    const int32_t per = (int32_t)udiv32(P1.K, P1.segK) / C.splits;
    U.sg0 = U.s * per;
    U.sg1 = U.sg0 + per;
  }
  return U;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_chain_kernel(const __grid_constant__ CUtensorMap mapA0, const __grid_constant__ CUtensorMap mapB0,
                      const __grid_constant__ CUtensorMap mapC0, const __grid_constant__ CUtensorMap mapZ0,
                      const __grid_constant__ CUtensorMap mapX0, const __grid_constant__ CUtensorMap mapA1,
                      const __grid_constant__ CUtensorMap mapB1, const __grid_constant__ CUtensorMap mapC1,
                      const __grid_constant__ CUtensorMap mapZ1, const __grid_constant__ CUtensorMap mapX1,
                      const __grid_constant__ CUtensorMap mapP, const __grid_constant__ GemmProblem P0,
                      const __grid_constant__ GemmProblem P1, const __grid_constant__ GemmProblem P1h,
                      const uint32_t wide0, const uint32_t wide1, const __grid_constant__ ChainArgs C) {
  using Cfg = Tc2Cfg<128>;
  constexpr int S = Cfg::STAGES;
  constexpr int BKP = Cfg::BKP;
  constexpr int BN = Cfg::BN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint8_t* stage_out = base_ptr + S * Cfg::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage_out + kEpiWarps * Cfg::STAGE_OUT);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * S + 5 + kEpiWarps);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* last_cta = const_cast<int*>(abort_flag) + 1;

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t final_bar = bar0 + 8u * (2 * S + 4);
  auto aux_bar = [&](int ew) { return bar0 + 8u * (2 * S + 5 + ew); };
  auto a_stage = [&](int s) { return base + (uint32_t)(s * Cfg::A_BYTES); };
  auto b_stage = [&](int s) { return base + (uint32_t)(S * Cfg::A_BYTES + s * Cfg::B_BYTES); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * kEpiWarps);
    }
    mbar_init(final_bar, 1);
    for (int e = 0; e < kEpiWarps; ++e) mbar_init(aux_bar(e), 1);
    *abort_flag = 0;
    *last_cta = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_holder), Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&mapA0);
    tma_prefetch_map(&mapB0);
    tma_prefetch_map(&mapA1);
    tma_prefetch_map(&mapB1);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int64_t nunits = C.units0 + C.units1;
  const int64_t nclusters = gridDim.x >> 1, cid = blockIdx.x >> 1;
  // both jobs have the same operand majors and input type (the launcher checks)
  const bool a_mn = P0.a.mn_major != 0, b_mn = P0.b.mn_major != 0;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      struct UnitLd {
        int32_t job, sg0, sg1, wait_idx;
        int64_t ak, bk;
        int32_t a_br, b_br, a_c1, b_c1;
        int32_t a_bc[2], b_bc[2], a_c0[2], b_c0[2];
        int32_t a_k0, a_blk0, b_k0, b_blk0;  // the unit's first segment: offset in its block, and the block
      };
      auto setup = [&](int64_t u, UnitLd& L) {
        const ChainUnit U = chain_unit(P0, P1, C, u);
        const GemmProblem& P = U.job ? P1 : P0;
        TileInfo T;
        uint32_t tm;
        decode_rows_slow(P, U.tile, rank, T, tm);
        L.job = U.job;
        L.sg0 = U.sg0;
        L.sg1 = U.sg1;
        L.wait_idx = U.job ? (int32_t)(tm * (uint32_t)C.splits) + U.s : -1;
        const int64_t am = T.m0 + op_off(P.a.hi1, P.a.lo1, P.a.base1, T.z, P.Hz);
        L.ak = op_off(P.a.hi2, P.a.lo2, P.a.base2, T.z, P.Hz);
        L.bk = op_off(P.b.hi1, P.b.lo1, P.b.base1, T.z, P.Hz);
        const int64_t bn = T.n0 + 128 * (int64_t)rank + op_off(P.b.hi2, P.b.lo2, P.b.base2, T.z, P.Hz);
        if (!a_mn) {
          L.a_br = (int32_t)udiv32(am, P.a.g.bh);
          L.a_c1 = (int32_t)(am - (int64_t)L.a_br * P.a.g.bh);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            L.a_bc[h] = (int32_t)udiv32(am + 64 * h, P.a.g.bw);
            L.a_c0[h] = (int32_t)(am + 64 * h - (int64_t)L.a_bc[h] * P.a.g.bw);
          }
        }
        if (!b_mn) {
          L.b_br = (int32_t)udiv32(bn, P.b.g.bh);
          L.b_c1 = (int32_t)(bn - (int64_t)L.b_br * P.b.g.bh);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            L.b_bc[h] = (int32_t)udiv32(bn + 64 * h, P.b.g.bw);
            L.b_c0[h] = (int32_t)(bn + 64 * h - (int64_t)L.b_bc[h] * P.b.g.bw);
          }
        }
        // the unit's first segment; later ones step from it by segK (which
        // divides every block extent along the contraction)
        const int64_t ka = L.ak + (int64_t)U.sg0 * P.segK, kb = L.bk + (int64_t)U.sg0 * P.segK;
        const int64_t akd = a_mn ? P.a.g.bh : P.a.g.bw, bkd = b_mn ? P.b.g.bh : P.b.g.bw;
        L.a_blk0 = (int32_t)udiv32(ka, akd);
        L.a_k0 = (int32_t)(ka - (int64_t)L.a_blk0 * akd);
        L.b_blk0 = (int32_t)udiv32(kb, bkd);
        L.b_k0 = (int32_t)(kb - (int64_t)L.b_blk0 * bkd);
      };
      uint32_t it = 0;
      bool ok = true;
      UnitLd cur = {}, nxt = {};
      if (cid < nunits) setup(cid, cur);
      for (int64_t u = cid; u < nunits && ok; u += nclusters) {
        const GemmProblem& P = cur.job ? P1 : P0;
        const CUtensorMap* mA = cur.job ? &mapA1 : &mapA0;
        const CUtensorMap* mB = cur.job ? &mapB1 : &mapB0;
        const uint32_t wide = cur.job ? wide1 : wide0;
        if (cur.wait_idx >= 0) {
          // job 1 reads rows of Y1 that job 0's epilogues store: wait for all of them
          if (!counter_wait_geq(C.ready + cur.wait_idx, C.ready_target, abort_flag, P.err)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();  // the TMA loads below see those stores
        }
        const int32_t segK = (int32_t)P.segK, tpsK = segK / BKP;
        const int32_t a_br = cur.a_br, b_br = cur.b_br;
        const int a_c1 = cur.a_c1, b_c1 = cur.b_c1;
        const int32_t a_bc[2] = {cur.a_bc[0], cur.a_bc[1]}, b_bc[2] = {cur.b_bc[0], cur.b_bc[1]};
        const int a_c0[2] = {cur.a_c0[0], cur.a_c0[1]}, b_c0[2] = {cur.b_c0[0], cur.b_c0[1]};
        const int qsa = log2_if_pow2(P.a.g.q), qsb = log2_if_pow2(P.b.g.q);
        const int32_t akd = (int32_t)(a_mn ? P.a.g.bh : P.a.g.bw), bkd = (int32_t)(b_mn ? P.b.g.bh : P.b.g.bw);
        int32_t a_k = cur.a_k0, a_blk = cur.a_blk0, b_k = cur.b_k0, b_blk = cur.b_blk0;
        bool next_ready = false;
        for (int32_t sg = cur.sg0; sg < cur.sg1 && ok; ++sg) {
          if (sg > cur.sg0) {  // step one segment (no division: segK divides the block extent)
            a_k += segK;
            if (a_k >= akd) {
              a_k -= akd;
              ++a_blk;
            }
            b_k += segK;
            if (b_k >= bkd) {
              b_k -= bkd;
              ++b_blk;
            }
          }
          int a_sh = 0, b_sh = 0;
          int a_shh[2], b_shh[2];
          if (!a_mn) {
            a_sh = shard_or_oob_q(P.a.g, a_br, a_blk, qsa);
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) a_shh[h] = shard_or_oob_q(P.a.g, a_blk, a_bc[h], qsa);
          }
          if (!b_mn) {
            b_sh = shard_or_oob_q(P.b.g, b_br, b_blk, qsb);
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) b_shh[h] = shard_or_oob_q(P.b.g, b_blk, b_bc[h], qsb);
          }
          for (int32_t kt = 0; kt < tpsK; ++kt) {
            const int s = (int)(it % S);
            const uint32_t ph = (it / S) & 1u;
            if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, P.err)) {
              ok = false;
              break;
            }
            const uint32_t fb = map_to_cta(full_bar(s), 0);
            if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * Cfg::STAGE_BYTES);
            const int kofs = kt * BKP;
            if (wide & 1u) {
              if (!a_mn)
                tma_load_4d_pair(a_stage(s), mA, fb, a_c1, (a_k + kofs) >> 6, a_sh);
              else
                tma_load_4d_pair(a_stage(s), mA, fb, a_k + kofs, a_c0[0] >> 6, a_shh[0]);
            } else if (!a_mn) {
#pragma unroll
              for (int c = 0; c < BKP / 64; ++c)
                tma_load_3d_pair(a_stage(s) + c * Cfg::KCHUNK, mA, fb, a_k + kofs + 64 * c, a_c1, a_sh);
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h)
                tma_load_3d_pair(a_stage(s) + h * Cfg::MNBOX, mA, fb, a_c0[h], a_k + kofs, a_shh[h]);
            }
            if (wide & 2u) {
              if (!b_mn)
                tma_load_4d_pair(b_stage(s), mB, fb, b_c1, (b_k + kofs) >> 6, b_sh);
              else
                tma_load_4d_pair(b_stage(s), mB, fb, b_k + kofs, b_c0[0] >> 6, b_shh[0]);
            } else if (!b_mn) {
#pragma unroll
              for (int c = 0; c < BKP / 64; ++c)
                tma_load_3d_pair(b_stage(s) + c * Cfg::KCHUNK, mB, fb, b_k + kofs + 64 * c, b_c1, b_sh);
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h)
                tma_load_3d_pair(b_stage(s) + h * Cfg::MNBOX, mB, fb, b_c0[h], b_k + kofs, b_shh[h]);
            }
            ++it;
            if (!next_ready) {  // the unit's first stage is in flight: prepare the next unit
              next_ready = true;
              if (u + nclusters < nunits) setup(u + nclusters, nxt);
            }
          }
        }
        cur = nxt;
      }
      if (!ok && leader) {
        const uint32_t first = it > (uint32_t)S ? it - S : 0u;
        for (uint32_t j = first; j < it; ++j) mbar_wait_drain(full_bar((int)(j % S)), (j / S) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer (even CTA)
      const uint32_t idesc = P0.in_f16 ? idesc_f16_f32(256, BN, a_mn ? 1 : 0, b_mn ? 1 : 0)
                                       : idesc_bf16_f32(256, BN, a_mn ? 1 : 0, b_mn ? 1 : 0);
      const uint64_t adesc0 =
          a_mn ? smem_desc_sw128(a_stage(0), Cfg::MNBOX, 1024u) : smem_desc_sw128(a_stage(0), 16u, 1024u);
      const uint64_t bdesc0 =
          b_mn ? smem_desc_sw128(b_stage(0), Cfg::MNBOX, 1024u) : smem_desc_sw128(b_stage(0), 16u, 1024u);
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int64_t u = cid; u < nunits && ok; u += nclusters) {
        const ChainUnit U = chain_unit(P0, P1, C, u);
        const GemmProblem& P = U.job ? P1 : P0;
        const int32_t tpsK = (int32_t)P.segK / BKP;
        const int buf = (int)(tc & 1u);
        const uint32_t tph = (tc >> 1) & 1u;
        if (!mbar_wait(tempty_bar(buf), tph ^ 1u, abort_flag, P.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
        bool first = true;
        for (int32_t sg = U.sg0; sg < U.sg1 && ok; ++sg) {
          for (int32_t kt = 0; kt < tpsK; ++kt) {
            const int s = (int)(it % S);
            const uint32_t ph = (it / S) & 1u;
            if (!mbar_wait(full_bar(s), ph, abort_flag, P.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t as0 = adesc0 + (uint64_t)((s * Cfg::A_BYTES) >> 4);
            const uint64_t bs0 = bdesc0 + (uint64_t)((s * Cfg::B_BYTES) >> 4);
#pragma unroll
            for (int k16 = 0; k16 < BKP / 16; ++k16) {
              const uint32_t kk = (uint32_t)(k16 >> 2) * Cfg::KCHUNK + (uint32_t)(k16 & 3) * 32u;
              const uint64_t ad = as0 + (uint64_t)((a_mn ? k16 * 2048u : kk) >> 4);
              const uint64_t bd = bs0 + (uint64_t)((b_mn ? k16 * 2048u : kk) >> 4);
              umma_bf16_pair(d_tmem, ad, bd, idesc, (first && k16 == 0) ? 0u : 1u);
            }
            first = false;
            umma_commit_pair_mc(empty_bar(s), 3);
            ++it;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(tfull_bar(buf), 3);
        ++tc;
      }
      umma_commit_pair_mc(final_bar, 1);
      mbar_wait_drain(final_bar, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    uint32_t tc = 0;
    uint32_t stores = 0;
    uint32_t aux_phase = 0;
    uint8_t* stg = stage_out + (warp - 2) * Cfg::STAGE_OUT;
    float cmax = 0.0f;
    for (int64_t u = cid; u < nunits; u += nclusters) {
      const ChainUnit U = chain_unit(P0, P1, C, u);
      const GemmProblem& P = U.job ? P1 : P0;
      TileInfo T;
      uint32_t tm;
      decode_rows_slow(P, U.tile, rank, T, tm);
      const int buf = (int)(tc & 1u);
      const uint32_t tph = (tc >> 1) & 1u;
      bool ok = lane == 0 ? mbar_wait(tfull_bar(buf), tph, abort_flag, P.err) : false;
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      // a contraction half writes its raw sums into its slot (the plain fp32
      // epilogue on rows s M + m of the scratch); every other unit its output
      const bool split = U.job == 1 && C.splits == 2;
      TileInfo Te = T;
      if (split) {
        Te.m0 += (int64_t)U.s * P1.M;
        Te.m_end += (int64_t)U.s * P1.M;
      }
      const GemmProblem& Pe = split ? P1h : P;
      const CUtensorMap* mc = split ? &mapP : U.job ? &mapC1 : &mapC0;
      const CUtensorMap* mz = split ? &mapP : U.job ? &mapZ1 : &mapZ0;
      const CUtensorMap* mx = split ? &mapP : U.job ? &mapX1 : &mapX0;
      epilogue_tile<BN, false>(Pe, Te, true, buf, tmem_base, warp, lane, stg, mc, mz, mx, aux_bar(warp - 2),
                               aux_phase, abort_flag, map_to_cta(tempty_bar(buf), 0), true, stores, cmax);
      ++tc;
      if (U.job == 0) {
        // this warp's share of the tile is in memory (not just read out of
        // shared memory) before the count says so
        if (lane == 0) {
          bulk_wait_all();
          fence_proxy_async_global();
          __threadfence();
          const uint32_t half = (uint32_t)C.splits == 1u ? 0u : (uint32_t)T.n0 / ((uint32_t)P0.N / 2u);
          counter_add_release(C.ready + tm * (uint32_t)C.splits + half, 1);
        }
        __syncwarp();
      } else if (split) {
        // the second of the two halves to reach this region adds them
        int prev = 0;
        if (lane == 0) {
          bulk_wait_all();
          fence_proxy_async_global();
          __threadfence();
          prev = atomicAdd(C.fix + ((int64_t)U.tile * 2 + rank) * kEpiWarps + (warp - 2), 1);
          __threadfence();
        }
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == 1)
          chain_fixup(C.part, P1.M, P1.N, P1.c.g, static_cast<__nv_bfloat16*>(const_cast<void*>(P1.c.ptr)),
                      static_cast<const __nv_bfloat16*>(P1.epi.bias), static_cast<const __nv_bfloat16*>(P1.epi.resid),
                      P1.epi.alpha, P1.epi.act, T.m0, T.n0, warp, lane);
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
  // the last CTA to leave zeroes the counters for the next launch (every
  // wait of this launch is over once all other CTAs have left)
  if (threadIdx.x == 0) {
    __threadfence();
    *last_cta = atomicAdd(C.exits, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (*last_cta) {
    __threadfence();
    for (int i = threadIdx.x; i < C.n_ready; i += blockDim.x) C.ready[i] = 0;
    for (int i = threadIdx.x; i < C.n_fix; i += blockDim.x) C.fix[i] = 0;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *C.exits = 0;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D map over a stored matrix: (column in shard, row in shard, shard).
tp3d_status make_map(CUtensorMap* m, const Grid& g, const void* ptr, uint32_t box_inner, uint32_t box_rows,
                     CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, int esz = 2,
                     CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return TP3D_ECUDA;
  cuuint64_t dims[3] = {(cuuint64_t)g.bw, (cuuint64_t)g.bh, (cuuint64_t)g.nshards()};
  cuuint64_t strides[2] = {(cuuint64_t)g.bw * esz, (cuuint64_t)(g.bh * g.bw * esz)};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TP3D_OK : TP3D_ECUDA;
}

// 4-D map over a stored bf16 matrix whose shard width is a multiple of 64:
// (column in a 64-column chunk, row in shard, chunk, shard).  A box of
// `chunks` chunks x `box_rows` rows lands in shared memory chunk after chunk,
// each chunk box_rows x 128 bytes with the 128-byte swizzle.  Returns false
// (and the caller keeps 3-D maps) if the driver rejects the encoding.
bool make_map_wide(CUtensorMap* m, const Grid& g, const void* ptr, uint32_t box_rows, uint32_t chunks) {
  auto fn = encode_fn();
  if (!fn || g.bw % 64 != 0) return false;
  cuuint64_t dims[4] = {64, (cuuint64_t)g.bh, (cuuint64_t)(g.bw / 64), (cuuint64_t)g.nshards()};
  cuuint64_t strides[3] = {(cuuint64_t)g.bw * 2, 128, (cuuint64_t)(g.bh * g.bw * 2)};
  cuuint32_t box[4] = {64, box_rows, chunks, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool H16>
tp3d_status launch(const tp3d_ctx* ctx, const GemmProblem& P, cudaStream_t s) {
  using Cfg = TcCfg<BN>;
  CUtensorMap ma, mb, mc, mz, mx;
  TP3D_TRY(make_map(&ma, P.a.g, P.a.ptr, 64, P.a.mn_major ? 64 : BM));
  TP3D_TRY(make_map(&mb, P.b.g, P.b.ptr, 64, P.b.mn_major ? 64 : BN));
  // output boxes: 32 rows x 32 columns (64-byte bf16 rows or 128-byte fp32 rows)
  if (P.epi.out_f32)
    TP3D_TRY(make_map(&mc, P.c.g, P.c.ptr, 16, 32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, CU_TENSOR_MAP_SWIZZLE_64B));
  else
    TP3D_TRY(make_map(&mc, P.c.g, P.c.ptr, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_64B));
  if (P.epi.zsave)
    TP3D_TRY(make_map(&mz, P.c.g, P.epi.zsave, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_64B));
  else
    mz = mc;
  const void* aux = P.epi.resid ? P.epi.resid : P.epi.gin;
  if (aux)
    TP3D_TRY(make_map(&mx, P.c.g, aux, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_64B));
  else
    mx = mc;
  TP3D_CUDA_TRY(cudaFuncSetAttribute(gemm_tc_kernel<BN, H16>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM));
  const int64_t tpsM = (P.segM + BM - 1) / BM, tpsN = (P.segN + BN - 1) / BN;
  const int64_t ntiles = (int64_t)P.Z * (P.M / P.segM) * tpsM * (P.N / P.segN) * tpsN;
  if (ntiles <= 0) return TP3D_OK;
  const int grid = (int)(ntiles < ctx->num_sms ? ntiles : ctx->num_sms);
  gemm_tc_kernel<BN, H16><<<grid, kThreads, Cfg::SMEM, s>>>(ma, mb, mc, mz, mx, P);
  return cudaGetLastError() == cudaSuccess ? TP3D_OK : TP3D_ECUDA;
}

// CTA pairs that fit on the device at once (0 if the query fails).
template <int KD, bool H16>
int pair_clusters(const tp3d_ctx* ctx) {
  static int cached[64] = {};
  const int dev = ctx->device & 63;
  if (cached[dev] != 0) return cached[dev] > 0 ? cached[dev] : 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Tc2Cfg<KD>::SMEM;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2 * (unsigned)(ctx->num_sms / 2));
  int n = 0;
  if (cudaFuncSetAttribute(gemm_tc2_kernel<KD, H16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Tc2Cfg<KD>::SMEM) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, gemm_tc2_kernel<KD, H16>, &cfg) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();
    cached[dev] = -1;
    return 0;
  }
  cached[dev] = n;
  return n;
}

template <int KD, bool H16>
tp3d_status launch_pair(const tp3d_ctx* ctx, const GemmProblem& P, cudaStream_t s) {
  using Cfg = Tc2Cfg<KD>;
  CUtensorMap ma, mb, mc, mz, mx;
  // One box per operand and stage where every stage's chunks lie in one
  // shard: K-major, the contraction segment (a multiple of KD) inside a
  // block row; MN-major, the CTA's 128 columns (128-aligned in a segment
  // that is a multiple of 128) inside a block whose width is a multiple of 128.
  uint32_t wide = 0;
  auto wide_ok = [&](const Operand& o, int64_t seg_mn) {
    return o.mn_major ? (o.g.bw % 128 == 0 && seg_mn % 128 == 0) : (o.g.bw % 64 == 0);
  };
  if (wide_ok(P.a, P.segM) && make_map_wide(&ma, P.a.g, P.a.ptr, P.a.mn_major ? KD : 128, P.a.mn_major ? 2 : KD / 64))
    wide |= 1u;
  else
    TP3D_TRY(make_map(&ma, P.a.g, P.a.ptr, 64, P.a.mn_major ? KD : 128));
  if (wide_ok(P.b, P.segN) && make_map_wide(&mb, P.b.g, P.b.ptr, P.b.mn_major ? KD : 128, P.b.mn_major ? 2 : KD / 64))
    wide |= 2u;
  else
    TP3D_TRY(make_map(&mb, P.b.g, P.b.ptr, 64, P.b.mn_major ? KD : 128));
  if (P.epi.out_f32)
    TP3D_TRY(make_map(&mc, P.c.g, P.c.ptr, 16, 32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, CU_TENSOR_MAP_SWIZZLE_64B));
  else
    TP3D_TRY(make_map(&mc, P.c.g, P.c.ptr, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_64B));
  if (P.epi.zsave)
    TP3D_TRY(make_map(&mz, P.c.g, P.epi.zsave, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_64B));
  else
    mz = mc;
  const void* aux = P.epi.resid ? P.epi.resid : P.epi.gin;
  if (aux)
    TP3D_TRY(make_map(&mx, P.c.g, aux, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_64B));
  else
    mx = mc;
  const int64_t ntiles = (int64_t)P.Z * (P.M / P.segM) * ((P.segM + 255) / 256) * (P.N / P.segN) *
                         ((P.segN + 255) / 256);
  if (ntiles <= 0) return TP3D_OK;
  const int max_clusters = pair_clusters<KD, H16>(ctx);
  if (max_clusters < 1) return TP3D_ECUDA;
  // the kernel decodes tiles and shard coordinates in 32-bit arithmetic
  const int64_t lim = INT32_MAX;
  if (P.M > lim || P.N > lim || P.K > lim || ntiles > lim || P.a.g.R > lim || P.a.g.C > lim || P.b.g.R > lim ||
      P.b.g.C > lim || P.c.g.R > lim || P.c.g.C > lim)
    return TP3D_EUNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int64_t nc = ntiles < max_clusters ? ntiles : max_clusters;
  cfg.gridDim = dim3(2 * (unsigned)nc);
  TP3D_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemm_tc2_kernel<KD, H16>, ma, mb, mc, mz, mx, P, wide));
  return TP3D_OK;
}

// The tensor maps of one CTA-pair problem with 128-deep stages (as launch_pair builds them).
struct PairMaps {
  CUtensorMap a, b, c, z, x;
  uint32_t wide;
};
tp3d_status pair_maps(const GemmProblem& P, PairMaps* m) {
  constexpr int KD = 128;
  m->wide = 0;
  auto wide_ok = [&](const Operand& o, int64_t seg_mn) {
    return o.mn_major ? (o.g.bw % 128 == 0 && seg_mn % 128 == 0) : (o.g.bw % 64 == 0);
  };
  if (wide_ok(P.a, P.segM) && make_map_wide(&m->a, P.a.g, P.a.ptr, P.a.mn_major ? KD : 128, P.a.mn_major ? 2 : KD / 64))
    m->wide |= 1u;
  else
    TP3D_TRY(make_map(&m->a, P.a.g, P.a.ptr, 64, P.a.mn_major ? KD : 128));
  if (wide_ok(P.b, P.segN) && make_map_wide(&m->b, P.b.g, P.b.ptr, P.b.mn_major ? KD : 128, P.b.mn_major ? 2 : KD / 64))
    m->wide |= 2u;
  else
    TP3D_TRY(make_map(&m->b, P.b.g, P.b.ptr, 64, P.b.mn_major ? KD : 128));
  if (P.epi.out_f32)
    TP3D_TRY(make_map(&m->c, P.c.g, P.c.ptr, 16, 32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, CU_TENSOR_MAP_SWIZZLE_64B));
  else
    TP3D_TRY(make_map(&m->c, P.c.g, P.c.ptr, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_64B));
  if (P.epi.zsave)
    TP3D_TRY(make_map(&m->z, P.c.g, P.epi.zsave, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_64B));
  else
    m->z = m->c;
  const void* aux = P.epi.resid ? P.epi.resid : P.epi.gin;
  if (aux)
    TP3D_TRY(make_map(&m->x, P.c.g, aux, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_64B));
  else
    m->x = m->c;
  return TP3D_OK;
}

// CTA pairs of the chained kernel that fit on the device at once (0: none).
int chain_clusters(const tp3d_ctx* ctx) {
  static int cached[64] = {};
  const int dev = ctx->device & 63;
  if (cached[dev] != 0) return cached[dev] > 0 ? cached[dev] : 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Tc2Cfg<128>::SMEM;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2 * (unsigned)(ctx->num_sms / 2));
  int n = 0;
  if (cudaFuncSetAttribute(gemm_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Tc2Cfg<128>::SMEM) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, gemm_chain_kernel, &cfg) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();
    cached[dev] = -1;
    return 0;
  }
  cached[dev] = n;
  return n;
}

bool same_grid(const Grid& x, const Grid& y) {
  return x.kind == y.kind && x.q == y.q && x.rb == y.rb && x.cb == y.cb && x.R == y.R && x.C == y.C && x.bh == y.bh &&
         x.bw == y.bw && x.copies == y.copies;
}

}  // namespace

// The chained launch's shape of work, or false if (P0, P1) do not qualify:
// the second problem's A is the first's output (same buffer and layout); whole
// 256 x 256 tiles; 128-deep stages; no batch windows, causal masks or fp16
// paths; and a working set (both inputs, the intermediate, the second
// weight) of at most 64 MiB, so that the row-tiles-slowest order costs no
// HBM re-reads (L2 is 126 MiB).  Two contraction halves for the second
// problem when that doubles its units without passing one wave of clusters.
bool chain_plan(const tp3d_ctx* ctx, const GemmProblem& P0, const GemmProblem& P1, ChainShape* sh) {
  const GemmProblem* Ps[2] = {&P0, &P1};
  for (const GemmProblem* P : Ps) {
    if (P->Z != 1 || P->Hz != 1 || P->causal != CAUSAL_NONE || P->in_f16 || P->epi.f16_cols || P->epi.alpha_dev ||
        P->epi.amax_out)
      return false;
    if (P->segM % 256 || P->segN % 256 || P->segK % 128 || P->M % P->segM || P->N % P->segN || P->K % P->segK)
      return false;
    if (P->M > INT32_MAX || P->N > INT32_MAX || P->K > INT32_MAX) return false;
    const Grid* gs[3] = {&P->a.g, &P->b.g, &P->c.g};
    for (const Grid* g : gs)
      if (g->bw % 8 || g->R > INT32_MAX || g->C > INT32_MAX) return false;
  }
  if (P0.a.mn_major != P1.a.mn_major || P0.b.mn_major != P1.b.mn_major) return false;
  if (P0.M != P1.M || P0.segM != P1.segM || P1.K != P0.N || P1.a.ptr != P0.c.ptr || P1.a.mn_major ||
      !same_grid(P1.a.g, P0.c.g) || P0.epi.out_f32)
    return false;
  const double ws = 2.0 * ((double)P0.M * P0.K + (double)P0.K * P0.N + (double)P0.M * P0.N + (double)P1.K * P1.N);
  if (ws > 64.0 * 1024 * 1024) return false;
  const int clusters = chain_clusters(ctx);
  if (clusters < 1) return false;
  const int64_t rows = P0.M / 256;
  sh->units0 = rows * (P0.N / 256);
  const int64_t tiles1 = rows * (P1.N / 256);
  const int64_t nseg1 = P1.K / P1.segK;
  // the halves' fix-up writes rows of 128 columns inside one block of the output
  const bool split_ok = nseg1 % 2 == 0 && (P0.N / 2) % P0.segN == 0 && P1.c.g.bw % 128 == 0 && !P1.epi.out_f32 &&
                        !P1.epi.zsave && !P1.epi.gin && P1.epi.act != EPI_GELU_BWD;
  sh->splits = (split_ok && 2 * tiles1 <= clusters) ? 2 : 1;
  sh->units1 = tiles1 * sh->splits;
  sh->n_ready = rows * sh->splits;
  sh->n_fix = sh->splits == 2 ? tiles1 * 2 * kEpiWarps : 0;
  sh->ready_target = 2 * kEpiWarps * (int32_t)((P0.N / 256) / sh->splits);
  sh->clusters = (int)((sh->units0 + sh->units1) < clusters ? (sh->units0 + sh->units1) : clusters);
  const size_t counters = (size_t)(sh->n_ready + sh->n_fix + 1) * sizeof(int);
  sh->counter_bytes = (counters + 255) & ~(size_t)255;
  sh->scratch_bytes = sh->counter_bytes + (sh->splits == 2 ? (size_t)(2 * P1.M * P1.N) * sizeof(float) : 0);
  return true;
}

// Launch the chain on `scratch` (chain_plan's scratch_bytes, 256-byte
// aligned; its counters zero, as every launch leaves them).
tp3d_status gemm_chain_tc(const tp3d_ctx* ctx, const GemmProblem& P0i, const GemmProblem& P1i, const ChainShape& sh,
                          void* scratch, cudaStream_t s) {
  GemmProblem P0 = P0i, P1 = P1i;
  P0.stall_after = P1.stall_after = -1;
  PairMaps m0, m1;
  TP3D_TRY(pair_maps(P0, &m0));
  TP3D_TRY(pair_maps(P1, &m1));
  ChainArgs C;
  C.units0 = sh.units0;
  C.units1 = sh.units1;
  C.splits = sh.splits;
  C.ready_target = sh.ready_target;
  int* counters = static_cast<int*>(scratch);
  C.ready = counters;
  C.fix = counters + sh.n_ready;
  C.exits = counters + sh.n_ready + sh.n_fix;
  C.n_ready = (int32_t)sh.n_ready;
  C.n_fix = (int32_t)sh.n_fix;
  float* part = sh.splits == 2 ? reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + sh.counter_bytes) : nullptr;
  C.part = part;
  // the halves' raw sums: job 1 with a dense fp32 output of 2 M rows (slot s = rows s M ..)
  GemmProblem P1h = P1;
  CUtensorMap mp = m1.c;
  if (part) {
    Grid gp{};
    gp.kind = TP3D_ROW;
    gp.q = 0;
    gp.rb = 1;
    gp.cb = 1;
    gp.R = 2 * P1.M;
    gp.C = P1.N;
    gp.bh = gp.R;
    gp.bw = gp.C;
    gp.copies = 1;
    P1h.c.g = gp;
    P1h.c.ptr = part;
    P1h.c.hi1 = P1h.c.lo1 = P1h.c.base1 = P1h.c.hi2 = P1h.c.lo2 = P1h.c.base2 = 0;
    P1h.epi = Epilogue{};
    P1h.epi.act = EPI_NONE;
    P1h.epi.out_f32 = 1;
    P1h.epi.alpha = 1.0f;
    TP3D_TRY(make_map(&mp, gp, part, 16, 32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, CU_TENSOR_MAP_SWIZZLE_64B));
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Tc2Cfg<128>::SMEM;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2 * (unsigned)sh.clusters);
  TP3D_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemm_chain_kernel, m0.a, m0.b, m0.c, m0.z, m0.x, m1.a, m1.b, m1.c, m1.z,
                                   m1.x, mp, P0, P1, P1h, m0.wide, m1.wide, C));
  return TP3D_OK;
}

tp3d_status gemm_bf16_tc(const tp3d_ctx* ctx, const GemmProblem& P0, cudaStream_t s) {
  GemmProblem P = P0;
  P.stall_after = ctx->stall_after;
  if (P.Z < 1 || P.Hz < 1 || P.M < 1 || P.N < 1 || P.K < 1) return TP3D_EINVAL;
  if (P.segM < 1 || P.segN < 1 || P.segK < 1 || P.M % P.segM || P.N % P.segN || P.K % P.segK) return TP3D_EINVAL;
  // every operand block must be at least one TMA box wide and tall enough
  // for its 16-byte row pitch; the tile shape is picked per problem.
  const Grid* gs[3] = {&P.a.g, &P.b.g, &P.c.g};
  for (const Grid* g : gs)
    if (g->bw % 8 != 0) return TP3D_EALIGN;
  if (P.segM % 8 || P.segN % 8) return TP3D_EUNSUPPORTED;
  // fp16 output columns: whole 32-column chunks, plain outputs only
  if (P.epi.f16_cols < 0 || P.epi.f16_cols % 32 ||
      ((P.epi.f16_cols > 0 || P.epi.amax_out) &&
       (P.epi.out_f32 || P.epi.zsave || P.epi.resid || P.epi.gin || P.epi.act != EPI_NONE)))
    return TP3D_EINVAL;
  // tile decode and the epilogue's block arithmetic run in 32 bits
  for (const Grid* g : gs)
    if (g->R > INT32_MAX || g->C > INT32_MAX) return TP3D_EUNSUPPORTED;
  if (P.M > INT32_MAX || P.N > INT32_MAX || P.K > INT32_MAX) return TP3D_EUNSUPPORTED;
  // a ragged contraction tile is exact only if one operand's block ends at the segment end
  if (P.segK % BK != 0) {
    const int64_t ka = P.a.mn_major ? P.a.g.bh : P.a.g.bw;
    const int64_t kb = P.b.mn_major ? P.b.g.bh : P.b.g.bw;
    if (ka != P.segK && kb != P.segK) return TP3D_EUNSUPPORTED;
  }
  // Pick the tile shape by a wave-count cost model: the time of one SM on a
  // 128 x 256 x K slice is one unit at the shape's measured efficiency
  // (CTA pairs move the least data per product and reach the highest).
  // Pairs need no causal mask and segments that hold whole 256 x 256 tiles.
  auto tiles = [&](int64_t tm, int64_t tn) {
    return (int64_t)P.Z * (P.M / P.segM) * ((P.segM + tm - 1) / tm) * (P.N / P.segN) * ((P.segN + tn - 1) / tn);
  };
  auto waves = [&](int64_t n, int64_t slots) { return (double)((n + slots - 1) / slots); };
  const int64_t sms = ctx->num_sms;
  const double c256 = P.segN > 128 ? waves(tiles(BM, 256), sms) / 0.60 : 1e30;
  const double c128 = waves(tiles(BM, 128), sms) * 0.5 / 0.45;
  const bool pairs_ok = P.causal == CAUSAL_NONE && P.segM >= 256 && P.segN >= 256;
  const double cpair = pairs_ok ? waves(tiles(256, 256), sms / 2) / 0.80 : 1e30;
  const bool h16 = P.epi.f16_cols > 0 || P.epi.alpha_dev != nullptr || P.epi.amax_out != nullptr;
  if (cpair <= c256 && cpair <= c128) {
    if (P.segK % 128 == 0) return h16 ? launch_pair<128, true>(ctx, P, s) : launch_pair<128, false>(ctx, P, s);
    return h16 ? launch_pair<64, true>(ctx, P, s) : launch_pair<64, false>(ctx, P, s);
  }
  if (c256 <= c128) return h16 ? launch<256, true>(ctx, P, s) : launch<256, false>(ctx, P, s);
  return h16 ? launch<128, true>(ctx, P, s) : launch<128, false>(ctx, P, s);
}

tp3d_status plan_segments(GemmProblem& P) {
  auto g = [](std::initializer_list<int64_t> xs) {
    int64_t r = 0;
    for (int64_t x : xs) r = gcd64(r, x < 0 ? -x : x);
    return r;
  };
  const int64_t aM = P.a.mn_major ? P.a.g.bw : P.a.g.bh, aK = P.a.mn_major ? P.a.g.bh : P.a.g.bw;
  const int64_t bK = P.b.mn_major ? P.b.g.bh : P.b.g.bw, bN = P.b.mn_major ? P.b.g.bw : P.b.g.bh;
  P.segM = g({aM, P.c.g.bh, P.M, P.a.hi1, P.a.lo1, P.a.base1, P.c.hi1, P.c.lo1, P.c.base1});
  P.segN = g({bN, P.c.g.bw, P.N, P.b.hi2, P.b.lo2, P.b.base2, P.c.hi2, P.c.lo2, P.c.base2});
  P.segK = g({aK, bK, P.K, P.a.hi2, P.a.lo2, P.a.base2, P.b.hi1, P.b.lo1, P.b.base1});
  if (P.segM <= 0 || P.segN <= 0 || P.segK <= 0) return TP3D_ESHAPE;
  return TP3D_OK;
}

}  // namespace tp3d
