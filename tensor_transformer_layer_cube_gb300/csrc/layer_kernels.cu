// layer_kernels.cu - the bandwidth-bound kernels of the GPT layer on the cube.
//
// "Maximizing Parallelism in Distributed Training for Huge Neural Networks"
// §3.2 builds the 3-D LayerNorm from the matrix-vector operations of §3.1.3
// (C = A * gamma, C = A + beta, Algorithms 7-8 and the gamma gradient
// sum(dC * A-hat)); the row statistics and the attention core are not
// partitioned by the page.  Here a row that the cube splits into q column
// blocks (CUBE_A: blocks l = 0..q-1 of shard row (i, j)) is handled by one
// warp that reads its q pieces, so the statistics are those of the whole
// row.  All of these kernels are HBM-bound: 16-byte vector accesses, fp32
// arithmetic, one pass over the data where possible.
#include <cudaTypedefs.h>

#include "layer_kernels.cuh"

namespace tp3d {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
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

// fp16 form of 8 values; a value beyond fp16's finite range raises TP3D_ERANGE
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

using bf16 = __nv_bfloat16;

// ------------------------------------------------------------------ LayerNorm
// y16 (or null): the same output in fp16, in y's layout
__global__ void __launch_bounds__(kThreads) ln_fwd_kernel(const Grid g, const bf16* __restrict__ x,
                                                          const bf16* __restrict__ gamma,
                                                          const bf16* __restrict__ beta, bf16* __restrict__ y,
                                                          __half* __restrict__ y16, int* err,
                                                          float* __restrict__ mean, float* __restrict__ rstd,
                                                          float eps) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * kWarps;
  const int64_t vpb = g.bw / 8;
  const float invC = 1.0f / (float)g.C;
  for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < g.R; r += nwarps) {
    const int64_t br = r / g.bh, rr = r - br * g.bh;
    float s1 = 0.0f;
    for (int32_t bc = 0; bc < g.cb; ++bc) {
      const uint4* p = reinterpret_cast<const uint4*>(x + g.block_base((int32_t)br, bc) + rr * g.bw);
      for (int64_t v = lane; v < vpb; v += 32) {
        float f[8];
        unpack8(p[v], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) s1 += f[e];
      }
    }
    const float mu = warp_sum(s1) * invC;
    float s2 = 0.0f;
    for (int32_t bc = 0; bc < g.cb; ++bc) {
      const uint4* p = reinterpret_cast<const uint4*>(x + g.block_base((int32_t)br, bc) + rr * g.bw);
      for (int64_t v = lane; v < vpb; v += 32) {
        float f[8];
        unpack8(p[v], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) s2 += (f[e] - mu) * (f[e] - mu);
      }
    }
    const float rs = rsqrtf(warp_sum(s2) * invC + eps);
    for (int32_t bc = 0; bc < g.cb; ++bc) {
      const int64_t off = g.block_base((int32_t)br, bc) + rr * g.bw;
      const uint4* p = reinterpret_cast<const uint4*>(x + off);
      uint4* q = reinterpret_cast<uint4*>(y + off);
      const uint4* gp = reinterpret_cast<const uint4*>(gamma + (int64_t)bc * g.bw);
      const uint4* bp = reinterpret_cast<const uint4*>(beta + (int64_t)bc * g.bw);
      for (int64_t v = lane; v < vpb; v += 32) {
        float f[8], gg[8], bb[8], o[8];
        unpack8(p[v], f);
        unpack8(gp[v], gg);
        unpack8(bp[v], bb);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = (f[e] - mu) * rs * gg[e] + bb[e];
        q[v] = pack8(o);
        if (y16) reinterpret_cast<uint4*>(y16 + off)[v] = pack8h(o, err);
      }
    }
    if (lane == 0) {
      mean[r] = mu;
      rstd[r] = rs;
    }
  }
}

__global__ void __launch_bounds__(kThreads) ln_bwd_kernel(const Grid g, const bf16* __restrict__ dy,
                                                          const bf16* __restrict__ x, const float* __restrict__ mean,
                                                          const float* __restrict__ rstd,
                                                          const bf16* __restrict__ gamma,
                                                          const bf16* __restrict__ dres, bf16* __restrict__ dx) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * kWarps;
  const int64_t vpb = g.bw / 8;
  const float invC = 1.0f / (float)g.C;
  for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < g.R; r += nwarps) {
    const int64_t br = r / g.bh, rr = r - br * g.bh;
    const float mu = mean[r], rs = rstd[r];
    float a = 0.0f, b = 0.0f;
    for (int32_t bc = 0; bc < g.cb; ++bc) {
      const int64_t off = g.block_base((int32_t)br, bc) + rr * g.bw;
      const uint4* dp = reinterpret_cast<const uint4*>(dy + off);
      const uint4* xp = reinterpret_cast<const uint4*>(x + off);
      const uint4* gp = reinterpret_cast<const uint4*>(gamma + (int64_t)bc * g.bw);
      for (int64_t v = lane; v < vpb; v += 32) {
        float d[8], xv[8], gg[8];
        unpack8(dp[v], d);
        unpack8(xp[v], xv);
        unpack8(gp[v], gg);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float dxh = d[e] * gg[e];
          a += dxh;
          b += dxh * (xv[e] - mu) * rs;
        }
      }
    }
    a = warp_sum(a) * invC;
    b = warp_sum(b) * invC;
    for (int32_t bc = 0; bc < g.cb; ++bc) {
      const int64_t off = g.block_base((int32_t)br, bc) + rr * g.bw;
      const uint4* dp = reinterpret_cast<const uint4*>(dy + off);
      const uint4* xp = reinterpret_cast<const uint4*>(x + off);
      const uint4* rp = reinterpret_cast<const uint4*>(dres + off);
      const uint4* gp = reinterpret_cast<const uint4*>(gamma + (int64_t)bc * g.bw);
      uint4* op = reinterpret_cast<uint4*>(dx + off);
      for (int64_t v = lane; v < vpb; v += 32) {
        float d[8], xv[8], gg[8], rv[8], o[8];
        unpack8(dp[v], d);
        unpack8(xp[v], xv);
        unpack8(gp[v], gg);
        unpack8(rp[v], rv);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = rv[e] + rs * (d[e] * gg[e] - a - (xv[e] - mu) * rs * b);
        op[v] = pack8(o);
      }
    }
  }
}

// LayerNorm forward with the whole row staged in shared memory: C = NV * 256,
// lane l holds columns 8 (l + 32 i) .. +7 for i < NV.  Every load of a row is
// an asynchronous 16-byte copy into the warp's slice of shared memory, all
// issued before the first use, so a warp spends one memory round trip per
// row while holding no registers for the row; the statistics take two passes
// over the staged row.  gamma and beta are staged once per CTA.  A CTA takes
// (8 + 2) NV KiB / 2 of shared memory and few registers, so a grid of one row
// per warp is resident at once (a row held in registers needs more than 64 of
// them per thread, and the grid then runs in two rounds).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <int NV>
__device__ __forceinline__ int64_t row_vec_off(const Grid& g, int64_t br, int64_t rr, int lane, int i) {
  const int32_t col = (lane + 32 * i) * 8;
  const int32_t bc = col / (int32_t)g.bw;
  return g.block_base((int32_t)br, bc) + rr * g.bw + (col - (int64_t)bc * g.bw);
}

template <int NV>
constexpr int ln_row_smem() { return (kWarps + 2) * NV * 32 * 16; }  // the CTA's rows, then gamma and beta

template <int NV>
__global__ void __launch_bounds__(kThreads) ln_fwd_row_kernel(const Grid g, const bf16* __restrict__ x,
                                                              const bf16* __restrict__ gamma,
                                                              const bf16* __restrict__ beta, bf16* __restrict__ y,
                                                              __half* __restrict__ y16, int* err,
                                                              float* __restrict__ mean, float* __restrict__ rstd,
                                                              float eps) {
  constexpr float invC = 1.0f / (float)(NV * 256);
  extern __shared__ uint4 ln_rows[];
  const uint4* sg = ln_rows + kWarps * NV * 32;
  const uint4* sb = sg + NV * 32;
  for (int i = threadIdx.x; i < NV * 32; i += kThreads) {
    ln_rows[kWarps * NV * 32 + i] = __ldg(reinterpret_cast<const uint4*>(gamma) + i);
    ln_rows[(kWarps + 1) * NV * 32 + i] = __ldg(reinterpret_cast<const uint4*>(beta) + i);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const uint4* row = ln_rows + (threadIdx.x >> 5) * NV * 32;  // this warp's row
  const uint32_t row_s = smem_u32(row);
  const int64_t nwarps = (int64_t)gridDim.x * kWarps;
  for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < g.R; r += nwarps) {
    const int64_t br = r / g.bh, rr = r - br * g.bh;
    // each lane copies, and later reads back, only its own 16-byte pieces
#pragma unroll
    for (int i = 0; i < NV; ++i)
      cp_async16(row_s + (uint32_t)(lane + 32 * i) * 16u, x + row_vec_off<NV>(g, br, rr, lane, i));
    cp_async_wait_all();
    float s1 = 0.0f;
#pragma unroll 2
    for (int i = 0; i < NV; ++i) {
      float f[8];
      unpack8(row[lane + 32 * i], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) s1 += f[e];
    }
    const float mu = warp_sum(s1) * invC;
    // each pass reads the row (and gamma, beta) from shared memory again, two
    // vectors at a time: values kept from a pass before, or all of a pass's
    // reads hoisted ahead, would cost a register per column
    asm volatile("" ::: "memory");
    float s2 = 0.0f;
#pragma unroll 2
    for (int i = 0; i < NV; ++i) {
      float f[8];
      unpack8(row[lane + 32 * i], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) s2 += (f[e] - mu) * (f[e] - mu);
    }
    const float rs = rsqrtf(warp_sum(s2) * invC + eps);
    asm volatile("" ::: "memory");
#pragma unroll 2
    for (int i = 0; i < NV; ++i) {
      float f[8], gg[8], bb[8], o[8];
      unpack8(row[lane + 32 * i], f);
      unpack8(sg[lane + 32 * i], gg);
      unpack8(sb[lane + 32 * i], bb);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = (f[e] - mu) * rs * gg[e] + bb[e];
      const int64_t off = row_vec_off<NV>(g, br, rr, lane, i);
      *reinterpret_cast<uint4*>(y + off) = pack8(o);
      if (y16) *reinterpret_cast<uint4*>(y16 + off) = pack8h(o, err);
    }
    if (lane == 0) {
      mean[r] = mu;
      rstd[r] = rs;
    }
  }
}

// ------------------------------------------------------------------ bf16 -> scaled fp16
// amax = max |x| over n bf16 values (n a multiple of 8), as the bits of a
// non-negative float (integer order = float order), by an atomic max per CTA.
__global__ void __launch_bounds__(kThreads) absmax_kernel(const bf16* __restrict__ x, int64_t n,
                                                          unsigned* __restrict__ amax) {
  __shared__ float red[kWarps];
  float m = 0.0f;
  const int64_t nv = n / 8;
  for (int64_t v = (int64_t)blockIdx.x * kThreads + threadIdx.x; v < nv; v += (int64_t)gridDim.x * kThreads) {
    float f[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(x) + v), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(f[e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < kWarps; ++k) m = fmaxf(m, red[k]);
    atomicMax(amax, __float_as_uint(m));
  }
}

// The power of two 2^k that puts amax in [2^14, 2^15) (1 for amax 0 or not
// finite).  Every finite bf16 value w then has |w 2^k| <= 2^15, and w 2^k is
// exact in fp16 when |w| >= amax 2^-28 (fp16's normal range holds bf16's 8
// significant bits); smaller magnitudes keep an absolute error below
// amax 2^-39.
__device__ __forceinline__ int f16_scale_exp(float amax) {
  if (!(amax > 0.0f) || !(amax <= 3.0e38f)) return 0;
  int e;
  frexpf(amax, &e);  // amax = m 2^e, m in [0.5, 1)
  return 15 - e;
}

// y = fp16(x 2^k) with k from amax; inv_scale = 2^-k (written by one thread).
// A non-finite amax raises TP3D_ERANGE.
__global__ void __launch_bounds__(kThreads) to_f16_scaled_kernel(const bf16* __restrict__ x, int64_t n,
                                                                 const unsigned* __restrict__ amax,
                                                                 __half* __restrict__ y,
                                                                 float* __restrict__ inv_scale, int* err) {
  const float am = __uint_as_float(*amax);
  const int k = f16_scale_exp(am);
  const float sc = ldexpf(1.0f, k);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *inv_scale = ldexpf(1.0f, -k);
    if (!(am <= 3.0e38f)) raise_error(err, TP3D_ERANGE);
  }
  const int64_t nv = n / 8;
  for (int64_t v = (int64_t)blockIdx.x * kThreads + threadIdx.x; v < nv; v += (int64_t)gridDim.x * kThreads) {
    float f[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(x) + v), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] *= sc;
    reinterpret_cast<uint4*>(y)[v] = pack8h(f, nullptr);
  }
}

// ------------------------------------------------------------------ column sums
// CTA (x, y): columns [256 x, +256) over the rows of part y (rows_per_part
// rows inside one row block); lane l of every warp holds columns 8l..8l+7,
// warps stride over rows with U rows' loads in flight (16, or 8 when each
// row brings two inputs); the 8 warps are
// summed in shared memory into the part's partial row.  The last CTA of a
// column strip to finish (an atomic count per strip, reset to zero after)
// adds the partial rows of all parts and writes the bf16 sums.
// LN: sums dy * (x - mean) * rstd into out and dy into out2 (the LayerNorm
// gamma and beta gradients); else sums x into out.
template <bool LN>
__global__ void __launch_bounds__(kThreads) colsum_kernel(const Grid g, const bf16* __restrict__ x,
                                                          const bf16* __restrict__ dy,
                                                          const float* __restrict__ mean,
                                                          const float* __restrict__ rstd, float* __restrict__ part,
                                                          float* __restrict__ part2, int64_t rows_per_part,
                                                          int* __restrict__ counters, bf16* __restrict__ out,
                                                          bf16* __restrict__ out2) {
  constexpr int U = LN ? 8 : 16;  // rows in flight per warp
  __shared__ float red[kWarps][257];
  __shared__ int is_last;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * 256 + lane * 8;
  const int64_t r0 = (int64_t)blockIdx.y * rows_per_part;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0}, acc2[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (c < g.C) {
    const int64_t br = r0 / g.bh, bc = c / g.bw;
    const int64_t base = g.block_base((int32_t)br, (int32_t)bc) + (r0 - br * g.bh) * g.bw + (c - bc * g.bw);
    for (int64_t rr0 = w; rr0 < rows_per_part; rr0 += (int64_t)kWarps * U) {
      uint4 xv[U], dv[U];
      float mu[U], rs[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t rr = rr0 + (int64_t)u * kWarps;
        if (rr < rows_per_part) {
          xv[u] = *reinterpret_cast<const uint4*>(x + base + rr * g.bw);
          if (LN) {
            dv[u] = *reinterpret_cast<const uint4*>(dy + base + rr * g.bw);
            mu[u] = mean[r0 + rr];
            rs[u] = rstd[r0 + rr];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (rr0 + (int64_t)u * kWarps >= rows_per_part) break;
        float f[8];
        unpack8(xv[u], f);
        if (!LN) {
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[e] += f[e];
        } else {
          float d[8];
          unpack8(dv[u], d);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            acc[e] += d[e] * (f[e] - mu[u]) * rs[u];
            acc2[e] += d[e];
          }
        }
      }
    }
  }
  const int64_t cc = (int64_t)blockIdx.x * 256 + threadIdx.x;
#pragma unroll
  for (int e = 0; e < 8; ++e) red[w][lane * 8 + e] = acc[e];
  __syncthreads();
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < kWarps; ++k) s += red[k][threadIdx.x];
  if (cc < g.C) part[(int64_t)blockIdx.y * g.C + cc] = s;
  if (LN) {
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 8; ++e) red[w][lane * 8 + e] = acc2[e];
    __syncthreads();
    s = 0.0f;
#pragma unroll
    for (int k = 0; k < kWarps; ++k) s += red[k][threadIdx.x];
    if (cc < g.C) part2[(int64_t)blockIdx.y * g.C + cc] = s;
  }
  // the last part of this strip to finish reduces all of them: the block's
  // writes are ordered before its arrival by the barrier and thread 0's
  // (cumulative) device-scope fence
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    is_last = atomicAdd(&counters[blockIdx.x], 1) == (int)gridDim.y - 1;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // warp w adds parts w, w + 8, ...; lane l columns 8l..8l+7 of the strip
  for (int which = 0; which < (LN ? 2 : 1); ++which) {
    const float* src = which == 0 ? part : part2;
    float t[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (c < g.C) {
      const int64_t np = gridDim.y;
      for (int64_t p0 = w; p0 < np; p0 += (int64_t)kWarps * 4) {
        float4 v[4][2];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t p = p0 + (int64_t)u * kWarps;
          if (p < np) {
            v[u][0] = __ldcg(reinterpret_cast<const float4*>(src + p * g.C + c));
            v[u][1] = __ldcg(reinterpret_cast<const float4*>(src + p * g.C + c + 4));
          } else {
            v[u][0] = v[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          t[0] += v[u][0].x;
          t[1] += v[u][0].y;
          t[2] += v[u][0].z;
          t[3] += v[u][0].w;
          t[4] += v[u][1].x;
          t[5] += v[u][1].y;
          t[6] += v[u][1].z;
          t[7] += v[u][1].w;
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 8; ++e) red[w][lane * 8 + e] = t[e];
    __syncthreads();
    float u = 0.0f;
#pragma unroll
    for (int k = 0; k < kWarps; ++k) u += red[k][threadIdx.x];
    if (cc < g.C) (which == 0 ? out : out2)[cc] = __float2bfloat16_rn(u);
  }
  if (threadIdx.x == 0) counters[blockIdx.x] = 0;
}

// ---------------------------------------------------- column sums fed by TMA
// The same sums as colsum_kernel, with the rows streamed through shared
// memory: warp 8 issues 256-column x 32-row TMA boxes into a ring of kSkStages
// stages (the data in flight takes no registers, so a CTA keeps up to
// kSkStages x 16 KiB per input moving), warps 0-7 read rows w, w + 8, w + 16,
// w + 24 of each box, lane l columns 8l..8l+7.  Then the partial rows and the
// last-CTA reduction of colsum_kernel.
constexpr int kSkStages = 6;               // boxes in flight (LN: 3, two inputs per box)
constexpr int kBoxRows = 32;
constexpr uint32_t kBoxBytes = kBoxRows * 256 * 2;
constexpr int kSkThreads = 288;

template <bool LN>
TP3D_HD constexpr int sk_stages() { return LN ? kSkStages / 2 : kSkStages; }
template <bool LN>
TP3D_HD constexpr int sk_smem() { return sk_stages<LN>() * (LN ? 2 : 1) * (int)kBoxBytes + kWarps * 257 * 4 + 256 + 128; }

template <bool LN>
__global__ void __launch_bounds__(kSkThreads) colsum_tma_kernel(const __grid_constant__ CUtensorMap mx,
                                                                const __grid_constant__ CUtensorMap mdy, const Grid g,
                                                                const float* __restrict__ mean,
                                                                const float* __restrict__ rstd,
                                                                float* __restrict__ part, float* __restrict__ part2,
                                                                int64_t rows_per_part, int* __restrict__ counters,
                                                                bf16* __restrict__ out, bf16* __restrict__ out2,
                                                                int* err) {
  constexpr int NS = sk_stages<LN>();
  constexpr uint32_t STAGE = (LN ? 2u : 1u) * kBoxBytes;
  extern __shared__ __align__(128) uint8_t sk_smem_raw[];
  uint8_t* ring = sk_smem_raw;
  float(*red)[257] = reinterpret_cast<float(*)[257]>(ring + NS * STAGE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + NS * STAGE + kWarps * 257 * 4);
  int* is_last = reinterpret_cast<int*>(bars + 2 * NS);
  volatile int* abort_flag = is_last + 1;
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int st) { return bar0 + 8u * st; };
  auto empty = [&](int st) { return bar0 + 8u * (NS + st); };
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t c0 = (int64_t)blockIdx.x * 256;
  const int64_t r0 = (int64_t)blockIdx.y * rows_per_part;
  const int nb = (int)(rows_per_part / kBoxRows);
  if (threadIdx.x == 0) {
    for (int st = 0; st < NS; ++st) {
      mbar_init(full(st), 1);
      mbar_init(empty(st), kWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0}, acc2[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  bool ok = true;
  if (w == kWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int32_t br = (int32_t)((uint32_t)r0 / (uint32_t)g.bh), bc = (int32_t)((uint32_t)c0 / (uint32_t)g.bw);
      const int sh = g.shard(br, bc);
      const int cin = (int)(c0 - (int64_t)bc * g.bw), rin0 = (int)(r0 - (int64_t)br * g.bh);
      int b = 0;
      for (; b < nb && ok; ++b) {
        const int st = b % NS;
        if (!(ok = mbar_wait(empty(st), ((b / NS) & 1) ^ 1, abort_flag, err))) break;
        mbar_arrive_expect_tx(full(st), STAGE);
        tma_load_3d(smem_u32(ring + st * STAGE), &mx, full(st), cin, rin0 + b * kBoxRows, sh);
        if (LN) tma_load_3d(smem_u32(ring + st * STAGE + kBoxBytes), &mdy, full(st), cin, rin0 + b * kBoxRows, sh);
      }
      if (!ok) {  // every issued box lands before the CTA may leave
        for (int j = b - NS > 0 ? b - NS : 0; j < b; ++j) {
          const unsigned long long t0 = globaltimer_ns();
          while (!mbar_try_wait(full(j % NS), (j / NS) & 1))
            if (globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    for (int b = 0; b < nb && ok; ++b) {
      const int st = b % NS;
      float mu[4], rs[4];
      if (LN) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int64_t r = r0 + (int64_t)b * kBoxRows + w + 8 * k;
          mu[k] = __ldg(mean + r);
          rs[k] = __ldg(rstd + r);
        }
      }
      bool got = lane == 0 ? mbar_wait(full(st), (b / NS) & 1, abort_flag, err) : false;
      got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      if (!(ok = got)) break;
      const uint8_t* box = ring + st * STAGE;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int row = w + 8 * k;
        float f[8];
        unpack8(*reinterpret_cast<const uint4*>(box + row * 512 + lane * 16), f);
        if (!LN) {
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[e] += f[e];
        } else {
          float d[8];
          unpack8(*reinterpret_cast<const uint4*>(box + kBoxBytes + row * 512 + lane * 16), d);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            acc[e] += d[e] * (f[e] - mu[k]) * rs[k];
            acc2[e] += d[e];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(st));
    }
  }
  // every role reaches here: an aborted CTA leaves without writing
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  if (!ok) return;
  const int tid = threadIdx.x;
  if (w < kWarps) {
#pragma unroll
    for (int e = 0; e < 8; ++e) red[w][lane * 8 + e] = acc[e];
  }
  __syncthreads();
  if (tid < 256) {
    float sum = 0.0f;
#pragma unroll
    for (int k = 0; k < kWarps; ++k) sum += red[k][tid];
    part[(int64_t)blockIdx.y * g.C + c0 + tid] = sum;
  }
  if (LN) {
    __syncthreads();
    if (w < kWarps) {
#pragma unroll
      for (int e = 0; e < 8; ++e) red[w][lane * 8 + e] = acc2[e];
    }
    __syncthreads();
    if (tid < 256) {
      float sum = 0.0f;
#pragma unroll
      for (int k = 0; k < kWarps; ++k) sum += red[k][tid];
      part2[(int64_t)blockIdx.y * g.C + c0 + tid] = sum;
    }
  }
  // the last part of this strip to finish reduces all of them (as colsum_kernel)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    *is_last = atomicAdd(&counters[blockIdx.x], 1) == (int)gridDim.y - 1;
  }
  __syncthreads();
  if (!*is_last) return;
  __threadfence();
  for (int which = 0; which < (LN ? 2 : 1); ++which) {
    const float* src = which == 0 ? part : part2;
    float t[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (w < kWarps) {
      const int64_t np = gridDim.y, c = c0 + lane * 8;
      for (int64_t p0 = w; p0 < np; p0 += (int64_t)kWarps * 4) {
        float4 v[4][2];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t pp = p0 + (int64_t)u * kWarps;
          if (pp < np) {
            v[u][0] = __ldcg(reinterpret_cast<const float4*>(src + pp * g.C + c));
            v[u][1] = __ldcg(reinterpret_cast<const float4*>(src + pp * g.C + c + 4));
          } else {
            v[u][0] = v[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          t[0] += v[u][0].x;
          t[1] += v[u][0].y;
          t[2] += v[u][0].z;
          t[3] += v[u][0].w;
          t[4] += v[u][1].x;
          t[5] += v[u][1].y;
          t[6] += v[u][1].z;
          t[7] += v[u][1].w;
        }
      }
    }
    __syncthreads();
    if (w < kWarps) {
#pragma unroll
      for (int e = 0; e < 8; ++e) red[w][lane * 8 + e] = t[e];
    }
    __syncthreads();
    if (tid < 256) {
      float u = 0.0f;
#pragma unroll
      for (int k = 0; k < kWarps; ++k) u += red[k][tid];
      (which == 0 ? out : out2)[c0 + tid] = __float2bfloat16_rn(u);
    }
  }
  if (tid == 0) counters[blockIdx.x] = 0;
}

PFN_cuTensorMapEncodeTiled_v12000 sk_encode() {
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

// (column in shard, row in shard, shard) map with 256 x 32 boxes, unswizzled
bool sk_map(CUtensorMap* m, const Grid& g, const void* ptr) {
  auto fn = sk_encode();
  if (!fn || !aligned16(ptr)) return false;
  cuuint64_t dims[3] = {(cuuint64_t)g.bw, (cuuint64_t)g.bh, (cuuint64_t)g.nshards()};
  cuuint64_t strides[2] = {(cuuint64_t)g.bw * 2, (cuuint64_t)(g.bh * g.bw * 2)};
  cuuint32_t box[3] = {256, (cuuint32_t)kBoxRows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The TMA-fed column sums, when every 256-column strip lies in one shard
// column and the parts divide the row blocks; false = use colsum_kernel.
template <bool LN>
bool launch_colsum_tma(const tp3d_ctx* ctx, const Grid& g, const void* x, const void* dy, const float* mean,
                       const float* rstd, float* part, float* part2, int* counters, void* out, void* out2,
                       cudaStream_t s, tp3d_status* st) {
  if (g.C % 256 || g.bw % 256 || g.bh % kBoxRows || g.R > INT32_MAX || g.C > INT32_MAX) return false;
  static int per_sm[64] = {};
  const int dev = ctx->device & 63;
  if (per_sm[dev] == 0) {
    int n = 0;
    if (cudaFuncSetAttribute(colsum_tma_kernel<LN>, cudaFuncAttributeMaxDynamicSharedMemorySize, sk_smem<LN>()) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, colsum_tma_kernel<LN>, kSkThreads, sk_smem<LN>()) !=
            cudaSuccess ||
        n < 1) {
      (void)cudaGetLastError();
      n = -1;
    }
    per_sm[dev] = n;
  }
  if (per_sm[dev] < 1) return false;
  const int64_t strips = g.C / 256, slots = (int64_t)per_sm[dev] * ctx->num_sms;
  // rows per part: the smallest power of two from 64 with one resident round
  int64_t rpp = 64;
  while (rpp < g.bh && strips * ((g.R + rpp - 1) / rpp) > slots) rpp *= 2;
  if (g.bh % rpp || g.R % rpp || g.R / rpp > 65535) return false;
  CUtensorMap mx, mdy;
  if (!sk_map(&mx, g, x)) return false;
  if (LN) {
    if (!sk_map(&mdy, g, dy)) return false;
  } else {
    mdy = mx;
  }
  const dim3 grid((unsigned)strips, (unsigned)(g.R / rpp));
  colsum_tma_kernel<LN><<<grid, kSkThreads, sk_smem<LN>(), s>>>(mx, mdy, g, mean, rstd, part, part2, rpp, counters,
                                                                static_cast<bf16*>(out), static_cast<bf16*>(out2),
                                                                ctx->d_err);
  *st = cudaGetLastError() == cudaSuccess ? TP3D_OK : TP3D_ECUDA;
  return true;
}

unsigned grid_for_rows(const tp3d_ctx* ctx, int64_t rows, int per_sm) {
  int64_t g = (rows + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)ctx->num_sms * per_sm;
  return (unsigned)(g < cap ? (g > 0 ? g : 1) : cap);
}

tp3d_status last_error() { return cudaGetLastError() == cudaSuccess ? TP3D_OK : TP3D_ECUDA; }

}  // namespace

template <int NV>
void ln_fwd_row(unsigned grid, cudaStream_t s, const Grid& g, const bf16* x, const bf16* gamma, const bf16* beta,
                bf16* y, __half* y16, int* err, float* mean, float* rstd, float eps) {
  if (ln_row_smem<NV>() > 48 * 1024)
    (void)cudaFuncSetAttribute(ln_fwd_row_kernel<NV>, cudaFuncAttributeMaxDynamicSharedMemorySize, ln_row_smem<NV>());
  ln_fwd_row_kernel<NV><<<grid, kThreads, ln_row_smem<NV>(), s>>>(g, x, gamma, beta, y, y16, err, mean, rstd, eps);
}

tp3d_status launch_ln_fwd(const tp3d_ctx* ctx, const Grid& g, const void* x, const void* gamma, const void* beta,
                          void* y, void* y16, float* mean, float* rstd, float eps, cudaStream_t s) {
  const unsigned grid = grid_for_rows(ctx, g.R, 16);
  const bf16 *xb = static_cast<const bf16*>(x), *gb = static_cast<const bf16*>(gamma),
             *bb = static_cast<const bf16*>(beta);
  bf16* yb = static_cast<bf16*>(y);
  __half* yh = static_cast<__half*>(y16);
  int* err = ctx->d_err;
  switch (g.C % 256 == 0 ? g.C / 256 : 0) {  // whole rows staged in shared memory where C = 256 NV
    case 2: ln_fwd_row<2>(grid, s, g, xb, gb, bb, yb, yh, err, mean, rstd, eps); break;
    case 4: ln_fwd_row<4>(grid, s, g, xb, gb, bb, yb, yh, err, mean, rstd, eps); break;
    case 8: ln_fwd_row<8>(grid, s, g, xb, gb, bb, yb, yh, err, mean, rstd, eps); break;
    case 16: ln_fwd_row<16>(grid, s, g, xb, gb, bb, yb, yh, err, mean, rstd, eps); break;
    default: ln_fwd_kernel<<<grid, kThreads, 0, s>>>(g, xb, gb, bb, yb, yh, err, mean, rstd, eps);
  }
  return last_error();
}

tp3d_status launch_to_f16_scaled(const tp3d_ctx* ctx, const void* x, int64_t n, unsigned* amax, void* y,
                                 float* inv_scale, cudaStream_t s) {
  if (n <= 0 || n % 8) return TP3D_EINVAL;
  TP3D_CUDA_TRY(cudaMemsetAsync(amax, 0, sizeof(unsigned), s));
  const int64_t blocks = (n / 8 + kThreads - 1) / kThreads, cap = (int64_t)ctx->num_sms * 8;
  const unsigned grid = (unsigned)(blocks < cap ? blocks : cap);
  absmax_kernel<<<grid, kThreads, 0, s>>>(static_cast<const bf16*>(x), n, amax);
  TP3D_CUDA_TRY(cudaGetLastError());
  to_f16_scaled_kernel<<<grid, kThreads, 0, s>>>(static_cast<const bf16*>(x), n, amax, static_cast<__half*>(y),
                                                 inv_scale, ctx->d_err);
  return last_error();
}

tp3d_status launch_ln_bwd(const tp3d_ctx* ctx, const Grid& g, const void* dy, const void* x, const float* mean,
                          const float* rstd, const void* gamma, const void* dres, void* dx, cudaStream_t s) {
  const unsigned grid = grid_for_rows(ctx, g.R, 16);
  const bf16 *db = static_cast<const bf16*>(dy), *xb = static_cast<const bf16*>(x),
             *gb = static_cast<const bf16*>(gamma), *rb = static_cast<const bf16*>(dres);
  bf16* ob = static_cast<bf16*>(dx);
  ln_bwd_kernel<<<grid, kThreads, 0, s>>>(g, db, xb, mean, rstd, gb, rb, ob);
  return last_error();
}

int64_t colsum_strips(const Grid& g) { return (g.C + 255) / 256; }
// the most parts any launch uses (64-row parts), for sizing the scratch
int64_t colsum_parts(const Grid& g) { return g.R / gcd64(g.bh, 64); }
// rows per part: the smallest power of two (64..1024, dividing the row
// block) for which every CTA is resident at once (one round, no tail wave)
template <bool LN>
int64_t colsum_rows(const tp3d_ctx* ctx, const Grid& g) {
  static int per_sm[64] = {};
  const int dev = ctx->device & 63;
  if (per_sm[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, colsum_kernel<LN>, kThreads, 0) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      n = 1;
    }
    per_sm[dev] = n;
  }
  const int64_t slots = (int64_t)per_sm[dev] * ctx->num_sms;
  int64_t p = 64;
  while (p < 1024 && colsum_strips(g) * ((g.R + p - 1) / p) > slots) p *= 2;
  return gcd64(g.bh, p);
}

tp3d_status launch_colsum(const tp3d_ctx* ctx, const Grid& g, const void* x, float* part, int* counters, void* out,
                          cudaStream_t s) {
  tp3d_status st;
  if (launch_colsum_tma<false>(ctx, g, x, nullptr, nullptr, nullptr, part, nullptr, counters, out, nullptr, s, &st))
    return st;
  const int64_t rpp = colsum_rows<false>(ctx, g);
  const dim3 grid((unsigned)colsum_strips(g), (unsigned)(g.R / rpp));
  if (grid.y > 65535u) return TP3D_EUNSUPPORTED;
  colsum_kernel<false><<<grid, kThreads, 0, s>>>(g, static_cast<const bf16*>(x), nullptr, nullptr, nullptr, part,
                                                 nullptr, rpp, counters, static_cast<bf16*>(out), nullptr);
  return last_error();
}

tp3d_status launch_ln_param_grads(const tp3d_ctx* ctx, const Grid& g, const void* dy, const void* x,
                                  const float* mean, const float* rstd, float* part, int* counters, void* out_g,
                                  void* out_b, cudaStream_t s) {
  {
    const int64_t np = g.R / gcd64(g.bh, 64);  // parts the scratch is sized for
    tp3d_status st;
    if (launch_colsum_tma<true>(ctx, g, x, dy, mean, rstd, part, part + np * g.C, counters, out_g, out_b, s, &st))
      return st;
  }
  const int64_t rpp = colsum_rows<true>(ctx, g);
  const dim3 grid((unsigned)colsum_strips(g), (unsigned)(g.R / rpp));
  if (grid.y > 65535u) return TP3D_EUNSUPPORTED;
  colsum_kernel<true><<<grid, kThreads, 0, s>>>(g, static_cast<const bf16*>(x), static_cast<const bf16*>(dy), mean,
                                                rstd, part, part + (int64_t)grid.y * g.C, rpp, counters,
                                                static_cast<bf16*>(out_g), static_cast<bf16*>(out_b));
  return last_error();
}

}  // namespace tp3d
