// gemm_simt.cu - the sharded, batched GEMM in fp32 on the CUDA cores
// (FFMA, no TF32), for fp32 problems.
//
// Same problem description as the tensor-core kernel (gemm.cuh); every
// element is addressed through its operand's layout, so the all-gathers of
// "Maximizing Parallelism in Distributed Training for Huge Neural Networks",
// Algorithm 1, are plain reads of the shards.  The contraction runs over k in
// ascending order - over the depth index l first to last - into one fp32
// accumulator per output element (the reduce-scatter over z).
#include "gemm.cuh"

namespace tp3d {

namespace {

constexpr int T = 16;

__device__ __forceinline__ float gelu_f(float x) { return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f)); }
__device__ __forceinline__ float gelu_grad_f(float x) {
  const float cdf = 0.5f * (1.0f + erff(x * 0.70710678118654752f));
  return cdf + x * 0.39894228040143268f * expf(-0.5f * x * x);
}

__device__ __forceinline__ bool causal_k_ok(const GemmProblem& P, int64_t m, int64_t k) {
  if (P.causal == CAUSAL_K_LE_M) return k <= m;
  if (P.causal == CAUSAL_K_GE_M) return k >= m;
  return true;
}

__global__ void __launch_bounds__(T * T) gemm_simt_kernel(const GemmProblem P) {
  __shared__ float As[T][T + 1];
  __shared__ float Bs[T][T + 1];
  const int32_t z = blockIdx.z;
  const int64_t m = (int64_t)blockIdx.y * T + threadIdx.y;
  const int64_t n = (int64_t)blockIdx.x * T + threadIdx.x;
  const float* A = static_cast<const float*>(P.a.ptr);
  const float* B = static_cast<const float*>(P.b.ptr);
  const int64_t am = op_off(P.a.hi1, P.a.lo1, P.a.base1, z, P.Hz), ak = op_off(P.a.hi2, P.a.lo2, P.a.base2, z, P.Hz);
  const int64_t bk = op_off(P.b.hi1, P.b.lo1, P.b.base1, z, P.Hz), bn = op_off(P.b.hi2, P.b.lo2, P.b.base2, z, P.Hz);
  float acc = 0.0f;
  for (int64_t k0 = 0; k0 < P.K; k0 += T) {
    {
      const int64_t mm = (int64_t)blockIdx.y * T + threadIdx.y, kk = k0 + threadIdx.x;
      float v = 0.0f;
      if (mm < P.M && kk < P.K)
        v = P.a.mn_major ? A[P.a.g.offset(ak + kk, am + mm)] : A[P.a.g.offset(am + mm, ak + kk)];
      As[threadIdx.y][threadIdx.x] = v;
    }
    {
      const int64_t kk = k0 + threadIdx.y, nn = (int64_t)blockIdx.x * T + threadIdx.x;
      float v = 0.0f;
      if (kk < P.K && nn < P.N)
        v = P.b.mn_major ? B[P.b.g.offset(bk + kk, bn + nn)] : B[P.b.g.offset(bn + nn, bk + kk)];
      Bs[threadIdx.y][threadIdx.x] = v;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < T; ++t)
      if (causal_k_ok(P, m, k0 + t)) acc = fmaf(As[threadIdx.y][t], Bs[t][threadIdx.x], acc);
    __syncthreads();
  }
  if (m >= P.M || n >= P.N) return;
  if (P.causal == CAUSAL_SKIP_UPPER && n > m) return;
  const int64_t gm = m + op_off(P.c.hi1, P.c.lo1, P.c.base1, z, P.Hz);
  const int64_t gn = n + op_off(P.c.hi2, P.c.lo2, P.c.base2, z, P.Hz);
  const int64_t off = P.c.g.offset(gm, gn);
  float x = acc * P.epi.alpha;
  if (P.epi.bias) x += static_cast<const float*>(P.epi.bias)[gn];
  if (P.epi.zsave) static_cast<float*>(P.epi.zsave)[off] = x;
  if (P.epi.act == EPI_GELU) x = gelu_f(x);
  else if (P.epi.act == EPI_GELU_BWD) x *= gelu_grad_f(static_cast<const float*>(P.epi.gin)[off]);
  if (P.epi.resid) x += static_cast<const float*>(P.epi.resid)[off];
  static_cast<float*>(const_cast<void*>(P.c.ptr))[off] = x;
}

}  // namespace

tp3d_status gemm_f32_simt(const tp3d_ctx*, const GemmProblem& P, cudaStream_t s) {
  if (P.Z < 1 || P.Hz < 1 || P.M < 1 || P.N < 1 || P.K < 1) return TP3D_EINVAL;
  dim3 grid((unsigned)((P.N + T - 1) / T), (unsigned)((P.M + T - 1) / T), (unsigned)P.Z);
  if (grid.y > 65535u || grid.z > 65535u) return TP3D_EUNSUPPORTED;
  gemm_simt_kernel<<<grid, dim3(T, T), 0, s>>>(P);
  return cudaGetLastError() == cudaSuccess ? TP3D_OK : TP3D_ECUDA;
}

}  // namespace tp3d
