// api.cu - the extern "C" entry points declared in include/tp3d.h: argument
// validation (all of it before any launch), problem planning, dispatch.
#include <stdlib.h>
#include <string.h>

#include "gemm.cuh"

namespace tp3d {
tp3d_status reshard(const tp3d_ctx* ctx, int64_t R, int64_t C, size_t esz, tp3d_layout sl, const void* src,
                    tp3d_layout dl, void* dst, cudaStream_t stream);

// One 3-D linear (Algorithm 1 + Algorithm 7 of "Maximizing Parallelism in
// Distributed Training for Huge Neural Networks") as a sharded GEMM problem.
tp3d_status plan_linear(const tp3d_ctx* ctx, int q, int y, int64_t M, int64_t N, int64_t K, const void* A,
                        const void* B, const void* bias, int act, void* C, GemmProblem* out) {
  GemmProblem P{};
  Grid ga, gb, gc;
  TP3D_TRY(make_grid(cube(y ? TP3D_CUBE_C : TP3D_CUBE_A, q), M, N, &ga));
  TP3D_TRY(make_grid(cube(y ? TP3D_CUBE_B_SWAP : TP3D_CUBE_B, q), N, K, &gb));
  TP3D_TRY(make_grid(cube(y ? TP3D_CUBE_A : TP3D_CUBE_C, q), M, K, &gc));
  P.Z = 1;
  P.Hz = 1;
  P.M = M;
  P.N = K;
  P.K = N;
  P.a.g = ga;
  P.a.ptr = A;
  P.a.mn_major = 0;  // A stored M x N: contraction contiguous
  P.b.g = gb;
  P.b.ptr = B;
  P.b.mn_major = 1;  // B stored N x K: output columns contiguous
  P.c.g = gc;
  P.c.ptr = C;
  P.epi.act = act ? EPI_GELU : EPI_NONE;
  P.epi.alpha = 1.0f;
  P.epi.bias = bias;
  P.err = ctx->d_err;
  TP3D_TRY(plan_segments(P));
  *out = P;
  return TP3D_OK;
}

// C (M x K) = act(A (M x N) B (N x K) + bias) with each operand in its own
// layout: one GEMM over the layouts' blocks (the contraction runs across the
// shards of A's columns / B's rows).
tp3d_status plan_layouts(const tp3d_ctx* ctx, tp3d_layout la, tp3d_layout lb, tp3d_layout lc, int64_t M, int64_t N,
                         int64_t K, const void* A, const void* B, const void* bias, int act, void* C,
                         GemmProblem* out) {
  GemmProblem P{};
  TP3D_TRY(make_grid(la, M, N, &P.a.g));
  TP3D_TRY(make_grid(lb, N, K, &P.b.g));
  TP3D_TRY(make_grid(lc, M, K, &P.c.g));
  P.Z = 1;
  P.Hz = 1;
  P.M = M;
  P.N = K;
  P.K = N;
  P.a.ptr = A;
  P.a.mn_major = 0;
  P.b.ptr = B;
  P.b.mn_major = 1;
  P.c.ptr = C;
  P.epi.act = act ? EPI_GELU : EPI_NONE;
  P.epi.alpha = 1.0f;
  P.epi.bias = bias;
  P.err = ctx->d_err;
  TP3D_TRY(plan_segments(P));
  *out = P;
  return TP3D_OK;
}

tp3d_status run_gemm(const tp3d_ctx* ctx, tp3d_dtype dt, const GemmProblem& P, cudaStream_t s) {
  return dt == TP3D_BF16 ? gemm_bf16_tc(ctx, P, s) : gemm_f32_simt(ctx, P, s);
}

static size_t esize(tp3d_dtype dt) { return dt == TP3D_BF16 ? 2 : 4; }

static tp3d_layout layout_of(int kind, int a, int b) {
  tp3d_layout l;
  l.kind = kind;
  l.q = 0;
  l.a = a;
  l.b = b;
  return l;
}

// The context's scratch, at least `bytes` long.  Growing it waits for the
// device (an earlier launch may still use the old one) and zeroes the new one.
tp3d_status ctx_scratch(tp3d_ctx* ctx, size_t bytes, void** out) {
  if (ctx->scratch_bytes < bytes) {
    if (ctx->scratch) {
      TP3D_CUDA_TRY(cudaDeviceSynchronize());
      TP3D_CUDA_TRY(cudaFree(ctx->scratch));
      ctx->scratch = nullptr;
      ctx->scratch_bytes = 0;
    }
    void* p = nullptr;
    TP3D_CUDA_TRY(cudaMalloc(&p, bytes));
    if (cudaMemset(p, 0, bytes) != cudaSuccess) {
      cudaFree(p);
      return TP3D_ECUDA;
    }
    ctx->scratch = p;
    ctx->scratch_bytes = bytes;
  }
  *out = ctx->scratch;
  return TP3D_OK;
}

}  // namespace tp3d

using namespace tp3d;

extern "C" {

tp3d_status tp3d_create(int device, tp3d_ctx** out) {
  if (!out) return TP3D_EINVAL;
  *out = nullptr;
  if (cudaSetDevice(device) != cudaSuccess) return TP3D_ECUDA;
  tp3d_ctx* c = static_cast<tp3d_ctx*>(calloc(1, sizeof(tp3d_ctx)));
  if (!c) return TP3D_ECUDA;
  c->device = device;
  c->stall_after = -1;
  int init[kErrWords] = {0, 0, 0, 0};
  const unsigned long long lim = kWaitLimitNs;
  memcpy(init + 2, &lim, sizeof(lim));
  if (cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaMalloc(&c->d_err, sizeof(init)) != cudaSuccess ||
      cudaMemcpy(c->d_err, init, sizeof(init), cudaMemcpyHostToDevice) != cudaSuccess) {
    if (c->d_err) cudaFree(c->d_err);
    free(c);
    return TP3D_ECUDA;
  }
  bool ok = true;
  for (int k = 0; k < 2; ++k) {
    ok = ok && cudaStreamCreateWithFlags(&c->side[k], cudaStreamNonBlocking) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&c->ev_join[k], cudaEventDisableTiming) == cudaSuccess;
  }
  ok = ok && cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaStreamCreateWithFlags(&c->gstream, cudaStreamNonBlocking) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&c->gev_in, cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&c->gev_out, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    tp3d_destroy(c);
    return TP3D_ECUDA;
  }
  *out = c;
  return TP3D_OK;
}

void tp3d_destroy(tp3d_ctx* ctx) {
  if (!ctx) return;
  if (ctx->d_err) cudaFree(ctx->d_err);
  for (int k = 0; k < 2; ++k) {
    if (ctx->side[k]) cudaStreamDestroy(ctx->side[k]);
    if (ctx->ev_join[k]) cudaEventDestroy(ctx->ev_join[k]);
  }
  if (ctx->ev_fork) cudaEventDestroy(ctx->ev_fork);
  if (ctx->gstream) cudaStreamSynchronize(ctx->gstream);  // no graph of this context still running
  graph_cache_free(ctx);
  if (ctx->gstream) cudaStreamDestroy(ctx->gstream);
  if (ctx->gev_in) cudaEventDestroy(ctx->gev_in);
  if (ctx->gev_out) cudaEventDestroy(ctx->gev_out);
  if (ctx->scratch) cudaFree(ctx->scratch);
  free(ctx);
}

const char* tp3d_status_string(tp3d_status s) {
  switch (s) {
    case TP3D_OK: return "ok";
    case TP3D_EINVAL: return "invalid argument";
    case TP3D_ESHAPE: return "shape not divisible as the layout requires";
    case TP3D_EALIGN: return "pointer or row pitch not 16-byte aligned";
    case TP3D_EDTYPE: return "dtype not supported by this call";
    case TP3D_ECUDA: return "CUDA error";
    case TP3D_ETIMEOUT: return "a bounded device-side wait ran out";
    case TP3D_EUNSUPPORTED: return "unsupported configuration";
    case TP3D_EOVERLAP: return "output overlaps an input";
    case TP3D_ERANGE: return "a value on the fp16 score path beyond fp16's range";
  }
  return "unknown status";
}

tp3d_status tp3d_sync_status(tp3d_ctx* ctx, void* stream) {
  if (!ctx) return TP3D_EINVAL;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return TP3D_ECUDA;
  int e = 0;
  if (cudaMemcpy(&e, ctx->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TP3D_ECUDA;
  if (e != 0 && cudaMemset(ctx->d_err, 0, sizeof(int)) != cudaSuccess) return TP3D_ECUDA;
  return static_cast<tp3d_status>(e);
}

tp3d_status tp3d_set_wait_limit_ns(tp3d_ctx* ctx, uint64_t ns) {
  if (!ctx) return TP3D_EINVAL;
  const unsigned long long lim = ns ? (unsigned long long)ns : kWaitLimitNs;
  if (cudaSetDevice(ctx->device) != cudaSuccess ||
      cudaMemcpy(ctx->d_err + 2, &lim, sizeof(lim), cudaMemcpyHostToDevice) != cudaSuccess)
    return TP3D_ECUDA;
  return TP3D_OK;
}

tp3d_status tp3d_inject_load_stall(tp3d_ctx* ctx, int64_t stages) {
  if (!ctx || stages < -1) return TP3D_EINVAL;
  ctx->stall_after = stages;
  return TP3D_OK;
}

tp3d_status tp3d_reshard(tp3d_ctx* ctx, int64_t R, int64_t C, size_t elem_bytes, tp3d_layout src_l, const void* src,
                         tp3d_layout dst_l, void* dst, void* stream) {
  if (!ctx) return TP3D_EINVAL;
  return reshard(ctx, R, C, elem_bytes, src_l, src, dst_l, dst, as_stream(stream));
}

tp3d_status tp3d_linear(tp3d_ctx* ctx, int q, int y, int64_t M, int64_t N, int64_t K, tp3d_dtype dtype,
                        const void* A, const void* B, const void* bias, int act, void* C, void* stream) {
  if (!ctx || !A || !B || !C) return TP3D_EINVAL;
  if (q < 1 || q > 16 || (y != 0 && y != 1) || (act != 0 && act != 1)) return TP3D_EINVAL;
  if (dtype != TP3D_F32 && dtype != TP3D_BF16) return TP3D_EDTYPE;
  if (M <= 0 || N <= 0 || K <= 0) return TP3D_EINVAL;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || (bias && !aligned16(bias))) return TP3D_EALIGN;
  GemmProblem P;
  TP3D_TRY(plan_linear(ctx, q, y, M, N, K, A, B, bias, act, C, &P));
  if (dtype == TP3D_BF16 && (P.a.g.bw % 8 || P.b.g.bw % 8 || P.c.g.bw % 8)) return TP3D_ESHAPE;
  const size_t es = esize(dtype);
  const size_t cb = (size_t)(M * K) * es;
  if (overlaps(C, cb, A, (size_t)(M * N) * es) || overlaps(C, cb, B, (size_t)(N * K) * es) ||
      overlaps(C, cb, bias, (size_t)K * es))
    return TP3D_EOVERLAP;
  return run_gemm(ctx, dtype, P, as_stream(stream));
}

tp3d_status tp3d_mlp(tp3d_ctx* ctx, int q, int64_t M, int64_t h, int64_t f, tp3d_dtype dtype, const void* X,
                     const void* W1, const void* b1, const void* W2, const void* b2, void* Y1, void* Y,
                     void* stream) {
  if (!ctx || !X || !W1 || !W2 || !Y1 || !Y) return TP3D_EINVAL;
  if (q < 1 || q > 16 || M <= 0 || h <= 0 || f <= 0) return TP3D_EINVAL;
  if (dtype != TP3D_BF16) return TP3D_EDTYPE;
  const void* ptrs[] = {X, W1, b1, W2, b2, Y1, Y};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return TP3D_EALIGN;
  GemmProblem P1, P2;
  TP3D_TRY(plan_linear(ctx, q, 0, M, h, f, X, W1, b1, 1, Y1, &P1));
  TP3D_TRY(plan_linear(ctx, q, 1, M, f, h, Y1, W2, b2, 0, Y, &P2));
  for (const GemmProblem* P : {&P1, &P2})
    if (P->a.g.bw % 8 || P->b.g.bw % 8 || P->c.g.bw % 8) return TP3D_ESHAPE;
  const size_t y1b = (size_t)(M * f) * 2, yb = (size_t)(M * h) * 2;
  const struct { const void* p; size_t n; } ins[] = {{X, (size_t)(M * h) * 2}, {W1, (size_t)(h * f) * 2},
                                                     {b1, (size_t)f * 2}, {W2, (size_t)(f * h) * 2},
                                                     {b2, (size_t)h * 2}};
  for (const auto& in : ins)
    if (overlaps(Y1, y1b, in.p, in.n) || overlaps(Y, yb, in.p, in.n)) return TP3D_EOVERLAP;
  if (overlaps(Y, yb, Y1, y1b)) return TP3D_EOVERLAP;
  const cudaStream_t s = as_stream(stream);
  // one chained launch where the block is small enough for it, else the two GEMMs
  ChainShape sh;
  if (chain_plan(ctx, P1, P2, &sh)) {
    void* scratch = nullptr;
    TP3D_TRY(ctx_scratch(ctx, sh.scratch_bytes, &scratch));
    return gemm_chain_tc(ctx, P1, P2, sh, scratch, s);
  }
  TP3D_TRY(gemm_bf16_tc(ctx, P1, s));
  return gemm_bf16_tc(ctx, P2, s);
}

tp3d_status tp3d_mlp_plan(tp3d_ctx* ctx, int q, int64_t M, int64_t h, int64_t f, int* launches, int* splits) {
  if (!ctx || !launches || !splits) return TP3D_EINVAL;
  if (q < 1 || q > 16 || M <= 0 || h <= 0 || f <= 0) return TP3D_EINVAL;
  // planning reads only the layouts: stand-in addresses (Y1's the same in both)
  static const uint8_t x = 0, w1 = 0, w2 = 0, y1 = 0, y = 0;
  GemmProblem P1, P2;
  TP3D_TRY(plan_linear(ctx, q, 0, M, h, f, &x, &w1, nullptr, 1, (void*)&y1, &P1));
  TP3D_TRY(plan_linear(ctx, q, 1, M, f, h, &y1, &w2, nullptr, 0, (void*)&y, &P2));
  for (const GemmProblem* P : {&P1, &P2})
    if (P->a.g.bw % 8 || P->b.g.bw % 8 || P->c.g.bw % 8) return TP3D_ESHAPE;
  ChainShape sh;
  if (chain_plan(ctx, P1, P2, &sh)) {
    *launches = 1;
    *splits = sh.splits;
  } else {
    *launches = 2;
    *splits = 0;
  }
  return TP3D_OK;
}

tp3d_status tp3d_mlp_layout(tp3d_ctx* ctx, int scheme, int p, int64_t M, int64_t h, int64_t f, tp3d_dtype dtype,
                            const void* X, const void* W1, const void* b1, const void* W2, const void* b2, void* Y1,
                            void* Y, void* stream) {
  if (scheme == TP3D_SCHEME_3D) return tp3d_mlp(ctx, p, M, h, f, dtype, X, W1, b1, W2, b2, Y1, Y, stream);
  if (!ctx || !X || !W1 || !W2 || !Y1 || !Y) return TP3D_EINVAL;
  if ((scheme != TP3D_SCHEME_1D && scheme != TP3D_SCHEME_2D) || p < 1 || p > 1024 || M <= 0 || h <= 0 || f <= 0)
    return TP3D_EINVAL;
  if (dtype != TP3D_BF16) return TP3D_EDTYPE;
  const void* ptrs[] = {X, W1, b1, W2, b2, Y1, Y};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return TP3D_EALIGN;
  tp3d_layout lx, lw1, ly1, lw2, ly;
  if (scheme == TP3D_SCHEME_1D) {
    lx = layout_of(TP3D_REPLICATED, 1, 1);
    lw1 = layout_of(TP3D_COL, p, 1);
    ly1 = layout_of(TP3D_COL, p, 1);
    lw2 = layout_of(TP3D_ROW, p, 1);
    ly = layout_of(TP3D_REPLICATED, 1, 1);
  } else {
    lx = lw1 = ly1 = lw2 = ly = layout_of(TP3D_BLOCK2D, p, p);
  }
  GemmProblem P1, P2;
  TP3D_TRY(plan_layouts(ctx, lx, lw1, ly1, M, h, f, X, W1, b1, 1, Y1, &P1));
  TP3D_TRY(plan_layouts(ctx, ly1, lw2, ly, M, f, h, Y1, W2, b2, 0, Y, &P2));
  for (const GemmProblem* P : {&P1, &P2})
    if (P->a.g.bw % 8 || P->b.g.bw % 8 || P->c.g.bw % 8) return TP3D_ESHAPE;
  const size_t y1b = (size_t)(M * f) * 2, yb = (size_t)(M * h) * 2;
  const struct { const void* p; size_t n; } ins[] = {{X, (size_t)(M * h) * 2}, {W1, (size_t)(h * f) * 2},
                                                     {b1, (size_t)f * 2}, {W2, (size_t)(f * h) * 2},
                                                     {b2, (size_t)h * 2}};
  for (const auto& in : ins)
    if (overlaps(Y1, y1b, in.p, in.n) || overlaps(Y, yb, in.p, in.n)) return TP3D_EOVERLAP;
  if (overlaps(Y, yb, Y1, y1b)) return TP3D_EOVERLAP;
  const cudaStream_t s = as_stream(stream);
  TP3D_TRY(gemm_bf16_tc(ctx, P1, s));
  return gemm_bf16_tc(ctx, P2, s);
}

}  // extern "C"
