// layer.cu - the pre-LN GPT decoder layer on the cube, forward and backward
// ("Maximizing Parallelism in Distributed Training for Huge Neural
// Networks", §3.2): a Self-Attention block and an MLP block, each two 3-D
// linears - the first with input group y = 0 (input CUBE_A, output CUBE_C),
// the second with y and z exchanged (input CUBE_C, output CUBE_A) - so the
// layer's output has its input's layout.  LayerNorm is the matrix-vector
// scaling and shift of §3.1.3 with whole-row statistics.  Backward follows
// the differentiation formulas of §3.1.2 (dA = dC B^T, dB = A^T dC; the
// attention products are the C = A B^T and C = A^T B forms), Algorithm 8
// read by its definition (bias gradient = column sums over every row) and
// §3.1.3's gamma gradient sum(dC * A-hat).
//
// The scores' inputs are carried in fp16 (11 significant bits against bf16's
// 8): the softmax backward magnifies their rounding by about the scores'
// magnitude, which for sharply peaked attention takes bf16 storage of the LN1
// output and of Q and K past 1e-2 of the exact layer.  So LN1 also writes an
// fp16 copy of its output, W_qkv is converted to fp16 scaled by a power of
// two (undone in the QKV product's epilogue), and that product stores Q and K
// in fp16, V in bf16; the attention kernels take it from there.
//
// The forward launches LayerNorm, the four linear GEMMs (QKV, output
// projection + residual, W1 + GELU, W2 + residual) and the fused causal
// attention forward; the backward its eight linear GEMMs, the fused attention
// backward, LayerNorm backward and the column sums of the bias / gamma / beta
// gradients.  They run on the caller's stream, except independent work that
// is forked onto the context's two side streams and joined back before the
// call returns (the forward's W_qkv conversion; the backward's weight
// gradients and column sums).  Attention reads each (batch, head) window in
// place from the CUBE_C shards of the QKV matrix (attention.cu).
#include <math.h>
#include <string.h>

#include <algorithm>

#include "attention.cuh"
#include "gemm.cuh"
#include "layer_kernels.cuh"

namespace tp3d {

tp3d_status plan_linear(const tp3d_ctx* ctx, int q, int y, int64_t M, int64_t N, int64_t K, const void* A,
                        const void* B, const void* bias, int act, void* C, GemmProblem* out);

namespace {

using bf16 = __nv_bfloat16;

struct Plan {
  int q, b, s, h, H, d, f;
  int64_t M, Z;
  float eps;
  // workspace offsets (bytes)
  size_t xn1, mean1, rstd1, qkv, lse, O, Hres, xn2, mean2, rstd2, z1, y1;  // saved by the forward
  size_t xn1h, wqkvh, misc;  // fp16 score-path operands; misc: max |W_qkv|, 1/scale, max |dO_r|^2, max |V|
  size_t delta, dz1, dxn, dH, dO, dqkv, part, counters;                    // scratch
  size_t part_floats, part_db1, part_dbqkv, total;  // float offsets of db1's and dbqkv's partials
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr int64_t kCounters = 2048;  // column-sum arrival counters in the workspace
constexpr int64_t kStripSlot = 256;  // counters of one column sum (slots 0..4)

tp3d_status make_plan(const tp3d_layer_cfg* c, Plan* p) {
  if (!c) return TP3D_EINVAL;
  if (c->q < 1 || c->q > 16 || c->batch < 1 || c->seq < 1 || c->hidden < 1 || c->heads < 1 || c->ffn < 1)
    return TP3D_EINVAL;
  if (c->dtype != TP3D_BF16) return TP3D_EDTYPE;
  if (!(c->eps > 0.0f)) return TP3D_EINVAL;
  Plan x{};
  x.q = c->q;
  x.b = c->batch;
  x.s = c->seq;
  x.h = c->hidden;
  x.H = c->heads;
  x.f = c->ffn;
  x.eps = c->eps;
  if (x.h % x.H) return TP3D_ESHAPE;
  x.d = x.h / x.H;
  x.M = (int64_t)x.b * x.s;
  x.Z = (int64_t)x.b * x.H;
  const int64_t q2 = (int64_t)x.q * x.q;
  if (x.M % q2 || x.h % q2 || x.f % q2 || (3 * (int64_t)x.h) % q2) return TP3D_ESHAPE;
  // every shard row a whole number of 16-byte vectors, heads and query tiles
  // inside shards (the causal tiles of the attention products are 128 rows)
  const int64_t m = x.M / q2;
  if ((x.h / q2) % 8 || (x.f / q2) % 8) return TP3D_ESHAPE;
  if ((x.d != 64 && x.d != 128) || x.s % 128 || m % 128 || ((x.h / x.q) % x.d)) return TP3D_EUNSUPPORTED;
  const int64_t M = x.M, h = x.h, f = x.f, Z = x.Z, s = x.s;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  x.xn1 = take(M * h * 2);
  x.mean1 = take(M * 4);
  x.rstd1 = take(M * 4);
  x.qkv = take(M * 3 * h * 2);
  x.lse = take(Z * s * 4);
  x.O = take(M * h * 2);
  x.Hres = take(M * h * 2);
  x.xn2 = take(M * h * 2);
  x.mean2 = take(M * 4);
  x.rstd2 = take(M * 4);
  x.z1 = take(M * f * 2);
  x.y1 = take(M * f * 2);
  x.xn1h = take(M * h * 2);
  x.wqkvh = take(3 * h * h * 2);
  x.misc = take(256);
  x.delta = take(Z * s * 4);
  x.dz1 = take(M * f * 2);
  x.dxn = take(M * h * 2);
  x.dH = take(M * h * 2);
  x.dO = take(M * h * 2);
  x.dqkv = take(M * 3 * h * 2);
  // column-sum partials: a region for each sum that may run beside another
  // (the gamma/beta sums [2 sets], dbo, db2, db1, dbqkv)
  Grid gc, ga, gq;
  TP3D_TRY(make_grid(cube(TP3D_CUBE_C, x.q), M, f, &gc));
  TP3D_TRY(make_grid(cube(TP3D_CUBE_A, x.q), M, h, &ga));
  TP3D_TRY(make_grid(cube(TP3D_CUBE_C, x.q), M, 3 * h, &gq));
  x.part_db1 = (size_t)(4 * colsum_parts(ga) * h);
  x.part_dbqkv = x.part_db1 + (size_t)(colsum_parts(gc) * f);
  x.part_floats = x.part_dbqkv + (size_t)(colsum_parts(gq) * 3 * h);
  x.part = take(x.part_floats * 4);
  // arrival counters: one per 256-column strip, kStripSlot apart for the sums that run together
  if ((f > 3 * h ? f : 3 * h) / 256 + 1 > kStripSlot) return TP3D_EUNSUPPORTED;
  x.counters = take(kCounters * 4);
  x.total = o;
  *p = x;
  return TP3D_OK;
}

// The attention windows: head t of sequence b reads rows [b*s, +s) of QKV at
// columns t*d (Q), h + t*d (K), 2h + t*d (V) and writes O at columns t*d.
AttnProblem attn_problem(const Plan& p, int* err) {
  AttnProblem A{};
  make_grid(cube(TP3D_CUBE_C, p.q), p.M, 3 * (int64_t)p.h, &A.qkv);
  make_grid(cube(TP3D_CUBE_C, p.q), p.M, p.h, &A.o);
  A.s = p.s;
  A.h = p.h;
  A.d = p.d;
  A.H = p.H;
  A.Z = p.Z;
  A.scale = 1.0f / sqrtf((float)p.d);
  A.err = err;
  return A;
}

tp3d_status run(const tp3d_ctx* ctx, GemmProblem& P, cudaStream_t s) {
  TP3D_TRY(plan_segments(P));
  return gemm_bf16_tc(ctx, P, s);
}

// dA = dC . W^T for a 3-D linear with input group y (MP3D Algorithm 2, first line)
tp3d_status plan_dgrad(const tp3d_ctx* ctx, int q, int y, int64_t M, int64_t Nin, int64_t Kout, const void* dC,
                       const void* W, void* dA, GemmProblem* out) {
  GemmProblem P{};
  TP3D_TRY(make_grid(cube(y ? TP3D_CUBE_A : TP3D_CUBE_C, q), M, Kout, &P.a.g));
  TP3D_TRY(make_grid(cube(y ? TP3D_CUBE_B_SWAP : TP3D_CUBE_B, q), Nin, Kout, &P.b.g));
  TP3D_TRY(make_grid(cube(y ? TP3D_CUBE_C : TP3D_CUBE_A, q), M, Nin, &P.c.g));
  P.Z = 1;
  P.Hz = 1;
  P.M = M;
  P.N = Nin;
  P.K = Kout;
  P.a.ptr = dC;
  P.a.mn_major = 0;
  P.b.ptr = W;  // stored Nin x Kout = n x k: K-major
  P.b.mn_major = 0;
  P.c.ptr = dA;
  P.epi.alpha = 1.0f;
  P.err = ctx->d_err;
  *out = P;
  return TP3D_OK;
}

// dW = A^T . dC for a 3-D linear with input group y (MP3D Algorithm 2, second line)
tp3d_status plan_wgrad(const tp3d_ctx* ctx, int q, int y, int64_t M, int64_t Nin, int64_t Kout, const void* A,
                       const void* dC, void* dW, GemmProblem* out) {
  GemmProblem P{};
  TP3D_TRY(make_grid(cube(y ? TP3D_CUBE_C : TP3D_CUBE_A, q), M, Nin, &P.a.g));
  TP3D_TRY(make_grid(cube(y ? TP3D_CUBE_A : TP3D_CUBE_C, q), M, Kout, &P.b.g));
  TP3D_TRY(make_grid(cube(y ? TP3D_CUBE_B_SWAP : TP3D_CUBE_B, q), Nin, Kout, &P.c.g));
  P.Z = 1;
  P.Hz = 1;
  P.M = Nin;
  P.N = Kout;
  P.K = M;
  P.a.ptr = A;  // stored M x Nin = k x m: MN-major
  P.a.mn_major = 1;
  P.b.ptr = dC;  // stored M x Kout = k x n: MN-major
  P.b.mn_major = 1;
  P.c.ptr = dW;
  P.epi.alpha = 1.0f;
  P.err = ctx->d_err;
  *out = P;
  return TP3D_OK;
}

tp3d_status colsum(const tp3d_ctx* ctx, int kind, int q, int64_t R, int64_t C, const void* x, float* part,
                   int* counters, void* out, cudaStream_t s) {
  Grid g;
  TP3D_TRY(make_grid(cube(kind, q), R, C, &g));
  return launch_colsum(ctx, g, x, part, counters, out, s);
}

}  // namespace

}  // namespace tp3d

using namespace tp3d;

extern "C" {

size_t tp3d_layer_workspace_bytes(const tp3d_layer_cfg* cfg) {
  Plan p;
  if (make_plan(cfg, &p) != TP3D_OK) return 0;
  return p.total;
}

static tp3d_status layer_fwd_enqueue(tp3d_ctx* ctx, const tp3d_layer_cfg* cfg, const tp3d_layer_params* w,
                                     const void* X, void* Y, void* workspace, cudaStream_t stream) {
  if (!ctx || !cfg || !w || !X || !Y || !workspace) return TP3D_EINVAL;
  Plan p;
  TP3D_TRY(make_plan(cfg, &p));
  const void* need[] = {w->ln1_g, w->ln1_b, w->w_qkv, w->b_qkv, w->w_o, w->b_o,
                        w->ln2_g, w->ln2_b, w->w_1, w->b_1, w->w_2, w->b_2};
  for (const void* ptr : need)
    if (!ptr) return TP3D_EINVAL;
  for (const void* ptr : need)
    if (!aligned16(ptr)) return TP3D_EALIGN;
  if (!aligned16(X) || !aligned16(Y) || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return TP3D_EALIGN;
  const int64_t M = p.M, h = p.h, f = p.f;
  if (overlaps(Y, M * h * 2, X, M * h * 2) || overlaps(workspace, p.total, X, M * h * 2) ||
      overlaps(workspace, p.total, Y, M * h * 2))
    return TP3D_EOVERLAP;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto W = [&](size_t off) { return static_cast<void*>(ws + off); };
  const cudaStream_t st = stream;
  const int q = p.q;

  Grid gA;
  TP3D_TRY(make_grid(cube(TP3D_CUBE_A, q), M, h, &gA));
  // The score path in fp16: W_qkv scaled by a power of two 2^k, the LN1
  // output in bf16 (for the weight gradient) and fp16, Q and K in fp16.  The
  // conversion of W_qkv runs on side stream 0 beside LN1 and is joined before
  // the QKV product.
  unsigned* misc = (unsigned*)W(p.misc);
  float* inv_scale = (float*)(misc + 1);
  TP3D_CUDA_TRY(cudaEventRecord(ctx->ev_fork, st));
  TP3D_CUDA_TRY(cudaStreamWaitEvent(ctx->side[0], ctx->ev_fork, 0));
  TP3D_TRY(launch_to_f16_scaled(ctx, w->w_qkv, 3 * h * h, misc, W(p.wqkvh), inv_scale, ctx->side[0]));
  TP3D_CUDA_TRY(cudaEventRecord(ctx->ev_join[0], ctx->side[0]));
  // LN1
  TP3D_TRY(launch_ln_fwd(ctx, gA, X, w->ln1_g, w->ln1_b, W(p.xn1), W(p.xn1h), (float*)W(p.mean1),
                         (float*)W(p.rstd1), p.eps, st));
  TP3D_CUDA_TRY(cudaStreamWaitEvent(st, ctx->ev_join[0], 0));
  // QKV = LN1(X) W_qkv + b_qkv   (y = 0: CUBE_A -> CUBE_C): fp16 product, 2^-k applied
  // in the epilogue, Q and K (columns below 2h) stored in fp16, V in bf16
  GemmProblem G;
  TP3D_TRY(plan_linear(ctx, q, 0, M, h, 3 * h, W(p.xn1h), W(p.wqkvh), w->b_qkv, 0, W(p.qkv), &G));
  G.in_f16 = 1;
  G.epi.alpha_dev = inv_scale;
  G.epi.f16_cols = 2 * h;
  G.epi.amax_out = misc + 3;  // max |V|, for the backward's bound on the score gradients
  TP3D_CUDA_TRY(cudaMemsetAsync(misc + 3, 0, sizeof(unsigned), st));
  TP3D_TRY(gemm_bf16_tc(ctx, G, st));
  // causal attention per (batch, head), fused: O = softmax(Q K^T / sqrt(d)) V
  TP3D_TRY(launch_attn_fwd(ctx, attn_problem(p, ctx->d_err), W(p.qkv), W(p.O), (float*)W(p.lse), st));
  // H = X + O W_o + b_o   (y = 1: CUBE_C -> CUBE_A)
  TP3D_TRY(plan_linear(ctx, q, 1, M, h, h, W(p.O), w->w_o, w->b_o, 0, W(p.Hres), &G));
  G.epi.resid = X;
  TP3D_TRY(gemm_bf16_tc(ctx, G, st));
  // LN2, then Y1 = GELU(Z1), Z1 = LN2(H) W_1 + b_1 saved
  TP3D_TRY(launch_ln_fwd(ctx, gA, W(p.Hres), w->ln2_g, w->ln2_b, W(p.xn2), nullptr, (float*)W(p.mean2),
                         (float*)W(p.rstd2), p.eps, st));
  TP3D_TRY(plan_linear(ctx, q, 0, M, h, f, W(p.xn2), w->w_1, w->b_1, 1, W(p.y1), &G));
  G.epi.zsave = W(p.z1);
  TP3D_TRY(gemm_bf16_tc(ctx, G, st));
  // Y = H + Y1 W_2 + b_2
  TP3D_TRY(plan_linear(ctx, q, 1, M, f, h, W(p.y1), w->w_2, w->b_2, 0, Y, &G));
  G.epi.resid = W(p.Hres);
  return gemm_bf16_tc(ctx, G, st);
}

static tp3d_status layer_bwd_enqueue(tp3d_ctx* ctx, const tp3d_layer_cfg* cfg, const tp3d_layer_params* w,
                                     const void* X, void* workspace, const void* dY, void* dX,
                                     const tp3d_layer_grads* g, cudaStream_t stream) {
  if (!ctx || !cfg || !w || !g || !X || !dY || !dX || !workspace) return TP3D_EINVAL;
  Plan p;
  TP3D_TRY(make_plan(cfg, &p));
  const void* need[] = {w->ln1_g, w->ln1_b, w->w_qkv, w->b_qkv, w->w_o, w->b_o, w->ln2_g, w->ln2_b, w->w_1,
                        w->b_1, w->w_2, w->b_2, g->ln1_g, g->ln1_b, g->w_qkv, g->b_qkv, g->w_o, g->b_o,
                        g->ln2_g, g->ln2_b, g->w_1, g->b_1, g->w_2, g->b_2};
  for (const void* ptr : need)
    if (!ptr) return TP3D_EINVAL;
  for (const void* ptr : need)
    if (!aligned16(ptr)) return TP3D_EALIGN;
  if (!aligned16(X) || !aligned16(dY) || !aligned16(dX) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return TP3D_EALIGN;
  const int64_t M = p.M, h = p.h, f = p.f;
  if (overlaps(dX, M * h * 2, dY, M * h * 2) || overlaps(dX, M * h * 2, X, M * h * 2) ||
      overlaps(workspace, p.total, dX, M * h * 2) || overlaps(workspace, p.total, dY, M * h * 2))
    return TP3D_EOVERLAP;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto W = [&](size_t off) { return static_cast<void*>(ws + off); };
  float* part = (float*)W(p.part);
  int* counters = (int*)W(p.counters);
  const cudaStream_t st = stream;
  // the column sums' arrival counters start at zero (each sum leaves them so)
  TP3D_CUDA_TRY(cudaMemsetAsync(counters, 0, kCounters * 4, st));
  const int q = p.q;
  GemmProblem G;
  Grid gA;
  TP3D_TRY(make_grid(cube(TP3D_CUBE_A, q), M, h, &gA));

  // Column sums that nothing later reads run beside the main stream, two or
  // three at once (each with its own partials and counters): their launch and
  // reduction tails overlap.  The main stream waits for them before its next
  // launch that could overwrite what they read, and before returning.
  auto fork = [&](int n) -> tp3d_status {  // side streams 0..n-1 start after everything on st so far
    TP3D_CUDA_TRY(cudaEventRecord(ctx->ev_fork, st));
    for (int k = 0; k < n; ++k) TP3D_CUDA_TRY(cudaStreamWaitEvent(ctx->side[k], ctx->ev_fork, 0));
    return TP3D_OK;
  };
  auto fork_to = [&](int k) -> tp3d_status {  // side stream k alone
    TP3D_CUDA_TRY(cudaEventRecord(ctx->ev_fork, st));
    TP3D_CUDA_TRY(cudaStreamWaitEvent(ctx->side[k], ctx->ev_fork, 0));
    return TP3D_OK;
  };
  auto join = [&](int n) -> tp3d_status {
    for (int k = 0; k < n; ++k) {
      TP3D_CUDA_TRY(cudaEventRecord(ctx->ev_join[k], ctx->side[k]));
      TP3D_CUDA_TRY(cudaStreamWaitEvent(st, ctx->ev_join[k], 0));
    }
    return TP3D_OK;
  };
  const int64_t pa = colsum_parts(gA) * h;  // floats of one M x h partial set

  // The weight gradients (nothing in the call reads them) go to side stream 1,
  // beside the chain of data gradients on the main stream.

  // ---- MLP block
  TP3D_TRY(fork_to(1));
  TP3D_TRY(plan_wgrad(ctx, q, 1, M, f, h, W(p.y1), dY, g->w_2, &G));                       // dW2 = Y1^T dY
  TP3D_TRY(run(ctx, G, ctx->side[1]));
  TP3D_TRY(plan_dgrad(ctx, q, 1, M, f, h, dY, w->w_2, W(p.dz1), &G));                      // dZ1 = (dY W2^T) GELU'(Z1)
  G.epi.act = EPI_GELU_BWD;
  G.epi.gin = W(p.z1);
  TP3D_TRY(run(ctx, G, st));
  // db1 on side stream 0 (its own partials and counters), dW1 on side stream 1
  TP3D_TRY(fork(2));
  TP3D_TRY(colsum(ctx, TP3D_CUBE_C, q, M, f, W(p.dz1), part + p.part_db1,
                  counters + 3 * kStripSlot, g->b_1, ctx->side[0]));                                      // db1
  TP3D_TRY(plan_wgrad(ctx, q, 0, M, h, f, W(p.xn2), W(p.dz1), g->w_1, &G));                // dW1 = LN2(H)^T dZ1
  TP3D_TRY(run(ctx, G, ctx->side[1]));
  TP3D_TRY(plan_dgrad(ctx, q, 0, M, h, f, W(p.dz1), w->w_1, W(p.dxn), &G));                // dLN2 = dZ1 W1^T
  TP3D_TRY(run(ctx, G, st));
  TP3D_TRY(launch_ln_bwd(ctx, gA, W(p.dxn), W(p.Hres), (const float*)W(p.mean2), (const float*)W(p.rstd2),
                         w->ln2_g, dY, W(p.dH), st));                                                  // dH
  // dbo, then dgamma2 and dbeta2 on side stream 0 (dLN2 in dxn is overwritten
  // by dLN1: joined before then); db2, then dWo on side stream 1
  TP3D_TRY(fork(2));
  TP3D_TRY(colsum(ctx, TP3D_CUBE_A, q, M, h, W(p.dH), part + 2 * pa, counters + kStripSlot, g->b_o,
                  ctx->side[0]));                                                                        // dbo
  TP3D_TRY(launch_ln_param_grads(ctx, gA, W(p.dxn), W(p.Hres), (const float*)W(p.mean2), (const float*)W(p.rstd2),
                                 part, counters, g->ln2_g, g->ln2_b, ctx->side[0]));
  TP3D_TRY(colsum(ctx, TP3D_CUBE_A, q, M, h, dY, part + 3 * pa, counters + 2 * kStripSlot, g->b_2,
                  ctx->side[1]));                                                                        // db2

  // ---- attention block
  TP3D_TRY(plan_wgrad(ctx, q, 1, M, h, h, W(p.O), W(p.dH), g->w_o, &G));                   // dWo = O^T dH
  TP3D_TRY(run(ctx, G, ctx->side[1]));
  TP3D_TRY(plan_dgrad(ctx, q, 1, M, h, h, W(p.dH), w->w_o, W(p.dO), &G));                  // dO = dH Wo^T
  TP3D_TRY(run(ctx, G, st));
  // attention backward, fused: dQ, dK, dV into dQKV (MP3D's C = A B^T and C = A^T B forms)
  TP3D_TRY(launch_attn_bwd(ctx, attn_problem(p, ctx->d_err), W(p.qkv), W(p.O), W(p.dO), (const float*)W(p.lse),
                           (float*)W(p.delta), (unsigned*)W(p.misc) + 2, W(p.dqkv), st));
  // dWqkv, then dbqkv on side stream 1
  TP3D_TRY(fork_to(1));
  TP3D_TRY(plan_wgrad(ctx, q, 0, M, h, 3 * h, W(p.xn1), W(p.dqkv), g->w_qkv, &G));         // dWqkv = LN1(X)^T dQKV
  TP3D_TRY(run(ctx, G, ctx->side[1]));
  TP3D_TRY(colsum(ctx, TP3D_CUBE_C, q, M, 3 * h, W(p.dqkv), part + p.part_dbqkv, counters + 4 * kStripSlot,
                  g->b_qkv, ctx->side[1]));                                                              // dbqkv
  // dgamma2 and dbeta2 have read dLN2 before dLN1 takes its place
  TP3D_CUDA_TRY(cudaEventRecord(ctx->ev_join[0], ctx->side[0]));
  TP3D_CUDA_TRY(cudaStreamWaitEvent(st, ctx->ev_join[0], 0));
  TP3D_TRY(plan_dgrad(ctx, q, 0, M, h, 3 * h, W(p.dqkv), w->w_qkv, W(p.dxn), &G));         // dLN1 = dQKV Wqkv^T
  TP3D_TRY(run(ctx, G, st));
  // dgamma1, dbeta1 on side stream 0 beside the LN1 backward (both only read dLN1)
  TP3D_TRY(fork_to(0));
  TP3D_TRY(launch_ln_param_grads(ctx, gA, W(p.dxn), X, (const float*)W(p.mean1), (const float*)W(p.rstd1), part,
                                 counters, g->ln1_g, g->ln1_b, ctx->side[0]));
  TP3D_TRY(launch_ln_bwd(ctx, gA, W(p.dxn), X, (const float*)W(p.mean1), (const float*)W(p.rstd1), w->ln1_g,
                         W(p.dH), dX, st));                                                            // dX
  return join(2);  // every side stream joined before returning
}

// The public calls: argument checks, then the launches above as a cached CUDA
// graph keyed by every argument (graph.cu; a stream under capture gets the
// launches directly).
struct FwdCall {
  tp3d_ctx* ctx;
  const tp3d_layer_cfg* cfg;
  const tp3d_layer_params* w;
  const void* X;
  void *Y, *workspace;
};
static tp3d_status fwd_thunk(void* a, cudaStream_t s) {
  const FwdCall* c = static_cast<const FwdCall*>(a);
  return layer_fwd_enqueue(c->ctx, c->cfg, c->w, c->X, c->Y, c->workspace, s);
}
struct BwdCall {
  tp3d_ctx* ctx;
  const tp3d_layer_cfg* cfg;
  const tp3d_layer_params* w;
  const void* X;
  void* workspace;
  const void* dY;
  void* dX;
  const tp3d_layer_grads* g;
};
static tp3d_status bwd_thunk(void* a, cudaStream_t s) {
  const BwdCall* c = static_cast<const BwdCall*>(a);
  return layer_bwd_enqueue(c->ctx, c->cfg, c->w, c->X, c->workspace, c->dY, c->dX, c->g, s);
}
struct CallKey {
  int32_t fn;
  tp3d_layer_cfg cfg;
  tp3d_layer_params w;
  tp3d_layer_grads g;
  const void *X, *dY;
  void *Y, *dX, *workspace, *stream;
  int64_t stall_after;
};

tp3d_status tp3d_layer_fwd(tp3d_ctx* ctx, const tp3d_layer_cfg* cfg, const tp3d_layer_params* w, const void* X,
                           void* Y, void* workspace, void* stream) {
  if (!ctx || !cfg || !w || !X || !Y || !workspace) return TP3D_EINVAL;
  Plan p;
  TP3D_TRY(make_plan(cfg, &p));
  CallKey k;
  memset(&k, 0, sizeof(k));
  k.fn = 1;
  k.cfg = *cfg;
  k.w = *w;
  k.X = X;
  k.Y = Y;
  k.workspace = workspace;
  k.stream = stream;
  k.stall_after = ctx->stall_after;
  FwdCall c{ctx, cfg, w, X, Y, workspace};
  return graph_call(ctx, &k, sizeof(k), as_stream(stream), fwd_thunk, &c);
}

tp3d_status tp3d_layer_bwd(tp3d_ctx* ctx, const tp3d_layer_cfg* cfg, const tp3d_layer_params* w, const void* X,
                           void* workspace, const void* dY, void* dX, const tp3d_layer_grads* g, void* stream) {
  if (!ctx || !cfg || !w || !g || !X || !dY || !dX || !workspace) return TP3D_EINVAL;
  Plan p;
  TP3D_TRY(make_plan(cfg, &p));
  CallKey k;
  memset(&k, 0, sizeof(k));
  k.fn = 2;
  k.cfg = *cfg;
  k.w = *w;
  k.g = *g;
  k.X = X;
  k.dY = dY;
  k.dX = dX;
  k.workspace = workspace;
  k.stream = stream;
  k.stall_after = ctx->stall_after;
  BwdCall c{ctx, cfg, w, X, workspace, dY, dX, g};
  return graph_call(ctx, &k, sizeof(k), as_stream(stream), bwd_thunk, &c);
}

}  // extern "C"
