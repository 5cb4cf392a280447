// mlp_noalloc.cu - tp3d_mlp_noalloc: the MLP block for callers that cannot
// allocate device memory.
//
// tp3d_mlp needs an M x f hidden-activation buffer between its two GEMMs and
// asks the caller for it.  Some callers have no way to provide one: code that
// runs where cudaMalloc is forbidden or unsafe (inside a region that must not
// synchronise the device, a runtime that has handed all of HBM to its own
// pool, a plugin that gets only the tensors it reads and writes).  For them
// this entry point keeps the hidden activation in a fixed-size array in
// device memory that belongs to this library (a file-scope __device__
// array, loaded with the library's device code and kept by every GPU that
// uses the library until the process exits).  It calls no cudaMalloc,
// cudaFree or allocating library routine.
//
// The kernels are the same ones tp3d_mlp launches, in the same order; only
// the addresses of the hidden activation and of the chained launch's scratch
// differ.
#include <mutex>

#include "gemm.cuh"

namespace tp3d {
// defined in api.cu
tp3d_status plan_linear(const tp3d_ctx* ctx, int q, int y, int64_t M, int64_t N, int64_t K, const void* A,
                        const void* B, const void* bias, int act, void* C, GemmProblem* out);
}  // namespace tp3d

using namespace tp3d;

namespace {

// Capacity of the static hidden-activation array: 8 Mi bf16 elements (16 MiB),
// i.e. M * f <= 8388608 (the q = 2 MLP with 2048 tokens and ffn 4096 fills it).
constexpr int64_t kMaxHiddenElems = int64_t(8) << 20;

static __device__ __align__(256) __nv_bfloat16 g_mlp_hidden[kMaxHiddenElems];
// The chained launch's counters and fp32 partial sums (M * h <= 8 Mi, 32 MiB);
// zero when the library loads, and every launch leaves the counters zero.
constexpr size_t kChainScratchBytes = (size_t(8) << 20) * sizeof(float) + (size_t(64) << 10);
static __device__ __align__(256) unsigned char g_mlp_chain[kChainScratchBytes];

// Host code may not use g_mlp_hidden's name as an address (it is a host-side
// stand-in); its device address is looked up once per device and cached.
constexpr int kMaxDevices = 64;
void* g_hidden_addr[kMaxDevices] = {};
std::mutex g_hidden_mu;

void* g_chain_addr[kMaxDevices] = {};

tp3d_status hidden_buffer(int device, void** out, void** chain) {
  if (device < 0 || device >= kMaxDevices) return TP3D_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_hidden_mu);
  if (!g_hidden_addr[device]) {
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return TP3D_ECUDA;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return TP3D_ECUDA;
    void *p = nullptr, *c = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_mlp_hidden);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&c, g_mlp_chain);
    if (prev != device) cudaSetDevice(prev);
    if (e != cudaSuccess || p == nullptr || c == nullptr) return TP3D_ECUDA;
    g_hidden_addr[device] = p;
    g_chain_addr[device] = c;
  }
  *out = g_hidden_addr[device];
  *chain = g_chain_addr[device];
  return TP3D_OK;
}

}  // namespace

extern "C" tp3d_status tp3d_mlp_noalloc(tp3d_ctx* ctx, int q, int64_t M, int64_t h, int64_t f, tp3d_dtype dtype,
                                        const void* X, const void* W1, const void* b1, const void* W2,
                                        const void* b2, void* Y, void* stream) {
  if (!ctx || !X || !W1 || !W2 || !Y) return TP3D_EINVAL;
  if (q < 1 || q > 16 || M <= 0 || h <= 0 || f <= 0) return TP3D_EINVAL;
  if (dtype != TP3D_BF16) return TP3D_EDTYPE;
  const void* ptrs[] = {X, W1, b1, W2, b2, Y};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return TP3D_EALIGN;
  if (M > kMaxHiddenElems / f) return TP3D_EUNSUPPORTED;  // M * f beyond the static array
  void *hidden = nullptr, *chain = nullptr;
  TP3D_TRY(hidden_buffer(ctx->device, &hidden, &chain));
  GemmProblem P1, P2;
  TP3D_TRY(plan_linear(ctx, q, 0, M, h, f, X, W1, b1, 1, hidden, &P1));
  TP3D_TRY(plan_linear(ctx, q, 1, M, f, h, hidden, W2, b2, 0, Y, &P2));
  for (const GemmProblem* P : {&P1, &P2})
    if (P->a.g.bw % 8 || P->b.g.bw % 8 || P->c.g.bw % 8) return TP3D_ESHAPE;
  const size_t yb = (size_t)(M * h) * 2;
  const struct { const void* p; size_t n; } ins[] = {{X, (size_t)(M * h) * 2}, {W1, (size_t)(h * f) * 2},
                                                     {b1, (size_t)f * 2}, {W2, (size_t)(f * h) * 2},
                                                     {b2, (size_t)h * 2}};
  for (const auto& in : ins)
    if (overlaps(Y, yb, in.p, in.n)) return TP3D_EOVERLAP;
  const cudaStream_t s = as_stream(stream);
  // the launches tp3d_mlp would make: the chained one on the static scratch
  ChainShape sh;
  if (chain_plan(ctx, P1, P2, &sh)) {
    if (sh.scratch_bytes > kChainScratchBytes) return TP3D_EUNSUPPORTED;
    return gemm_chain_tc(ctx, P1, P2, sh, chain, s);
  }
  TP3D_TRY(gemm_bf16_tc(ctx, P1, s));
  return gemm_bf16_tc(ctx, P2, s);
}
