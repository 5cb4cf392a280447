// graph.cu - CUDA graphs of whole calls, cached per context.
//
// A layer call enqueues about thirty launches, each with tensor maps to
// encode and launch attributes to set on the host.  Called again with the
// same arguments, that host work repeats unchanged; when it takes longer
// than the GPU's previous work, the GPU idles between launches.  So the
// first call with a given argument set records its launches into a CUDA
// graph (stream capture), and later calls with the same arguments launch
// that graph.  The argument set is the call's own bytes (configuration,
// parameter pointers, workspace, stream, the context's test hook), compared
// exactly; the graph reads every buffer at run time, so new contents in the
// same buffers need no new graph.
//
// The graph runs on a stream of the context, ordered after the caller's
// stream by an event and the caller's stream after it by another, so the call
// keeps the semantics of enqueuing on the caller's stream (including the
// legacy default stream, which cannot be captured).  A call made while the
// caller's stream is itself being captured enqueues directly into that
// capture.
#include <string.h>

#include <vector>

#include "common.cuh"

namespace tp3d {

namespace {

struct GraphEntry {
  std::vector<unsigned char> key;
  cudaGraphExec_t exec;
  uint64_t used;
};
struct GraphCache {
  std::vector<GraphEntry> entries;
  uint64_t tick = 0;
};
constexpr size_t kMaxGraphs = 8;

}  // namespace

tp3d_status graph_call(tp3d_ctx* ctx, const void* key, size_t key_bytes, cudaStream_t st,
                       tp3d_status (*enqueue)(void* arg, cudaStream_t s), void* arg) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return TP3D_ECUDA;
  if (cs != cudaStreamCaptureStatusNone || !ctx->gstream) return enqueue(arg, st);
  if (!ctx->graphs) ctx->graphs = new GraphCache();
  GraphCache* gc = static_cast<GraphCache*>(ctx->graphs);
  const unsigned char* k = static_cast<const unsigned char*>(key);
  GraphEntry* hit = nullptr;
  for (GraphEntry& e : gc->entries)
    if (e.key.size() == key_bytes && memcmp(e.key.data(), k, key_bytes) == 0) hit = &e;
  if (!hit) {
    // record the call's launches on the context's stream
    TP3D_CUDA_TRY(cudaStreamBeginCapture(ctx->gstream, cudaStreamCaptureModeRelaxed));
    const tp3d_status s = enqueue(arg, ctx->gstream);
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(ctx->gstream, &g);
    if (s != TP3D_OK || e != cudaSuccess || !g) {
      if (g) cudaGraphDestroy(g);
      (void)cudaGetLastError();
      return s != TP3D_OK ? s : TP3D_ECUDA;
    }
    cudaGraphExec_t ex = nullptr;
    const cudaError_t ie = cudaGraphInstantiate(&ex, g, 0);
    cudaGraphDestroy(g);
    if (ie != cudaSuccess) return TP3D_ECUDA;
    if (gc->entries.size() >= kMaxGraphs) {  // drop the least recently used
      size_t lru = 0;
      for (size_t i = 1; i < gc->entries.size(); ++i)
        if (gc->entries[i].used < gc->entries[lru].used) lru = i;
      cudaGraphExecDestroy(gc->entries[lru].exec);
      gc->entries.erase(gc->entries.begin() + (long)lru);
    }
    gc->entries.push_back(GraphEntry{std::vector<unsigned char>(k, k + key_bytes), ex, 0});
    hit = &gc->entries.back();
  }
  hit->used = ++gc->tick;
  TP3D_CUDA_TRY(cudaEventRecord(ctx->gev_in, st));
  TP3D_CUDA_TRY(cudaStreamWaitEvent(ctx->gstream, ctx->gev_in, 0));
  TP3D_CUDA_TRY(cudaGraphLaunch(hit->exec, ctx->gstream));
  TP3D_CUDA_TRY(cudaEventRecord(ctx->gev_out, ctx->gstream));
  TP3D_CUDA_TRY(cudaStreamWaitEvent(st, ctx->gev_out, 0));
  return TP3D_OK;
}

void graph_cache_free(tp3d_ctx* ctx) {
  if (!ctx->graphs) return;
  GraphCache* gc = static_cast<GraphCache*>(ctx->graphs);
  for (GraphEntry& e : gc->entries) cudaGraphExecDestroy(e.exec);
  delete gc;
  ctx->graphs = nullptr;
}

}  // namespace tp3d
