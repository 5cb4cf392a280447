// layer.cu - the GPT decoder layer on the cube (forward and backward).
#include "gemm.cuh"

using namespace tp3d;

extern "C" {

size_t tp3d_layer_workspace_bytes(const tp3d_layer_cfg* cfg) {
  (void)cfg;
  return 0;
}

tp3d_status tp3d_layer_fwd(tp3d_ctx* ctx, const tp3d_layer_cfg* cfg, const tp3d_layer_params* p, const void* X,
                           void* Y, void* workspace, void* stream) {
  (void)ctx; (void)cfg; (void)p; (void)X; (void)Y; (void)workspace; (void)stream;
  return TP3D_EUNSUPPORTED;
}

tp3d_status tp3d_layer_bwd(tp3d_ctx* ctx, const tp3d_layer_cfg* cfg, const tp3d_layer_params* p, const void* X,
                           void* workspace, const void* dY, void* dX, const tp3d_layer_grads* g, void* stream) {
  (void)ctx; (void)cfg; (void)p; (void)X; (void)workspace; (void)dY; (void)dX; (void)g; (void)stream;
  return TP3D_EUNSUPPORTED;
}

}  // extern "C"
