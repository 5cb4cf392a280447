// layer_kernels.cuh - host launchers of the layer's bandwidth-bound kernels
// (layer_kernels.cu): LayerNorm forward/backward and column sums.  All read and write matrices through
// their layout grid, so a row that the cube splits over q shards is read from
// those q shards.
#pragma once

#include "common.cuh"

namespace tp3d {

// y = (x - mean) * rstd * gamma + beta per row of the R x C matrix x (layout g,
// y in the same layout); mean / rstd (fp32, R each) are saved.  y16, if not
// null, receives the same values in fp16 (a value beyond fp16's range raises
// TP3D_ERANGE in the context's error word).
tp3d_status launch_ln_fwd(const tp3d_ctx* ctx, const Grid& g, const void* x, const void* gamma, const void* beta,
                          void* y, void* y16, float* mean, float* rstd, float eps, cudaStream_t s);

// y = fp16(x 2^k) for n bf16 values (n a multiple of 8), 2^k the power of two
// that puts max |x| in [2^14, 2^15); *inv_scale = 2^-k (device float).  `amax`
// is one device word of scratch.  Two launches and a 4-byte memset on s.
tp3d_status launch_to_f16_scaled(const tp3d_ctx* ctx, const void* x, int64_t n, unsigned* amax, void* y,
                                 float* inv_scale, cudaStream_t s);

// dx = dres + rstd * (dxh - mean(dxh) - xh * mean(dxh * xh)), dxh = dy * gamma,
// xh = (x - mean) * rstd, per row (dy, x, dres, dx in layout g).
tp3d_status launch_ln_bwd(const tp3d_ctx* ctx, const Grid& g, const void* dy, const void* x, const float* mean,
                          const float* rstd, const void* gamma, const void* dres, void* dx, cudaStream_t s);

// LayerNorm parameter gradients: out_g = column sums of dy * (x - mean) *
// rstd, out_b = column sums of dy (bf16, C each).  Scratch: `part` holds
// 2 * colsum_parts(g) rows of C floats; `counters` (colsum_strips(g) ints,
// zero on entry) is zero again on exit.
tp3d_status launch_ln_param_grads(const tp3d_ctx* ctx, const Grid& g, const void* dy, const void* x,
                                  const float* mean, const float* rstd, float* part, int* counters, void* out_g,
                                  void* out_b, cudaStream_t s);

// Column sums of the R x C bf16 matrix x (layout g) into the bf16 vector
// `out`, in one launch: partial rows in `part` (colsum_parts(g) rows of C
// floats), reduced by the last CTA of each 256-column strip; `counters`
// (colsum_strips(g) ints, zero on entry) is zero again on exit.
int64_t colsum_parts(const Grid& g);
int64_t colsum_strips(const Grid& g);
tp3d_status launch_colsum(const tp3d_ctx* ctx, const Grid& g, const void* x, float* part, int* counters, void* out,
                          cudaStream_t s);

}  // namespace tp3d
