// attention.cuh - fused causal attention of the GPT layer on the cube
// (attention.cu): forward and backward per (batch, head) window of the QKV
// matrix, on the sm_103a tensor cores, without materialising the score or
// probability matrices.
#pragma once

#include "common.cuh"

namespace tp3d {

struct AttnProblem {
  Grid qkv;          // QKV (M x 3h) layout: Q at columns t*d, K at h + t*d (fp16), V at 2h + t*d (bf16)
  Grid o;            // O / dO (M x h) layout: head t at columns t*d
  int64_t s, h, d, H, Z;  // sequence, hidden, head size, heads, batch * heads
  float scale;       // 1 / sqrt(d)
  int* err;
};

// O = softmax(Q K^T * scale, causal) V per (batch, head); lse[z*s + r] gets
// the row's log-sum-exp of the scaled scores (natural log).
tp3d_status launch_attn_fwd(const tp3d_ctx* ctx, const AttnProblem& A, const void* qkv, void* o, float* lse,
                            cudaStream_t s);

// Backward: given dO, O, lse, writes dQ, dK, dV into dqkv (QKV's layout,
// bf16); `delta` (Z*s floats) is scratch for rowsum(dO * O).  `dmax` (two
// words) bounds the fp16 score gradients: dmax[1] = max |V| over every
// element (bits of a float, written with QKV), dmax[0] is scratch.
tp3d_status launch_attn_bwd(const tp3d_ctx* ctx, const AttnProblem& A, const void* qkv, const void* o,
                            const void* dO, const float* lse, float* delta, unsigned* dmax, void* dqkv,
                            cudaStream_t s);

}  // namespace tp3d
