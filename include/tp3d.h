/*
 * tp3d.h - C ABI of the 3-D tensor-parallel layer cube on one GB300.
 *
 * The method is the load-balanced 3-D parallel matrix multiplication and the
 * 3-D parallel Transformer layer of "Maximizing Parallelism in Distributed
 * Training for Huge Neural Networks" (Bian, Xu, Wang, You; arXiv 2105.14450),
 * written MP3D below, plus the layout conversion ("resharding") between the
 * sharding specs of "On Optimizing the Communication of Model Parallelism"
 * (arXiv 2211.05322) §2, written CMR below.  Every virtual device (i, j, l)
 * of the q x q x q cube is a shard in one GPU's memory; the all-gathers are
 * reads at shard offsets, the depth reduce-scatter is accumulation across
 * l inside one kernel, the bias broadcast is an epilogue read.
 *
 * Storage.  A sharded matrix is ONE caller-owned device buffer that holds
 * every virtual device's shard back to back, in device order
 * d = (i*q + j)*q + l (cube layouts) or mesh order (other layouts); each
 * shard is dense and row-major.  A replicated layout holds every copy.  A
 * vector (bias, LayerNorm gamma/beta) is the plain contiguous vector: the
 * diagonal layout of MP3D §3.1.1 (b_ji on devices j = l) concatenated in
 * (j, i) order is exactly that.
 *
 * Ownership.  The caller allocates every tensor and workspace (PyTorch in the
 * bundled binding).  The library allocates only its context: one device
 * error word, two side streams with three events, and host-side caches.  All
 * compute calls are asynchronous on the given CUDA stream (a cudaStream_t
 * passed as void*; NULL = the legacy default stream).  A call that runs
 * independent launches on the context's side streams (tp3d_layer_fwd,
 * tp3d_layer_bwd) forks them from the given stream and joins them back into
 * it before returning,
 * so its work is ordered on the given stream as a whole; calls of one context
 * must not run concurrently on different streams.  Inputs are read-only;
 * outputs must not alias inputs.
 *
 * Errors.  Arguments are validated on the host before anything is launched;
 * a failed check returns its status and launches nothing.  There are no
 * exceptions, aborts or prints.  A failed launch returns TP3D_ECUDA.  Kernel
 * waits are bounded (tp3d_set_wait_limit_ns): a wait that runs out sets the
 * context's device error word, the kernel returns, and tp3d_sync_status()
 * reports TP3D_ETIMEOUT.
 */
#ifndef TP3D_H
#define TP3D_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TP3D_OK = 0,
  TP3D_EINVAL = 1,       /* null pointer, bad enum, bad q, negative size          */
  TP3D_ESHAPE = 2,       /* a size not divisible as the layout requires          */
  TP3D_EALIGN = 3,       /* pointer not 16-byte aligned / row pitch not 16 bytes  */
  TP3D_EDTYPE = 4,       /* dtype not supported by this call                      */
  TP3D_ECUDA = 5,        /* a CUDA runtime or driver call failed                  */
  TP3D_ETIMEOUT = 6,     /* a bounded device-side wait ran out                    */
  TP3D_EUNSUPPORTED = 7, /* valid request outside what the kernels implement      */
  TP3D_EOVERLAP = 8,     /* output buffer overlaps an input buffer               */
  TP3D_ERANGE = 9        /* a value on the layer's fp16 score path (LN1 output,
                            Q, K) beyond fp16's finite range; raised by a kernel
                            and reported by tp3d_sync_status                     */
} tp3d_status;

typedef enum { TP3D_F32 = 0, TP3D_BF16 = 1 } tp3d_dtype;

/* Layout kinds.  For an R x C matrix on a q-cube (m = R/q^2 etc. as in
 * MP3D §3.1.1), device (i, j, l) holds:
 *   CUBE_A       rows [i*R/q + j*R/q^2, +R/q^2), cols [l*C/q, +C/q)     (A_ijl)
 *   CUBE_B       rows [l*R/q, +R/q), cols [j*C/q + i*C/q^2, +C/q^2)      (B_lji)
 *   CUBE_C       rows [i*R/q + l*R/q^2, +R/q^2), cols [j*C/q, +C/q)      (C_ilj)
 *   CUBE_B_SWAP  CUBE_B with directions y and z exchanged:
 *                rows [j*R/q, +R/q), cols [l*C/q + i*C/q^2, +C/q^2)      (B_jli)
 * Mesh layouts (CMR §2 sharding specs), shard number = mesh device number:
 *   ROW      a-way row split (S^01 R), shard s = rows [s*R/a, +R/a)
 *   COL      a-way column split (R S^01)
 *   BLOCK2D  a x b mesh, S^0 S^1: shard r*b + c = rows block r, cols block c
 *   REPLICATED a full copies (R R)
 * A dense unsharded matrix is ROW with a = 1.                               */
typedef enum {
  TP3D_CUBE_A = 0,
  TP3D_CUBE_B = 1,
  TP3D_CUBE_C = 2,
  TP3D_CUBE_B_SWAP = 3,
  TP3D_ROW = 4,
  TP3D_COL = 5,
  TP3D_BLOCK2D = 6,
  TP3D_REPLICATED = 7
} tp3d_layout_kind;

/* kind; q for CUBE_*; a for ROW/COL/REPLICATED (shards or copies);
 * a x b mesh for BLOCK2D.  Unused fields are ignored.                        */
typedef struct {
  int32_t kind;
  int32_t q;
  int32_t a;
  int32_t b;
} tp3d_layout;

typedef struct tp3d_ctx tp3d_ctx;

/* Creates a context on CUDA device `device` (made current).  Owns one device
 * error word.  Returns TP3D_EINVAL for a null `out`, TP3D_ECUDA if the device
 * cannot be used.                                                            */
tp3d_status tp3d_create(int device, tp3d_ctx** out);
void tp3d_destroy(tp3d_ctx* ctx);
const char* tp3d_status_string(tp3d_status s);

/* Synchronises `stream`, then reads and clears the device error word:
 * TP3D_ETIMEOUT if a bounded wait ran out since the last call, TP3D_ERANGE
 * if a layer call met a value its fp16 score path cannot hold, TP3D_ECUDA if
 * the stream reported an error, else TP3D_OK.                               */
tp3d_status tp3d_sync_status(tp3d_ctx* ctx, void* stream);

/* Failure detection (no counterpart on the pages; the bounded waits are this
 * library's own).  Every wait inside a kernel gives up after the context's
 * wait limit, 4 s unless set here; a wait that runs out sets TP3D_ETIMEOUT in
 * the device error word, the kernel's CTAs let everything they issued land
 * (loads, products, stores), free their tensor memory and return, and the
 * context stays usable.  `ns` = 0 restores 4 s.  The limit lives in device
 * memory and is written synchronously: it applies to kernels launched after
 * the call returns; do not call it while this context's work is in flight
 * or during stream capture.  TP3D_ECUDA if the write fails.                 */
tp3d_status tp3d_set_wait_limit_ns(tp3d_ctx* ctx, uint64_t ns);

/* Test hook for the timeout path: from now on, the GEMM kernels of this
 * context's calls stop loading operands after `stages` contraction stages of
 * each launch (after letting the loads they issued land), so the tensor-core
 * issuer's next wait can only run out (-1 turns the hook off; the default).
 * Host-side state only; TP3D_EINVAL for stages < -1.                         */
tp3d_status tp3d_inject_load_stall(tp3d_ctx* ctx, int64_t stages);

/* Resharding (CMR §2, cross-mesh resharding; MP3D §3.1.1 cube layouts):
 * writes into `dst` (layout dst_l) the same R x C matrix that `src` holds in
 * layout src_l.  Every destination element receives the bits of the same
 * global element; elements are moved as raw `elem_bytes`-byte words
 * (1, 2, 4 or 8), so the copy is bit-exact for any dtype.  A replicated
 * source is read from copy 0; a replicated destination gets every copy.
 * TP3D_ESHAPE if R or C do not divide as either layout requires;
 * TP3D_EOVERLAP if the two buffers overlap.                                  */
tp3d_status tp3d_reshard(tp3d_ctx* ctx, int64_t R, int64_t C, size_t elem_bytes,
                         tp3d_layout src_l, const void* src,
                         tp3d_layout dst_l, void* dst, void* stream);

/* 3-D linear, MP3D Algorithm 1 (+ Algorithm 7 for the bias): C = A.B (+ b),
 * then GELU if act == 1 (exact erf form).  A is M x N, B is N x K, C is
 * M x K (N is the contraction).  Input group index y (MP3D §3.2):
 *   y = 0: A in CUBE_A, B in CUBE_B, C in CUBE_C;
 *   y = 1: directions exchanged: A in CUBE_C, B in CUBE_B_SWAP, C in CUBE_A.
 * The depth reduce-scatter (sum over l, ascending) happens in fp32 inside the
 * kernel; each device's rows of C_ij are written once.  bias: K-vector of
 * `dtype`, or NULL.  dtype TP3D_BF16 runs the tcgen05 tensor-core kernel
 * (bf16 in, fp32 accumulate, bf16 out); TP3D_F32 runs fp32 FFMA (no TF32).
 * TP3D_ESHAPE unless M % q^2 == 0, N % q == 0, K % q^2 == 0 (and, for bf16,
 * every shard's row length a multiple of 8 elements).                        */
tp3d_status tp3d_linear(tp3d_ctx* ctx, int q, int y, int64_t M, int64_t N, int64_t K,
                        tp3d_dtype dtype, const void* A, const void* B, const void* bias,
                        int act, void* C, void* stream);

/* MLP block on the cube (MP3D §3.2; the column-split GEMM + GELU followed by
 * the row-split GEMM with summed partials of "Transformer Training 11: Model
 * Parallelism", "Tensor parallelism"):
 *   Y1 = GELU(X.W1 + b1)   (3-D linear with y = 0: X CUBE_A, W1 CUBE_B, Y1 CUBE_C)
 *   Y  = Y1.W2 + b2        (3-D linear with y = 1: W2 CUBE_B_SWAP, Y CUBE_A)
 * X: M x h, W1: h x f, W2: f x h, b1: f, b2: h (either bias may be NULL).
 * Y1 (M x f, CUBE_C) is caller-owned scratch that also returns the hidden
 * activation.  bf16 only.
 *
 * A block whose operands (X, W1, Y1, W2) total at most 64 MiB runs as ONE
 * persistent launch (the row tiles of the first GEMM feed the second's
 * contraction as soon as they are stored; the second GEMM's contraction may
 * be cut in two halves whose fp32 partial sums are added in a fixed order);
 * a larger block runs as two GEMM launches.  tp3d_mlp_plan says which.  The
 * one launch uses a device scratch owned by the context (counters and, with
 * two halves, M x h fp32 partial sums): the first call that needs it, or
 * more of it, allocates it (cudaMalloc, after a cudaDeviceSynchronize if it
 * replaces a smaller one), so make that call before any stream capture, and
 * order the context's tp3d_mlp calls on one stream (they share the scratch).
 * The launch's clusters wait on each other's progress with bounded waits; a
 * wait that runs out (only possible if the device cannot keep its clusters
 * resident, e.g. beside another such launch) raises TP3D_ETIMEOUT.          */
tp3d_status tp3d_mlp(tp3d_ctx* ctx, int q, int64_t M, int64_t h, int64_t f, tp3d_dtype dtype,
                     const void* X, const void* W1, const void* b1, const void* W2,
                     const void* b2, void* Y1, void* Y, void* stream);

/* How tp3d_mlp (and tp3d_mlp_noalloc) run a bf16 block of these sizes on
 * this context's device: *launches = 1 for the one chained launch, with
 * *splits = 1 or 2 (the second GEMM's contraction halves), or 2 for two GEMM
 * launches (*splits = 0).  Launches nothing; errors as tp3d_mlp's shape
 * checks.                                                                    */
tp3d_status tp3d_mlp_plan(tp3d_ctx* ctx, int q, int64_t M, int64_t h, int64_t f, int* launches, int* splits);

/* The same MLP block in the layouts the pages compare the cube with
 * ("Maximizing Parallelism in Distributed Training for Huge Neural
 * Networks" §2 and §4: Megatron's 1-D and Optimus' 2-D SUMMA partitioning),
 * computed on this GPU by the same tensor-core GEMM.
 *   TP3D_SCHEME_1D, p = t devices (Megatron): X (M x h) replicated; W1
 *     COL(t) (each device f/t columns), b1 split the same way, Y1 COL(t);
 *     W2 ROW(t); Y replicated.  The all-reduce of the row-split GEMM is its
 *     contraction across the t shards.  A replicated matrix is stored once
 *     (every virtual device reads that copy).
 *   TP3D_SCHEME_2D, p = q, a q x q mesh (SUMMA): X, W1, Y1, W2, Y in
 *     BLOCK2D(q, q) (block (r, c) = device r*q + c); C_rc = sum_k A_rk B_kc.
 *   TP3D_SCHEME_3D, p = q: the cube, exactly tp3d_mlp.
 * Biases are plain vectors (either may be NULL).  bf16 only.  TP3D_ESHAPE
 * when a dimension is not divisible by the scheme's block counts or a block's
 * row is not a multiple of 8 elements; other errors as tp3d_mlp.             */
typedef enum { TP3D_SCHEME_1D = 1, TP3D_SCHEME_2D = 2, TP3D_SCHEME_3D = 3 } tp3d_scheme;
tp3d_status tp3d_mlp_layout(tp3d_ctx* ctx, int scheme, int p, int64_t M, int64_t h, int64_t f, tp3d_dtype dtype,
                            const void* X, const void* W1, const void* b1, const void* W2, const void* b2, void* Y1,
                            void* Y, void* stream);

/* tp3d_mlp without the hidden-activation argument, for callers that cannot
 * allocate device memory: code that must not call cudaMalloc (it would
 * synchronise the device, or the process's memory is all handed to another
 * pool), or that is given only the tensors it reads and writes.  The paper
 * has no counterpart; this is a convenience of this library.
 *
 * Same computation, kernels and order as tp3d_mlp.  The hidden activation
 * Y1 lives in a fixed array of 8 Mi bf16 elements (16 MiB) in this
 * library's device memory, which every GPU that loads the library keeps
 * until the process exits; M * f must be <= 8388608, else TP3D_EUNSUPPORTED
 * and nothing is launched.  The chained launch's scratch is a second fixed
 * array (32 MiB: M * h <= 8388608 when that launch cuts the contraction in
 * two, else TP3D_EUNSUPPORTED).  The call allocates nothing.
 *   - The first call on a device looks up the array's device address (one
 *     cudaGetSymbolAddress with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - Every call, on every stream, shares the arrays, which keep the last
 *     call's contents; calls that overlap on the GPU race.  Y1 is fully
 *     written before it is read, so nothing needs clearing between calls.
 * Other arguments, layouts and errors as tp3d_mlp.                           */
tp3d_status tp3d_mlp_noalloc(tp3d_ctx* ctx, int q, int64_t M, int64_t h, int64_t f, tp3d_dtype dtype,
                             const void* X, const void* W1, const void* b1, const void* W2,
                             const void* b2, void* Y, void* stream);

/* GPT decoder layer (MP3D §3.2), pre-LN:
 *   H = X + Attn(LN1(X)),  Y = H + MLP(LN2(H))
 * LN: biased variance, eps; attention: causal, `heads` heads of
 * d = hidden/heads, QKV columns packed [Q | K | V], head t at columns
 * t*d .. t*d+d-1 of each; GELU exact.  Token row = batch*seq + position.
 * Layouts: X, Y, dX, dY in CUBE_A (M x hidden, M = batch*seq); W_qkv
 * (hidden x 3 hidden) and W_1 (hidden x ffn) in CUBE_B; W_o (hidden x hidden)
 * and W_2 (ffn x hidden) in CUBE_B_SWAP; vectors plain.  Parameters,
 * activations and gradients are bf16; LN and softmax statistics fp32.
 *
 * Score path in fp16.  The softmax backward amplifies a relative error u of
 * the scores' inputs by about the scores' own magnitude, so with sharply
 * peaked attention (|scores| of 5 and more) bf16's u = 2^-9 on the LN1
 * output and on Q and K alone puts dQ, dK and everything upstream of them
 * beyond 1e-2 of the exact layer.  The layer therefore keeps the inputs of
 * the scores in fp16 (u = 2^-11): the LN1 output feeding the QKV product,
 * a copy of W_qkv scaled by a power of two (2^k |w|max in [2^14, 2^15),
 * undone in the product's epilogue), Q and K, and the score gradients dS
 * (scaled by a power of two from a bound on max_r |dO_r| max |V|, undone in
 * the dQ and dK epilogues).  V, P, O and every gradient stay bf16.  A value
 * of the LN1 output or of Q or K beyond 65504 in magnitude raises
 * TP3D_ERANGE (read with tp3d_sync_status); magnitudes below fp16's normal
 * range (2^-14) keep an absolute precision of 2^-25 there.                   */
typedef struct {
  int32_t q, batch, seq, hidden, heads, ffn;
  int32_t dtype; /* tp3d_dtype; TP3D_BF16 only */
  float eps;
} tp3d_layer_cfg;

typedef struct {
  const void *ln1_g, *ln1_b, *w_qkv, *b_qkv, *w_o, *b_o;
  const void *ln2_g, *ln2_b, *w_1, *b_1, *w_2, *b_2;
} tp3d_layer_params;

typedef struct {
  void *ln1_g, *ln1_b, *w_qkv, *b_qkv, *w_o, *b_o;
  void *ln2_g, *ln2_b, *w_1, *b_1, *w_2, *b_2;
} tp3d_layer_grads;

/* Bytes of the caller-owned workspace that tp3d_layer_fwd fills with the
 * activations the backward needs, plus the backward's own scratch.  Returns 0
 * for an invalid configuration.                                              */
size_t tp3d_layer_workspace_bytes(const tp3d_layer_cfg* cfg);

/* Forward.  `workspace` (>= tp3d_layer_workspace_bytes, 256-byte aligned)
 * receives the saved activations.  TP3D_EUNSUPPORTED unless seq % 128 == 0,
 * d == 64 or 128, and every shard dimension a multiple of 64.                */
tp3d_status tp3d_layer_fwd(tp3d_ctx* ctx, const tp3d_layer_cfg* cfg, const tp3d_layer_params* p,
                           const void* X, void* Y, void* workspace, void* stream);

/* Backward: given X, the workspace filled by tp3d_layer_fwd with the same
 * parameters, and dY, writes dX and every parameter gradient (each in its
 * parameter's layout and dtype).  The workspace's scratch part is
 * overwritten; its saved part is preserved.                                  */
tp3d_status tp3d_layer_bwd(tp3d_ctx* ctx, const tp3d_layer_cfg* cfg, const tp3d_layer_params* p,
                           const void* X, void* workspace, const void* dY, void* dX,
                           const tp3d_layer_grads* g, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TP3D_H */
