// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

constexpr int kDim = 128;  // kd == vd: the only head size the kernels serve

// Launch modes of launch_steps.
//   kOverlapNone: an ordinary launch.
//   kOverlapPrologue: a programmatic dependent of the previous kernel on the
//     stream, which must not write S_in (the kernel starts loading the
//     state before it waits for that kernel): the layer prologue.
//   kOverlapAny: a programmatic dependent of whatever kernel came before;
//     the kernel reads nothing before that kernel has ended, so it only
//     takes over the launch and the start of its CTAs.  Applied to grids
//     that fill every CTA slot; smaller grids launch ordinarily.
constexpr int kOverlapNone = 0, kOverlapPrologue = 1, kOverlapAny = 2;
// Launches of more tokens than this start ordinarily: a long launch gains
// nothing from an earlier start, and its CTAs would wait on SM slots beside
// the previous launch's last CTAs.
constexpr int kOverlapMaxTokens = 16;

// Token-serial update of every head over M tokens (gdn_step, gdn_step_m and
// the fp32 prefill path).  Pointers and layouts as in gdn.h; S_out may equal
// S_in.  ckpt may be nullptr.  overlap: one of the modes above.
// host_inputs: some token input is in mapped host memory (single-token
// launches then use larger CTAs, whose warps share the inputs in L1).
cudaError_t launch_steps(const float *S_in, float *S_out, float *ckpt,
                         const float *q, const float *k, const float *v,
                         const float *g, const float *beta, float *o, int B,
                         int kh, int vh, int M, cudaStream_t stream,
                         int overlap = kOverlapNone, bool host_inputs = false);

// Layer prologue (conv1d + SiLU with a width-4 history, q/k normalisation,
// gates) writing the token inputs q, k, v, g, beta of M tokens.  hist_in and
// hist_out must not overlap.  overlap: launch as a programmatic dependent of
// the kernel before it; the prologue reads and writes nothing before that
// kernel has ended, and only then lets its own dependents start.
cudaError_t launch_layer_prologue(const float *hist_in, float *hist_out,
                                  const float *x, const float *conv_w,
                                  const float *a, const float *b,
                                  const float *A_log, const float *dt_bias,
                                  float eps, float *q, float *k, float *v,
                                  float *g, float *beta, int B, int kh, int vh,
                                  int M, cudaStream_t stream,
                                  bool overlap = false);

// Gated RMSNorm of `rows` rows of 128 channels (see gdn_gated_rmsnorm_m);
// y may equal o.
cudaError_t launch_gate_norm(const float *o, const float *z, const float *w,
                             float *y, float eps, size_t rows,
                             cudaStream_t stream);

// Per-sequence conv-history rollback (see gdn_layer_hist_rollback).
cudaError_t launch_hist_rollback(float *hist, const float *hist_snap,
                                 const float *x, const int *m_dev, int *err_dev,
                                 int B, int M, int conv_dim,
                                 cudaStream_t stream);

// dst[i] = src[i] for n floats (n % 4 == 0, both 16-byte aligned).
cudaError_t launch_copy(float *dst, const float *src, size_t n,
                        cudaStream_t stream);

// Per-sequence rollback copy (see gdn_rollback_seq).
cudaError_t launch_rollback_seq(float *S, const float *snap, const float *ckpt,
                                const int *m_dev, int *err_dev, int B, int vh,
                                int M, cudaStream_t stream);

// Chunked tensor-core prefill (defined in gdn_prefill.cu).
size_t prefill_workspace_bytes(int B, int kh, int vh, int T, int chunk,
                               int precision);
// precision: 1 = split-bf16 (three products), 2 = bf16 (one product).
cudaError_t launch_prefill_chunked(float *S, const float *q, const float *k,
                                   const float *v, const float *g,
                                   const float *beta, float *o, int B, int kh,
                                   int vh, int T, int precision,
                                   void *workspace, cudaStream_t stream);
cudaError_t prefill_timeouts(unsigned int *count);
// Ring waits of the multi-token kernel that ran out (gdn_decode.cu).
cudaError_t steps_timeouts(unsigned int *count);

}  // namespace gdn

struct gdn_shape;

namespace gdn {

// The checks gdn_layer_step_m makes of every argument except its workspace
// (a gdn.h status; GDN_OK also for B == 0).  Defined in gdn_api.cu.
int layer_step_check(const gdn_shape *s, int M, int ck, float eps,
                     const float *S_in, float *S_out, float *ckpt,
                     const float *hist_in, float *hist_out, const float *x,
                     const float *conv_w, const float *a, const float *b,
                     const float *A_log, const float *dt_bias, float *o);

}  // namespace gdn
