// The layer core around the recurrence: depthwise causal conv1d + SiLU with
// a rolling history, q/k normalisation and the gates, computed once per
// channel by a streaming prologue kernel that writes exactly the token
// inputs of the state kernel (q, k, v, g, beta).
//
// What it computes, per sequence b and token m ("Kestrel_VLLM - 24 · GDN
// linear attention to GPU", section 3 and figure 1 steps 2-4):
//   conv:  every channel ch of the raw mixed projection x (q channels
//          first, then k, then v) is a width-4 causal convolution over the
//          previous three inputs (the history, oldest first) and the current
//          one, then SiLU; the history stores the inputs and moves by one per
//          token;
//   norm:  q and k scaled by 1 / sqrt(sum of squares + eps) per key head (the
//          article names the step; x / sqrt(|x|^2 + eps) is this library's
//          reading);
//   gates: beta = 1 / (1 + exp(-b)),
//          g = -exp(A_log) softplus(a + dt_bias), softplus(x) = x above 20,
//          exp(x) below -20, log1p(exp(x)) otherwise.
//
// Why a separate kernel.  The state kernel spreads every value head over 16
// warps, and 3 value heads share a key head, so per-key-head work folded into
// it repeats dozens of times (measured: the fused variant took 109-174 us per
// 64 x 48-head decode step against 70 us for the update alone).  Here each
// warp owns one 128-channel row (a key head's q or k, or a value head's v) of
// one token: one coalesced pass over x, the history and the weights, and the
// outputs stay in L2 for the state kernel that follows on the same stream.

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kConvK = 4;
constexpr unsigned kFull = 0xffffffffu;

struct PrologueArgs {
  const float *x, *conv_w, *hist_in;
  float *hist_out;
  const float *a, *b, *A_log, *dt_bias;
  float *q, *k, *v, *g, *beta;
  float eps;
  int B, M, kh, vh, conv_dim;
};

// Row i of the window sequence [hist_in rows, x rows of this launch].
__device__ __forceinline__ const float *seq_row(const PrologueArgs &P, int b,
                                                int i) {
  return i < kConvK - 1
             ? P.hist_in + ((size_t)b * (kConvK - 1) + i) * P.conv_dim
             : P.x + ((size_t)b * P.M + (i - (kConvK - 1))) * P.conv_dim;
}

__device__ __forceinline__ float silu(float x) {
  return __fmul_rn(x, __frcp_rn(__fadd_rn(1.0f, expf(-x))));
}

// One warp per (sequence, token, row); rows 0 .. kh-1 are q heads, kh ..
// 2kh-1 k heads, 2kh .. 2kh+vh-1 v heads, and row 2kh+vh computes the gates
// of every value head.  Lane l owns channels 4l .. 4l+3 of its row.
__global__ void __launch_bounds__(128)
    layer_prologue_kernel(const PrologueArgs P) {
  // behind the kernel before it (which may write x, the history or the
  // state): nothing is read or written before that kernel has ended
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the state kernel that follows may start now: it loads the state (which
  // this kernel never writes, and whose last writer has ended) and waits for
  // these results before reading them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const size_t gw = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int rows = 2 * P.kh + P.vh + 1;
  const size_t total = (size_t)P.B * P.M * rows;
  if (gw >= total) return;
  const int row = (int)(gw % rows);
  const size_t bm = gw / rows;
  const int b = (int)(bm / P.M), m = (int)(bm % P.M);

  if (row == rows - 1) {  // gates
    for (int h = lane; h < P.vh; h += 32) {
      const size_t gi = bm * P.vh + h;
      const float xa = __fadd_rn(__ldg(P.a + gi), __ldg(P.dt_bias + h));
      float sp;
      if (xa > 20.0f)
        sp = xa;
      else if (xa < -20.0f)
        sp = expf(xa);
      else
        sp = log1pf(expf(xa));
      P.g[gi] = __fmul_rn(-expf(__ldg(P.A_log + h)), sp);
      P.beta[gi] = __frcp_rn(__fadd_rn(1.0f, expf(-__ldg(P.b + gi))));
    }
    return;
  }

  const int c = row * kDim + 4 * lane;  // channel of the mixed projection
  const float4 *w4 = reinterpret_cast<const float4 *>(P.conv_w + (size_t)c * kConvK);
  const float4 w[4] = {__ldg(w4), __ldg(w4 + 1), __ldg(w4 + 2), __ldg(w4 + 3)};
  float4 r[kConvK];
#pragma unroll
  for (int j = 0; j < kConvK; ++j)
    r[j] = __ldg(reinterpret_cast<const float4 *>(seq_row(P, b, m + j) + c));
  float y[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float *we = &w[e].x;
    float acc = __fmul_rn(we[0], (&r[0].x)[e]);
#pragma unroll
    for (int j = 1; j < kConvK; ++j) acc = __fmaf_rn(we[j], (&r[j].x)[e], acc);
    y[e] = silu(acc);
  }
  float *dst;
  if (row < 2 * P.kh) {  // q or k: unit L2 norm over the 128 channels
    float ss = __fmul_rn(y[0], y[0]);
    ss = __fmaf_rn(y[1], y[1], ss);
    ss = __fmaf_rn(y[2], y[2], ss);
    ss = __fmaf_rn(y[3], y[3], ss);
#pragma unroll
    for (int off = 16; off; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, off));
    const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(ss, P.eps)));
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = __fmul_rn(y[e], inv);
    const int hh = row < P.kh ? row : row - P.kh;
    dst = (row < P.kh ? P.q : P.k) + (bm * P.kh + hh) * kDim;
  } else {
    dst = P.v + (bm * P.vh + (row - 2 * P.kh)) * kDim;
  }
  *reinterpret_cast<float4 *>(dst + 4 * lane) = make_float4(y[0], y[1], y[2], y[3]);
  if (m == P.M - 1) {  // history after the launch: window taps 1 .. 3
    float *hb = P.hist_out + (size_t)b * (kConvK - 1) * P.conv_dim + c;
#pragma unroll
    for (int j = 1; j < kConvK; ++j)
      *reinterpret_cast<float4 *>(hb + (size_t)(j - 1) * P.conv_dim) = r[j];
  }
}

// Gated RMSNorm on the update's output, one warp per (sequence, token, value
// head) row of 128 channels ("24 · GDN linear attention to GPU", figure 1
// step 6; the article runs it one value head at a time and prints no
// formula):  y = w * o / sqrt(mean(o^2) + eps) * silu(z).  Lane l owns
// channels 4l .. 4l+3; the sum of squares is a fixed xor tree, so every lane
// holds the same bits.  o is read with ordinary loads because y may be o.
// Launched as a programmatic dependent of the previous kernel on the stream,
// it waits for that kernel's results before touching any memory.
__global__ void __launch_bounds__(256)
    gate_norm_kernel(const float *o, const float *__restrict__ z,
                     const float *__restrict__ w, float *y, float eps,
                     size_t rows) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const size_t row = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= rows) return;
  const size_t off = row * kDim + 4 * lane;
  const float4 ov = *reinterpret_cast<const float4 *>(o + off);
  const float4 zv = __ldg(reinterpret_cast<const float4 *>(z + off));
  const float4 wv = __ldg(reinterpret_cast<const float4 *>(w + 4 * lane));
  float ss = __fmul_rn(ov.x, ov.x);
  ss = __fmaf_rn(ov.y, ov.y, ss);
  ss = __fmaf_rn(ov.z, ov.z, ss);
  ss = __fmaf_rn(ov.w, ov.w, ss);
#pragma unroll
  for (int d = 16; d; d >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, d));
  // mean over the 128 channels: the scale by 2^-7 is exact
  const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(ss, 0.0078125f), eps)));
  const float *oe = &ov.x, *ze = &zv.x, *we = &wv.x;
  float out[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    out[e] = __fmul_rn(__fmul_rn(__fmul_rn(oe[e], r), we[e]), silu(ze[e]));
  *reinterpret_cast<float4 *>(y + off) = make_float4(out[0], out[1], out[2], out[3]);
}

// History after m_dev[b] tokens of a launch = rows m .. m+2 of
// [hist_snap rows, x rows], as a flat copy over every 16-byte element of
// the B x 3 x conv_dim history: each thread has kRollUnroll loads in flight
// before its stores.  Replayed from a CUDA graph it took 4.06 us a call for
// 64 sequences and 2.67 us for 8, against 5.13 and 4.88 us for one CTA per
// sequence with a load-store loop.  A count outside 0..M leaves that
// sequence's history untouched and raises the error flag.
constexpr int kRollUnroll = 4;
__global__ void hist_rollback_kernel(float4 *__restrict__ hist,
                                     const float *__restrict__ hist_snap,
                                     const float *__restrict__ x,
                                     const int *__restrict__ m_dev,
                                     int *__restrict__ err, int M,
                                     int conv_dim, size_t total4) {
  const size_t n4 = (size_t)conv_dim / 4;
  const size_t per_seq = (kConvK - 1) * n4;
  const size_t base = (size_t)blockIdx.x * blockDim.x * kRollUnroll + threadIdx.x;
  float4 r[kRollUnroll];
  bool take[kRollUnroll];
#pragma unroll
  for (int u = 0; u < kRollUnroll; ++u) {
    const size_t e = base + (size_t)u * blockDim.x;
    take[u] = false;
    if (e >= total4) continue;
    const size_t b = e / per_seq;
    const size_t rem = e - b * per_seq;
    const int j = (int)(rem / n4);
    const size_t c = rem - (size_t)j * n4;
    const int m = __ldg(m_dev + b);
    if (m < 0 || m > M) {
      if (err) *err = 1;
      continue;
    }
    const int i = m + j;
    const float *src = i < kConvK - 1
                           ? hist_snap + (b * (kConvK - 1) + i) * (size_t)conv_dim
                           : x + (b * M + (i - (kConvK - 1))) * (size_t)conv_dim;
    r[u] = __ldg(reinterpret_cast<const float4 *>(src) + c);
    take[u] = true;
  }
#pragma unroll
  for (int u = 0; u < kRollUnroll; ++u)
    if (take[u]) hist[base + (size_t)u * blockDim.x] = r[u];
}

}  // namespace

cudaError_t launch_layer_prologue(const float *hist_in, float *hist_out,
                                  const float *x, const float *conv_w,
                                  const float *a, const float *b,
                                  const float *A_log, const float *dt_bias,
                                  float eps, float *q, float *k, float *v,
                                  float *g, float *beta, int B, int kh, int vh,
                                  int M, cudaStream_t stream, bool overlap) {
  PrologueArgs P;
  P.x = x;
  P.conv_w = conv_w;
  P.hist_in = hist_in;
  P.hist_out = hist_out;
  P.a = a;
  P.b = b;
  P.A_log = A_log;
  P.dt_bias = dt_bias;
  P.q = q;
  P.k = k;
  P.v = v;
  P.g = g;
  P.beta = beta;
  P.eps = eps;
  P.B = B;
  P.M = M;
  P.kh = kh;
  P.vh = vh;
  P.conv_dim = 2 * kh * kDim + vh * kDim;
  const size_t warps = (size_t)B * M * (2 * kh + vh + 1);
  if (warps == 0) return cudaSuccess;
  const size_t blocks = (warps + 3) / 4;
  if (blocks > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, layer_prologue_kernel, P);
}

cudaError_t launch_gate_norm(const float *o, const float *z, const float *w,
                             float *y, float eps, size_t rows,
                             cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const size_t blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gate_norm_kernel, o, z, w, y, eps, rows);
}

cudaError_t launch_hist_rollback(float *hist, const float *hist_snap,
                                 const float *x, const int *m_dev, int *err_dev,
                                 int B, int M, int conv_dim,
                                 cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const size_t total4 = (size_t)B * (kConvK - 1) * (size_t)(conv_dim / 4);
  const size_t blocks = (total4 + 256 * kRollUnroll - 1) / (256 * kRollUnroll);
  if (blocks > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  hist_rollback_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      reinterpret_cast<float4 *>(hist), hist_snap, x, m_dev, err_dev, M,
      conv_dim, total4);
  return cudaGetLastError();
}

}  // namespace gdn
