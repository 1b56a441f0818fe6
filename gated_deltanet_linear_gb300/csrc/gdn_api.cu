// C ABI of libgdn_gb300.so: argument validation on the host, then one
// asynchronous launch on the caller's stream.  Declarations and the contract
// of every entry point are in include/gdn.h.
//
// Conventions follow the articles' device library: device pointers plus a
// stream, no implicit synchronisation ("24 · GDN linear attention to GPU",
// section 11, the device-pointer layer step), an int status where a
// refusal is an error code rather than a silent fallback (same article,
// section 8; "34 · batched M rows", section 3.5), and no truncation of a
// request that does not fit (article 24, section 10).

#include <stdint.h>
#include <string.h>

#include "gdn.h"
#include "gdn_internal.cuh"

namespace {

struct Buf {
  const void *p;
  size_t bytes;
};

bool overlaps(const Buf &a, const Buf &b) {
  if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
  const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
  return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// The caller's current device, or -1 (the CUDA error is cleared).
int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return dev;
}

// One attribute query per pointer.  Device memory of `dev` and managed
// memory pass.  Token inputs and outputs (allow_host) may also live in
// page-locked host memory that is mapped into the device's address space at
// the same address (any cudaHostAlloc / cudaMallocHost block under unified
// addressing): kernels then read and write it over the host link, and *host
// is set.  Pageable memory is refused.
int classify_ptr(const void *p, int dev, bool allow_host, bool *host) {
  cudaPointerAttributes attr;
  memset(&attr, 0, sizeof(attr));
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return GDN_EPTR;
  }
  if (attr.type == cudaMemoryTypeManaged) return GDN_OK;
  if (attr.type == cudaMemoryTypeHost) {
    if (!allow_host || attr.devicePointer != p) return GDN_EPTR;
    if (host) *host = true;
    return GDN_OK;
  }
  if (attr.type != cudaMemoryTypeDevice) return GDN_EPTR;
  return attr.device == dev ? GDN_OK : GDN_EPTR;
}

// Device (or managed) memory of the current device.
int check_device_ptr(const void *p) {
  const int dev = current_device();
  if (dev < 0) return GDN_ECUDA;
  return classify_ptr(p, dev, false, nullptr);
}

int check_shape(const gdn_shape *s) {
  if (!s) return GDN_EINVAL;
  if (s->B < 0 || s->kh <= 0 || s->vh <= 0) return GDN_ESHAPE;
  if (s->kd != gdn::kDim || s->vd != gdn::kDim) return GDN_ESHAPE;
  if (s->vh % s->kh) return GDN_ESHAPE;
  return GDN_OK;
}

// Every buffer: non-null, 16-byte aligned, device memory (or, for token
// inputs and outputs, allow_host: mapped page-locked host memory; *any_host
// is then set if one is).  A pointer already checked in the same list is
// not queried again.
int check_list(const Buf *b, int n, bool allow_host, bool *any_host) {
  for (int i = 0; i < n; ++i) {
    if (!b[i].p) return GDN_EINVAL;
    if (!aligned16(b[i].p)) return GDN_EALIGN;
  }
  const int dev = current_device();
  if (dev < 0) return GDN_ECUDA;
  for (int i = 0; i < n; ++i) {
    bool seen = false;
    for (int j = 0; j < i && !seen; ++j) seen = b[j].p == b[i].p;
    if (seen) continue;
    const int r = classify_ptr(b[i].p, dev, allow_host, any_host);
    if (r != GDN_OK) return r;
  }
  return GDN_OK;
}

int check_bufs(const Buf *b, int n) { return check_list(b, n, false, nullptr); }

int check_io_bufs(const Buf *b, int n, bool *any_host = nullptr) {
  return check_list(b, n, true, any_host);
}

int status_of(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ECUDA; }

size_t state_floats(const gdn_shape *s) {
  return (size_t)s->B * s->vh * s->kd * s->vd;
}

// Validate and launch M serial tokens (shared by gdn_step, gdn_step_m and
// the fp32 prefill path).
// *host_inputs (if given) is set when a token input is host memory.
int steps_common_check(const gdn_shape *s, int M, const float *S_in,
                       float *S_out, float *ckpt, const float *q,
                       const float *k, const float *v, const float *g,
                       const float *beta, float *o,
                       bool *host_inputs = nullptr) {
  int r = check_shape(s);
  if (r) return r;
  if (M < 1 || M > GDN_MAX_TOKENS) return GDN_ERANGE;
  if (s->B == 0) return GDN_OK;
  const size_t sb = state_floats(s) * 4;
  const size_t qkb = (size_t)s->B * M * s->kh * s->kd * 4;
  const size_t vb = (size_t)s->B * M * s->vh * s->vd * 4;
  const size_t gb = (size_t)s->B * M * s->vh * 4;
  Buf in[] = {{S_in, sb}, {q, qkb}, {k, qkb}, {v, vb}, {g, gb}, {beta, gb}};
  Buf out[] = {{S_out, sb}, {o, vb}, {ckpt, sb * (size_t)M}};
  const int nout = ckpt ? 3 : 2;
  // the state and the checkpoints in device memory; token inputs and o
  // also in mapped page-locked host memory
  Buf dev_bufs[] = {in[0], out[0], out[2]};
  r = check_bufs(dev_bufs, ckpt ? 3 : 2);
  if (r) return r;
  r = check_io_bufs(in + 1, 5, host_inputs);
  if (r) return r;
  r = check_io_bufs(out + 1, 1);
  if (r) return r;
  // Outputs never overlap inputs or each other; the one exception is an
  // in-place state (S_out == S_in exactly).
  for (int i = 0; i < nout; ++i) {
    for (int j = 0; j < 6; ++j) {
      if (i == 0 && j == 0 && out[0].p == in[0].p) continue;
      if (overlaps(out[i], in[j])) return GDN_EALIAS;
    }
    for (int j = i + 1; j < nout; ++j)
      if (overlaps(out[i], out[j])) return GDN_EALIAS;
  }
  return GDN_OK;
}

int steps_common(const gdn_shape *s, int M, const float *S_in, float *S_out,
                 float *ckpt, const float *q, const float *k, const float *v,
                 const float *g, const float *beta, float *o,
                 cudaStream_t stream) {
  bool host_inputs = false;
  const int r = steps_common_check(s, M, S_in, S_out, ckpt, q, k, v, g, beta, o,
                                   &host_inputs);
  if (r || s->B == 0) return r;
  cudaGetLastError();  // start from a clean per-thread error state
  // a programmatic dependent of the previous kernel, reading nothing
  // before it ends (launch_steps keeps the ordinary launch for grids that
  // do not fill the GPU)
  return status_of(gdn::launch_steps(S_in, S_out, ckpt, q, k, v, g, beta, o,
                                     s->B, s->kh, s->vh, M, stream,
                                     gdn::kOverlapAny, host_inputs));
}

}  // namespace

extern "C" {

int gdn_step(const gdn_shape *shape, float *S, const float *q, const float *k,
             const float *v, const float *g, const float *beta, float *o,
             gdn_stream_t stream) {
  return steps_common(shape, 1, S, S, nullptr, q, k, v, g, beta, o,
                      (cudaStream_t)stream);
}

int gdn_step_m(const gdn_shape *shape, int M, const float *S_in, float *S_out,
               float *ckpt, const float *q, const float *k, const float *v,
               const float *g, const float *beta, float *o,
               gdn_stream_t stream) {
  return steps_common(shape, M, S_in, S_out, ckpt, q, k, v, g, beta, o,
                      (cudaStream_t)stream);
}

int gdn_mark(const gdn_shape *shape, const float *S, float *snap,
             gdn_stream_t stream) {
  int r = check_shape(shape);
  if (r) return r;
  if (shape->B == 0) return GDN_OK;
  const size_t n = state_floats(shape);
  Buf b[] = {{S, n * 4}, {snap, n * 4}};
  r = check_bufs(b, 2);
  if (r) return r;
  if (overlaps(b[0], b[1])) return GDN_EALIAS;
  cudaGetLastError();
  return status_of(gdn::launch_copy(snap, S, n, (cudaStream_t)stream));
}

int gdn_rollback(const gdn_shape *shape, int M, int m, const float *snap,
                 const float *ckpt, float *S, gdn_stream_t stream) {
  int r = check_shape(shape);
  if (r) return r;
  if (M < 1 || M > GDN_MAX_TOKENS || m < 0 || m > M) return GDN_ERANGE;
  if (shape->B == 0) return GDN_OK;
  const size_t n = state_floats(shape);
  const float *src = m == 0 ? snap : (ckpt ? ckpt + (size_t)(m - 1) * n : nullptr);
  Buf b[] = {{src, n * 4}, {S, n * 4}};
  r = check_bufs(b, 2);
  if (r) return r;
  if (overlaps(b[0], b[1])) return GDN_EALIAS;
  cudaGetLastError();
  return status_of(gdn::launch_copy(S, src, n, (cudaStream_t)stream));
}

int gdn_rollback_seq(const gdn_shape *shape, int M, const int *m_dev,
                     const float *snap, const float *ckpt, float *S,
                     int *err_dev, gdn_stream_t stream) {
  int r = check_shape(shape);
  if (r) return r;
  if (M < 1 || M > GDN_MAX_TOKENS) return GDN_ERANGE;
  if (shape->B == 0) return GDN_OK;
  const size_t n = state_floats(shape);
  Buf b[] = {{snap, n * 4}, {ckpt, n * 4 * (size_t)M}, {S, n * 4},
             {m_dev, (size_t)shape->B * 4}};
  r = check_bufs(b, 4);
  if (r) return r;
  if (err_dev) {
    if (((uintptr_t)err_dev & 3u) != 0) return GDN_EALIGN;
    r = check_device_ptr(err_dev);
    if (r) return r;
  }
  for (int j = 0; j < 4; ++j)
    if (j != 2 && overlaps(b[2], b[j])) return GDN_EALIAS;
  cudaGetLastError();
  return status_of(gdn::launch_rollback_seq(S, snap, ckpt, m_dev, err_dev,
                                            shape->B, shape->vh, M,
                                            (cudaStream_t)stream));
}

size_t gdn_prefill_workspace(const gdn_shape *shape, int T, int chunk,
                             int precision) {
  if (check_shape(shape) || T < 1 || T > GDN_MAX_TOKENS) return 0;
  if (precision != GDN_PREC_FP32 && chunk != 64) return 0;
  return gdn::prefill_workspace_bytes(shape->B, shape->kh, shape->vh, T, chunk,
                                      precision);
}

int gdn_prefill(const gdn_shape *shape, int T, float *S, const float *q,
                const float *k, const float *v, const float *g,
                const float *beta, float *o, int chunk, int precision,
                void *workspace, size_t ws_bytes, gdn_stream_t stream) {
  (void)workspace;
  (void)ws_bytes;
  if (precision == GDN_PREC_FP32)
    return steps_common(shape, T, S, S, nullptr, q, k, v, g, beta, o,
                        (cudaStream_t)stream);
  if (precision != GDN_PREC_BF16X3 && precision != GDN_PREC_BF16)
    return GDN_ERANGE;
  int r = check_shape(shape);
  if (r) return r;
  if (T < 1 || T > GDN_MAX_TOKENS || chunk != 64) return GDN_ERANGE;
  // the copy engine addresses a sequence's rows of q, k, o with strides below 2^40 bytes
  if ((unsigned long long)T * (unsigned long long)shape->vh >= (1ull << 31)) return GDN_ERANGE;
  if (shape->B == 0) return GDN_OK;
  const size_t sb = state_floats(shape) * 4;
  const size_t qkb = (size_t)shape->B * T * shape->kh * shape->kd * 4;
  const size_t vb = (size_t)shape->B * T * shape->vh * shape->vd * 4;
  const size_t gb = (size_t)shape->B * T * shape->vh * 4;
  Buf in[] = {{q, qkb}, {k, qkb}, {v, vb}, {g, gb}, {beta, gb}};
  Buf out[] = {{S, sb}, {o, vb}};
  r = check_bufs(in, 5);
  if (r) return r;
  r = check_bufs(out, 2);
  if (r) return r;
  for (int i = 0; i < 2; ++i)
    for (int j = 0; j < 5; ++j)
      if (overlaps(out[i], in[j])) return GDN_EALIAS;
  if (overlaps(out[0], out[1])) return GDN_EALIAS;
  cudaGetLastError();
  return status_of(gdn::launch_prefill_chunked(
      S, q, k, v, g, beta, o, shape->B, shape->kh, shape->vh, T, precision,
      nullptr, (cudaStream_t)stream));
}

int gdn_prefill_timeouts(unsigned int *count) {
  if (!count) return GDN_EINVAL;
  cudaGetLastError();
  return status_of(gdn::prefill_timeouts(count));
}

int gdn_wait_timeouts(unsigned int *count) {
  if (!count) return GDN_EINVAL;
  cudaGetLastError();
  unsigned int a = 0, b = 0;
  const int r = status_of(gdn::prefill_timeouts(&a));
  if (r) return r;
  const int r2 = status_of(gdn::steps_timeouts(&b));
  if (r2) return r2;
  *count = a + b;
  return GDN_OK;
}

}  // extern "C"

namespace {

size_t round16(size_t n) { return (n + 15) & ~(size_t)15; }

struct LayerSizes {
  size_t conv_dim, hb, xb, wb, ab, pb, qb, vb, gb;
};

LayerSizes layer_sizes(const gdn_shape *s, int M, int ck) {
  LayerSizes z;
  z.conv_dim = (size_t)2 * s->kh * s->kd + (size_t)s->vh * s->vd;
  z.hb = (size_t)s->B * (ck - 1) * z.conv_dim * 4;
  z.xb = (size_t)s->B * M * z.conv_dim * 4;
  z.wb = z.conv_dim * ck * 4;
  z.ab = (size_t)s->B * M * s->vh * 4;
  z.pb = (size_t)s->vh * 4;
  z.qb = (size_t)s->B * M * s->kh * s->kd * 4;
  z.vb = (size_t)s->B * M * s->vh * s->vd * 4;
  z.gb = z.ab;
  return z;
}

// Validation shared by the two layer entry points; outputs q..beta may be
// NULL (checked by the caller).
int check_layer(const gdn_shape *s, int M, int ck, float eps,
                const float *hist_in, float *hist_out, const float *x,
                const float *conv_w, const float *a, const float *b,
                const float *A_log, const float *dt_bias) {
  int r = check_shape(s);
  if (r) return r;
  if (ck != 4) return GDN_ESHAPE;
  if (M < 1 || M > GDN_MAX_TOKENS) return GDN_ERANGE;
  if (!(eps >= 0.0f) || eps > 3.0e38f) return GDN_EINVAL;
  if (s->B == 0) return GDN_OK;
  const LayerSizes z = layer_sizes(s, M, ck);
  Buf in[] = {{hist_in, z.hb}, {x, z.xb}, {conv_w, z.wb}, {a, z.ab},
              {b, z.ab}, {A_log, z.pb}, {dt_bias, z.pb}, {hist_out, z.hb}};
  r = check_bufs(in, 8);
  if (r) return r;
  for (int j = 0; j < 7; ++j)
    if (overlaps(in[7], in[j])) return GDN_EALIAS;
  return GDN_OK;
}

// gdn_layer_step_m's checks of every argument but the workspace, in the
// order that call makes them: the layer inputs and history, then the
// state, checkpoints and o (device memory; o may also be mapped host
// memory), then their overlaps.
int layer_step_args(const gdn_shape *s, int M, int ck, float eps,
                    const float *S_in, float *S_out, float *ckpt,
                    const float *hist_in, float *hist_out, const float *x,
                    const float *conv_w, const float *a, const float *b,
                    const float *A_log, const float *dt_bias, float *o) {
  int r = check_layer(s, M, ck, eps, hist_in, hist_out, x, conv_w, a, b, A_log,
                      dt_bias);
  if (r || s->B == 0) return r;
  const LayerSizes z = layer_sizes(s, M, ck);
  const size_t sb = state_floats(s) * 4;
  Buf dev_bufs[] = {{S_in, sb}, {S_out, sb}, {ckpt, sb * (size_t)M}};
  r = check_bufs(dev_bufs, ckpt ? 3 : 2);
  if (r) return r;
  Buf ob{o, z.vb};
  r = check_io_bufs(&ob, 1);
  if (r) return r;
  Buf outs[] = {dev_bufs[0], dev_bufs[1], ob, dev_bufs[2]};
  const int n = ckpt ? 4 : 3;
  for (int i = 1; i < n; ++i)
    for (int j = 0; j < i; ++j) {
      if (i == 1 && j == 0 && S_out == S_in) continue;
      if (overlaps(outs[i], outs[j])) return GDN_EALIAS;
    }
  return GDN_OK;
}

}  // namespace

extern "C" {

int gdn_layer_prologue_m(const gdn_shape *s, int M, int ck, float eps,
                         const float *hist_in, float *hist_out,
                         const float *x, const float *conv_w, const float *a,
                         const float *b, const float *A_log,
                         const float *dt_bias, float *q, float *k, float *v,
                         float *g, float *beta, gdn_stream_t stream) {
  int r = check_layer(s, M, ck, eps, hist_in, hist_out, x, conv_w, a, b, A_log,
                      dt_bias);
  if (r || s->B == 0) return r;
  const LayerSizes z = layer_sizes(s, M, ck);
  Buf in[] = {{hist_in, z.hb}, {x, z.xb}, {conv_w, z.wb}, {a, z.ab},
              {b, z.ab}, {A_log, z.pb}, {dt_bias, z.pb}, {hist_out, z.hb}};
  Buf out[] = {{q, z.qb}, {k, z.qb}, {v, z.vb}, {g, z.gb}, {beta, z.gb}};
  r = check_bufs(out, 5);
  if (r) return r;
  for (int i = 0; i < 5; ++i) {
    for (int j = 0; j < 8; ++j)
      if (overlaps(out[i], in[j])) return GDN_EALIAS;
    for (int j = i + 1; j < 5; ++j)
      if (overlaps(out[i], out[j])) return GDN_EALIAS;
  }
  cudaGetLastError();
  return status_of(gdn::launch_layer_prologue(
      hist_in, hist_out, x, conv_w, a, b, A_log, dt_bias, eps, q, k, v, g,
      beta, s->B, s->kh, s->vh, M, (cudaStream_t)stream,
      M <= gdn::kOverlapMaxTokens));
}

size_t gdn_layer_workspace(const gdn_shape *s, int M) {
  if (check_shape(s) || M < 1 || M > GDN_MAX_TOKENS) return 0;
  const LayerSizes z = layer_sizes(s, M, 4);
  return round16(z.qb) * 2 + round16(z.vb) + round16(z.gb) * 2;
}

int gdn_layer_step_m(const gdn_shape *s, int M, int ck, float eps,
                     const float *S_in, float *S_out, float *ckpt,
                     const float *hist_in, float *hist_out, const float *x,
                     const float *conv_w, const float *a, const float *b,
                     const float *A_log, const float *dt_bias, float *o,
                     void *workspace, size_t ws_bytes, gdn_stream_t stream) {
  int r = check_layer(s, M, ck, eps, hist_in, hist_out, x, conv_w, a, b, A_log,
                      dt_bias);
  if (r || s->B == 0) return r;
  const size_t need = gdn_layer_workspace(s, M);
  if (ws_bytes < need) return GDN_ERANGE;
  const LayerSizes z = layer_sizes(s, M, ck);
  Buf ws{workspace, need};
  r = check_bufs(&ws, 1);
  if (r) return r;
  // the workspace must not overlap any argument of either step
  const size_t sb = state_floats(s) * 4;
  Buf all[] = {{S_in, sb}, {S_out, sb}, {ckpt, sb * (size_t)M},
               {hist_in, z.hb}, {hist_out, z.hb}, {x, z.xb}, {conv_w, z.wb},
               {a, z.ab}, {b, z.ab}, {A_log, z.pb}, {dt_bias, z.pb},
               {o, z.vb}};
  for (int j = 0; j < 12; ++j)
    if (overlaps(ws, all[j])) return GDN_EALIAS;
  char *w = static_cast<char *>(workspace);
  float *q = reinterpret_cast<float *>(w);
  float *k = reinterpret_cast<float *>(w + round16(z.qb));
  float *v = reinterpret_cast<float *>(w + 2 * round16(z.qb));
  float *g = reinterpret_cast<float *>(w + 2 * round16(z.qb) + round16(z.vb));
  float *beta = reinterpret_cast<float *>(w + 2 * round16(z.qb) + round16(z.vb) +
                                          round16(z.gb));
  // the state call validates its own arguments before anything is launched
  const gdn_shape *sh = s;
  r = steps_common_check(sh, M, S_in, S_out, ckpt, q, k, v, g, beta, o);
  if (r) return r;
  cudaGetLastError();
  // the prologue starts behind the kernel before it (short launches) and
  // touches nothing before that kernel has ended
  cudaError_t e = gdn::launch_layer_prologue(
      hist_in, hist_out, x, conv_w, a, b, A_log, dt_bias, eps, q, k, v, g,
      beta, s->B, s->kh, s->vh, M, (cudaStream_t)stream,
      M <= gdn::kOverlapMaxTokens);
  if (e != cudaSuccess) return GDN_ECUDA;
  // the update overlaps the prologue's tail: it loads the state, which the
  // prologue never writes, before it waits for q, k, v, g, beta
  return status_of(gdn::launch_steps(S_in, S_out, ckpt, q, k, v, g, beta, o,
                                     s->B, s->kh, s->vh, M,
                                     (cudaStream_t)stream, gdn::kOverlapPrologue));
}

int gdn_layer_hist_rollback(const gdn_shape *s, int M, int ck,
                            const int *m_dev, const float *hist_snap,
                            const float *x, float *hist, int *err_dev,
                            gdn_stream_t stream) {
  int r = check_shape(s);
  if (r) return r;
  if (ck != 4) return GDN_ESHAPE;
  if (M < 1 || M > GDN_MAX_TOKENS) return GDN_ERANGE;
  if (s->B == 0) return GDN_OK;
  const size_t conv_dim = (size_t)2 * s->kh * s->kd + (size_t)s->vh * s->vd;
  const size_t hb = (size_t)s->B * (ck - 1) * conv_dim * 4;
  Buf b[] = {{hist_snap, hb}, {x, (size_t)s->B * M * conv_dim * 4}, {hist, hb},
             {m_dev, (size_t)s->B * 4}};
  r = check_bufs(b, 4);
  if (r) return r;
  if (err_dev) {
    if (((uintptr_t)err_dev & 3u) != 0) return GDN_EALIGN;
    r = check_device_ptr(err_dev);
    if (r) return r;
  }
  for (int j = 0; j < 4; ++j)
    if (j != 2 && overlaps(b[2], b[j])) return GDN_EALIAS;
  cudaGetLastError();
  return status_of(gdn::launch_hist_rollback(hist, hist_snap, x, m_dev, err_dev,
                                             s->B, M, (int)conv_dim,
                                             (cudaStream_t)stream));
}

int gdn_gated_rmsnorm_m(const gdn_shape *s, int M, float eps, const float *o,
                        const float *z, const float *w, float *y,
                        gdn_stream_t stream) {
  int r = check_shape(s);
  if (r) return r;
  if (M < 1 || M > GDN_MAX_TOKENS) return GDN_ERANGE;
  if (!(eps >= 0.0f) || eps > 3.0e38f) return GDN_EINVAL;
  if (s->B == 0) return GDN_OK;
  const size_t rows = (size_t)s->B * M * s->vh;
  const size_t ob = rows * s->vd * 4;
  Buf b[] = {{o, ob}, {z, ob}, {w, (size_t)s->vd * 4}, {y, ob}};
  r = check_bufs(b, 4);
  if (r) return r;
  // y may be o exactly (in place); otherwise no output overlap
  if (y != o && overlaps(b[3], b[0])) return GDN_EALIAS;
  if (overlaps(b[3], b[1]) || overlaps(b[3], b[2])) return GDN_EALIAS;
  cudaGetLastError();
  return status_of(gdn::launch_gate_norm(o, z, w, y, eps, rows,
                                         (cudaStream_t)stream));
}

const char *gdn_strerror(int status) {
  switch (status) {
    case GDN_OK: return "success";
    case GDN_EINVAL: return "invalid argument (NULL pointer or bad value)";
    case GDN_ESHAPE: return "unsupported shape (kd == vd == 128, vh % kh == 0, B >= 0)";
    case GDN_EALIGN: return "pointer not 16-byte aligned";
    case GDN_ECUDA: return "CUDA runtime error or kernel launch failure";
    case GDN_ERANGE: return "count out of range (M, m, T, chunk, precision or workspace)";
    case GDN_EPTR: return "pointer is not device memory of the current device";
    case GDN_EALIAS: return "buffers overlap where they must not";
    case GDN_ESCRATCH:
      return "request needs more than the static scratch of "
             "gdn_layer_step_m_noalloc (GDN_NOALLOC_SCRATCH_BYTES)";
    default: return "unknown status";
  }
}

int gdn_version(void) { return 100; }

}  // extern "C"

namespace gdn {
int layer_step_check(const gdn_shape *s, int M, int ck, float eps,
                     const float *S_in, float *S_out, float *ckpt,
                     const float *hist_in, float *hist_out, const float *x,
                     const float *conv_w, const float *a, const float *b,
                     const float *A_log, const float *dt_bias, float *o) {
  return layer_step_args(s, M, ck, eps, S_in, S_out, ckpt, hist_in, hist_out,
                         x, conv_w, a, b, A_log, dt_bias, o);
}
}  // namespace gdn
