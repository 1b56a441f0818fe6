// gdn_layer_step_m_noalloc: the layer step (prologue + state update) for
// callers that cannot allocate device memory, with its intermediate q, k, v,
// g and beta in a scratch array that the library itself holds.
//
// Who cannot allocate.  gdn_layer_step_m asks its caller for a workspace.
// Some callers have no way to provide one: a plain C host that is handed only
// the device pointers of a layer's tensors by an embedding runtime whose
// caching allocator it cannot reach, or a decode loop that must not call
// cudaMalloc between steps, because cudaMalloc can synchronise the device and
// can fail under memory pressure in the middle of a serving step.  This entry
// point takes the same inputs and outputs and allocates nothing.
//
// The scratch.  A file-scope __device__ array of GDN_NOALLOC_SCRATCH_BYTES
// (16 MiB).  The CUDA runtime creates it when the library's device code is
// loaded on a GPU, and that GPU holds it until the process exits.  In host
// code its name is only a host-side stand-in for the symbol, never a device
// address: the address is looked up with cudaGetSymbolAddress, once per
// device, with that device current, on the first call made on that device.
// Make that first call before any stream capture starts.  The lookup is
// tied to the device's CUDA context: after cudaDeviceReset the runtime
// loads the device code again (possibly at another address), and the next
// call repeats the set-up in the new context instead of using the old
// address.
//
// Status codes.  Every argument is checked as gdn_layer_step_m checks it
// first; GDN_ESCRATCH is returned only for a request that is otherwise
// valid and larger than the array.
//
// Sharing.  Every call on a device uses the same array and leaves its
// contents behind.  Nothing in it has to start at zero: the prologue writes
// every byte of q, k, v, g and beta that the update then reads, so nothing is
// cleared.  Two calls whose work overlaps on the GPU (different streams, no
// ordering between them) race on the array and give wrong results; order
// such calls on one stream or with events.

#include <cudaTypedefs.h>

#include <mutex>

#include "gdn.h"
#include "gdn_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char
    g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

struct Setup {
  unsigned long long ctx_id;  // context the address belongs to (0: none yet)
  void *addr;
};

std::mutex g_setup_mutex;
Setup g_setup[kMaxDevices];  // guarded by g_setup_mutex

// The driver's current-context queries, reached through the runtime (the
// library does not link the driver library); null if unavailable.
struct CtxQueries {
  PFN_cuCtxGetCurrent_v4000 current = nullptr;
  PFN_cuCtxGetId_v12000 id = nullptr;
};

const CtxQueries &ctx_queries() {
  static CtxQueries q;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000,
                                         cudaEnableDefault, &r) == cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      q.current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000,
                                         cudaEnableDefault, &r) == cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      q.id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return q;
}

// Unique id of the calling thread's current context, 0 if there is none.
unsigned long long current_ctx_id() {
  const CtxQueries &q = ctx_queries();
  if (!q.current || !q.id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (q.current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (q.id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch on the current device, looked up once per
// device and context (the set-up).
int scratch_of_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GDN_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return GDN_ECUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  Setup &st = g_setup[dev];
  unsigned long long id = current_ctx_id();
  if (!st.addr || id == 0 || id != st.ctx_id) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return GDN_ECUDA;
    }
    // the lookup makes the device's context current if it was not yet
    if (id == 0) id = current_ctx_id();
    st.addr = p;
    st.ctx_id = id;  // 0 (queries unavailable): the set-up runs every call
  }
  *out = st.addr;
  return GDN_OK;
}

}  // namespace

extern "C" int gdn_layer_step_m_noalloc(
    const gdn_shape *s, int M, int ck, float eps, const float *S_in,
    float *S_out, float *ckpt, const float *hist_in, float *hist_out,
    const float *x, const float *conv_w, const float *a, const float *b,
    const float *A_log, const float *dt_bias, float *o, gdn_stream_t stream) {
  // every argument but the workspace first, with gdn_layer_step_m's status
  const int r = gdn::layer_step_check(s, M, ck, eps, S_in, S_out, ckpt,
                                      hist_in, hist_out, x, conv_w, a, b,
                                      A_log, dt_bias, o);
  if (r || s->B == 0) return r;
  const size_t need = gdn_layer_workspace(s, M);
  if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ESCRATCH;
  void *scratch = nullptr;
  const int rs = scratch_of_current_device(&scratch);
  if (rs) return rs;
  return gdn_layer_step_m(s, M, ck, eps, S_in, S_out, ckpt, hist_in, hist_out,
                          x, conv_w, a, b, A_log, dt_bias, o, scratch,
                          (size_t)GDN_NOALLOC_SCRATCH_BYTES, stream);
}
