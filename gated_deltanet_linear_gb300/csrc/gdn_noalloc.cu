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
// Make that first call before any stream capture starts.
//
// Sharing.  Every call on a device uses the same array and leaves its
// contents behind.  Nothing in it has to start at zero: the prologue writes
// every byte of q, k, v, g and beta that the update then reads, so nothing is
// cleared.  Two calls whose work overlaps on the GPU (different streams, no
// ordering between them) race on the array and give wrong results; order
// such calls on one stream or with events.

#include <mutex>

#include "gdn.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char
    g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

std::mutex g_setup_mutex;
void *g_scratch_of_device[kMaxDevices];  // guarded by g_setup_mutex

// Device address of the scratch on the current device (set-up on first use).
int scratch_of_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GDN_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return GDN_ECUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_of_device[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return GDN_ECUDA;
    }
    g_scratch_of_device[dev] = p;
  }
  *out = g_scratch_of_device[dev];
  return GDN_OK;
}

}  // namespace

extern "C" int gdn_layer_step_m_noalloc(
    const gdn_shape *s, int M, int ck, float eps, const float *S_in,
    float *S_out, float *ckpt, const float *hist_in, float *hist_out,
    const float *x, const float *conv_w, const float *a, const float *b,
    const float *A_log, const float *dt_bias, float *o, gdn_stream_t stream) {
  if (!s) return GDN_EINVAL;
  // a bad shape or count gets the same status as from gdn_layer_step_m
  const size_t need = gdn_layer_workspace(s, M);
  if (need == 0 || s->B == 0)
    return gdn_layer_step_m(s, M, ck, eps, S_in, S_out, ckpt, hist_in,
                            hist_out, x, conv_w, a, b, A_log, dt_bias, o,
                            nullptr, 0, stream);
  if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ESCRATCH;
  void *scratch = nullptr;
  const int r = scratch_of_current_device(&scratch);
  if (r) return r;
  return gdn_layer_step_m(s, M, ck, eps, S_in, S_out, ckpt, hist_in, hist_out,
                          x, conv_w, a, b, A_log, dt_bias, o, scratch,
                          (size_t)GDN_NOALLOC_SCRATCH_BYTES, stream);
}
