// decode_noalloc.cu -- nd_swa_sink_decode_noalloc: the decode step for callers
// that cannot hand the library a workspace buffer.
//
// Who needs it: code that runs where allocating device memory is not
// allowed or not possible -- a real-time serving loop that must not call
// cudaMalloc (it can synchronise the device and stall every stream), or an
// embedding host (another runtime, a plugin ABI) that owns all device memory
// and gives the plugin only its input and output buffers.
//
// How: the split-K partials that nd_swa_sink_decode keeps in the caller's
// workspace live here in one file-scope device array of fixed size.  Host
// code never passes the array's name to a kernel (in host code that name is
// a host-side shadow, not a device address); it looks up the device address
// once per device with cudaGetSymbolAddress and passes that pointer as the
// workspace of the ordinary decode entry point.
#include <cuda_runtime.h>

#include <mutex>

#include "nd.h"
#include "nd_internal.h"

namespace {

// Shared by every call on a device, held by every device that loads libnd
// until the process exits.  Each call writes every partial it later reads,
// so nothing here has to start at zero.
static __device__ __align__(256) unsigned char g_decode_scratch[ND_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on device `dev`, which is current (set
// up on the first call per device).  Returns the CUDA error of the lookup.
cudaError_t scratch_address(int dev, void **out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int nd_swa_sink_decode_noalloc(const void *q, const nd_kv_cache *cache, int n_q_heads,
                                          int window, void *out, float *lse, nd_stream_t stream) {
  // the same argument checks, in the same order, as nd_swa_sink_decode, so a
  // shape it refuses is refused here for the same reason
  int st = nd::validate_decode(q, cache, n_q_heads, window, out);
  if (st != ND_OK || cache->batch == 0) return st;
  const size_t need = nd_swa_sink_decode_workspace_size(cache->batch, n_q_heads, cache->n_kv_heads,
                                                        cache->head_dim, cache->sink_cap + cache->ring_cap);
  if (need > ND_NOALLOC_SCRATCH_BYTES) return ND_ERR_WORKSPACE;
  int dev = 0;
  if ((st = nd::check_device(&dev)) != ND_OK) return st;
  void *scratch = nullptr;
  const cudaError_t e = scratch_address(dev, &scratch);
  if (e != cudaSuccess) {
    cudaGetLastError();  // reported through the status, not left sticky
    return nd::fail_cuda(e);
  }
  return nd_swa_sink_decode(q, cache, n_q_heads, window, out, lse, scratch, ND_NOALLOC_SCRATCH_BYTES,
                            stream);
}
