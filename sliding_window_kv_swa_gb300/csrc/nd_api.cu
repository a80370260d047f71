// nd_api.cu -- the extern "C" entry points of libnd (see include/nd.h):
// host-side argument validation, workspace carving and kernel dispatch.
// Nothing here allocates memory; nothing here synchronises except
// nd_device_errors().
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "nd.h"
#include "nd_internal.h"

namespace nd {

// Device error word: kernels OR flags into it (bounded waits that gave up,
// cache metadata out of range).  One copy per device the module is loaded on.
__device__ int g_device_errors = 0;

namespace {

thread_local int t_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_err_ptr[kMaxDevices] = {};
int g_arch_ok[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other

}  // namespace

int fail_cuda(cudaError_t e) {
  t_last_cuda_error = int(e);
  return ND_ERR_CUDA;
}

// Returns ND_OK if the current device is an sm_103 part.
int check_device(int *dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return ND_ERR_UNSUPPORTED;
  if (dev_out) *dev_out = dev;
  int ok = __atomic_load_n(&g_arch_ok[dev], __ATOMIC_ACQUIRE);
  if (ok == 0) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e != cudaSuccess) return fail_cuda(e);
    e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return fail_cuda(e);
    ok = (major == 10 && minor == 3) ? 1 : -1;
    __atomic_store_n(&g_arch_ok[dev], ok, __ATOMIC_RELEASE);
  }
  return ok == 1 ? ND_OK : ND_ERR_UNSUPPORTED;
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int finish(cudaError_t e) { return e == cudaSuccess ? ND_OK : fail_cuda(e); }

int validate_cache(const nd_kv_cache *c) {
  if (!c) return ND_ERR_INVALID_ARG;
  if (c->batch < 0 || c->n_kv_heads <= 0 || c->sink_cap < 0 || c->ring_cap < 0)
    return ND_ERR_INVALID_ARG;
  if (c->head_dim <= 0 || c->head_dim % 32) return ND_ERR_INVALID_ARG;
  if (c->batch == 0) return ND_OK;
  if (!c->k_codes || !c->v_codes || !c->k_scale || !c->v_scale || !c->sink_len ||
      !c->ring_start || !c->ring_len || !c->seq_len)
    return ND_ERR_INVALID_ARG;
  if (!aligned16(c->k_codes) || !aligned16(c->v_codes) || !aligned16(c->k_scale) ||
      !aligned16(c->v_scale))
    return ND_ERR_INVALID_ARG;
  return ND_OK;
}

}  // namespace

int validate_decode(const void *q, const nd_kv_cache *cache, int n_q_heads, int window, const void *out) {
  int st = validate_cache(cache);
  if (st != ND_OK) return st;
  if (window < 1 || n_q_heads <= 0 || n_q_heads % cache->n_kv_heads) return ND_ERR_INVALID_ARG;
  const int G = n_q_heads / cache->n_kv_heads;
  if (G > 8) return ND_ERR_UNSUPPORTED;
  if (cache->head_dim != 64 && cache->head_dim != 128) return ND_ERR_UNSUPPORTED;
  if (cache->batch == 0) return ND_OK;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return ND_ERR_INVALID_ARG;
  if (cache->sink_cap + cache->ring_cap <= 0) return ND_ERR_INVALID_ARG;
  return ND_OK;
}

int *device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  int *p = __atomic_load_n(&g_err_ptr[dev], __ATOMIC_ACQUIRE);
  if (p) return p;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_err_ptr[dev]) {
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_device_errors) != cudaSuccess) return nullptr;
    __atomic_store_n(&g_err_ptr[dev], static_cast<int *>(addr), __ATOMIC_RELEASE);
  }
  return g_err_ptr[dev];
}

}  // namespace nd

using namespace nd;

extern "C" {

const char *nd_version(void) { return "nd 0.1.0 sm_103a"; }

const char *nd_status_string(int status) {
  switch (status) {
    case ND_OK: return "ND_OK";
    case ND_ERR_INVALID_ARG: return "ND_ERR_INVALID_ARG";
    case ND_ERR_UNSUPPORTED: return "ND_ERR_UNSUPPORTED";
    case ND_ERR_CUDA: return "ND_ERR_CUDA";
    case ND_ERR_WORKSPACE: return "ND_ERR_WORKSPACE";
    case ND_ERR_DEVICE: return "ND_ERR_DEVICE";
    default: return "ND_ERR_UNKNOWN";
  }
}

int nd_last_cuda_error(void) { return t_last_cuda_error; }

int nd_device_errors(int *flags_out, int clear) {
  if (!flags_out) return ND_ERR_INVALID_ARG;
  int st = check_device(nullptr);
  if (st != ND_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail_cuda(e);
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_errors, sizeof(int));
  if (e != cudaSuccess) return fail_cuda(e);
  *flags_out = v;
  if (clear && v) {
    int zero = 0;
    e = cudaMemcpyToSymbol(g_device_errors, &zero, sizeof(int));
    if (e != cudaSuccess) return fail_cuda(e);
  }
  return ND_OK;
}

int nd_kv_append_quant(const nd_kv_cache *cache, const void *k_new, const void *v_new,
                       int to_sink, nd_stream_t stream) {
  int st = validate_cache(cache);
  if (st != ND_OK) return st;
  if (cache->batch == 0) return ND_OK;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return ND_ERR_INVALID_ARG;
  if (!to_sink && cache->ring_cap <= 0) return ND_ERR_INVALID_ARG;
  if (to_sink && cache->sink_cap <= 0) return ND_ERR_INVALID_ARG;
  const int d = cache->head_dim;
  if (d != 32 && d != 64 && d != 128 && d != 256) return ND_ERR_UNSUPPORTED;
  if ((st = check_device(nullptr)) != ND_OK) return st;
  return finish(launch_kv_append_quant(*cache, k_new, v_new, to_sink ? 1 : 0, device_error_word(),
                                       reinterpret_cast<cudaStream_t>(stream)));
}

int nd_kv_quant_rows(const void *x, int64_t n_rows, int head_dim, int8_t *codes, float *scales,
                     nd_stream_t stream) {
  if (n_rows < 0) return ND_ERR_INVALID_ARG;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128 && head_dim != 256)
    return head_dim > 0 && head_dim % 32 == 0 ? ND_ERR_UNSUPPORTED : ND_ERR_INVALID_ARG;
  if (n_rows == 0) return ND_OK;
  if (!x || !codes || !scales || !aligned16(x) || !aligned16(codes) || !aligned16(scales))
    return ND_ERR_INVALID_ARG;
  int st = check_device(nullptr);
  if (st != ND_OK) return st;
  return finish(launch_kv_quant_rows(x, n_rows, head_dim, codes, scales,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

size_t nd_kv_cache_from_prefill_workspace_size(int cache_batch, int sink_cap, int ring_cap) {
  if (cache_batch <= 0 || sink_cap < 0 || ring_cap <= 0) return 0;
  return round_up(size_t(cache_batch) * kv_fill_plan_ints(sink_cap, ring_cap) * sizeof(int32_t), 256);
}

int nd_kv_cache_from_prefill(const nd_kv_cache *cache, const void *k, const void *v, int batch, int T,
                             const int32_t *seg_ids, const uint8_t *sink, const int32_t *src_row,
                             const int32_t *src_seg, void *workspace, size_t workspace_bytes,
                             nd_stream_t stream) {
  int st = validate_cache(cache);
  if (st != ND_OK) return st;
  if (batch < 0 || T < 0) return ND_ERR_INVALID_ARG;
  if (cache->ring_cap <= 0) return ND_ERR_INVALID_ARG;
  const int d = cache->head_dim;
  if (d != 32 && d != 64 && d != 128 && d != 256) return ND_ERR_UNSUPPORTED;
  if (cache->batch == 0) return ND_OK;
  if (!src_row || (seg_ids && !src_seg)) return ND_ERR_INVALID_ARG;
  if (size_t(batch) * T > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return ND_ERR_INVALID_ARG;
  const size_t need = nd_kv_cache_from_prefill_workspace_size(cache->batch, cache->sink_cap, cache->ring_cap);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ND_ERR_WORKSPACE;
  if ((st = check_device(nullptr)) != ND_OK) return st;
  return finish(launch_kv_fill(*cache, k, v, batch, T, seg_ids, sink, src_row, src_seg,
                               static_cast<int32_t *>(workspace), device_error_word(),
                               reinterpret_cast<cudaStream_t>(stream)));
}

size_t nd_swa_sink_decode_workspace_size(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                         int max_slots) {
  if (batch <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_slots <= 0) return 0;
  return decode_workspace_bytes(batch, n_q_heads, head_dim, max_slots, n_kv_heads);
}

int nd_swa_sink_decode(const void *q, const nd_kv_cache *cache, int n_q_heads, int window,
                       void *out, float *lse, void *workspace, size_t workspace_bytes,
                       nd_stream_t stream) {
  int st = validate_decode(q, cache, n_q_heads, window, out);
  if (st != ND_OK || cache->batch == 0) return st;
  const int max_slots = cache->sink_cap + cache->ring_cap;  // every physical slot is walked
  DecodePlan pl = plan_decode(cache->batch, cache->n_kv_heads, max_slots, cache->head_dim);
  if (pl.n_split > 1) {
    size_t need = size_t(cache->batch) * n_q_heads * pl.n_split * (cache->head_dim + 2) * sizeof(float);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ND_ERR_WORKSPACE;
  }
  if ((st = check_device(nullptr)) != ND_OK) return st;
  return finish(launch_decode(q, *cache, n_q_heads, window, out, lse, workspace, workspace_bytes,
                              device_error_word(), reinterpret_cast<cudaStream_t>(stream)));
}

// Shared by nd_swa_sink_decode_step and its host-buffer form; every pointer
// is a device pointer and the arguments are already validated.
static int decode_step_device(const void *q, const nd_kv_cache *cache, const void *k_new,
                              const void *v_new, int n_q_heads, int window, void *out, float *lse,
                              void *workspace, size_t workspace_bytes, cudaStream_t s) {
  const int max_slots = cache->sink_cap + cache->ring_cap;
  int *err = device_error_word();
  if (decode_step_fuses(cache->batch, cache->n_kv_heads, max_slots, cache->head_dim))
    return finish(launch_decode(q, *cache, n_q_heads, window, out, lse, workspace, workspace_bytes, err, s,
                                k_new, v_new));
  cudaError_t e = launch_kv_append_quant(*cache, k_new, v_new, 0, err, s);
  if (e != cudaSuccess) return finish(e);
  return finish(launch_decode(q, *cache, n_q_heads, window, out, lse, workspace, workspace_bytes, err, s));
}

// Argument checks shared by both forms of the step (pointer alignment is
// checked where the pointers are device pointers).
static int check_step_args(const nd_kv_cache *cache, int n_q_heads, int window) {
  int st = validate_cache(cache);
  if (st != ND_OK) return st;
  if (window < 1 || n_q_heads <= 0 || n_q_heads % cache->n_kv_heads) return ND_ERR_INVALID_ARG;
  const int G = n_q_heads / cache->n_kv_heads;
  if (G > 8) return ND_ERR_UNSUPPORTED;
  if (cache->head_dim != 64 && cache->head_dim != 128) return ND_ERR_UNSUPPORTED;
  if (cache->ring_cap <= 0) return ND_ERR_INVALID_ARG;
  return ND_OK;
}

static size_t split_scratch_bytes(const nd_kv_cache *cache, int n_q_heads) {
  const int max_slots = cache->sink_cap + cache->ring_cap;
  DecodePlan pl = plan_decode(cache->batch, cache->n_kv_heads, max_slots, cache->head_dim);
  return pl.n_split > 1 ? size_t(cache->batch) * n_q_heads * pl.n_split * (cache->head_dim + 2) * sizeof(float)
                        : 0;
}

int nd_swa_sink_decode_step(const void *q, const nd_kv_cache *cache, const void *k_new,
                            const void *v_new, int n_q_heads, int window, void *out, float *lse,
                            void *workspace, size_t workspace_bytes, nd_stream_t stream) {
  int st = check_step_args(cache, n_q_heads, window);
  if (st != ND_OK) return st;
  if (cache->batch == 0) return ND_OK;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return ND_ERR_INVALID_ARG;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return ND_ERR_INVALID_ARG;
  const size_t need = split_scratch_bytes(cache, n_q_heads);
  if (need && (!workspace || workspace_bytes < need || !aligned16(workspace))) return ND_ERR_WORKSPACE;
  if ((st = check_device(nullptr)) != ND_OK) return st;
  return decode_step_device(q, cache, k_new, v_new, n_q_heads, window, out, lse, workspace, workspace_bytes,
                            reinterpret_cast<cudaStream_t>(stream));
}

// Device staging for the host-buffer step, at the front of its workspace:
// q, k_new, v_new back to back (each a multiple of 128 bytes: head_dim is 64
// or 128), then out and lse back to back, then the decode's own split
// scratch.  Back to back so the packed form moves each side in one copy.
struct HostStepLayout {
  size_t q, kn, vn, out, lse, split, total;
};
static HostStepLayout host_step_layout(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                       int max_slots) {
  HostStepLayout L;
  const size_t qb = size_t(batch) * n_q_heads * head_dim * 2, kb = size_t(batch) * n_kv_heads * head_dim * 2;
  L.q = 0;
  L.kn = L.q + qb;
  L.vn = L.kn + kb;
  L.out = round_up(L.vn + kb, 256);
  L.lse = L.out + qb;
  L.split = L.lse + round_up(size_t(batch) * n_q_heads * sizeof(float), 256);
  L.total = L.split + decode_workspace_bytes(batch, n_q_heads, head_dim, max_slots, n_kv_heads);
  return L;
}

size_t nd_swa_sink_decode_step_host_workspace_size(int batch, int n_q_heads, int n_kv_heads,
                                                   int head_dim, int max_slots) {
  if (batch <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_slots <= 0) return 0;
  return host_step_layout(batch, n_q_heads, n_kv_heads, head_dim, max_slots).total;
}

// Device address of a page-locked host buffer, or NULL when `p` is not
// page-locked memory the device can address.
static void *mapped_host(const void *p) {
  cudaPointerAttributes a;
  if (!p || cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// The host-buffer step.  packed_in: q_host holds q, k_new, v_new back to
// back; packed_out: lse follows out in out_host.  Page-locked, 16-byte
// aligned host buffers are read (q, k_new, v_new) and written (out, lse) in
// place by the step's own kernels over the host link -- no copy launches
// and no staging; any other host memory is staged in the workspace by
// cudaMemcpyAsync (one copy per buffer each way).
static int decode_step_host(const void *q_host, const nd_kv_cache *cache, const void *k_new_host,
                            const void *v_new_host, bool packed_in, int n_q_heads, int window,
                            void *out_host, float *lse_host, bool packed_out, void *workspace,
                            size_t workspace_bytes, nd_stream_t stream) {
  int st = check_step_args(cache, n_q_heads, window);
  if (st != ND_OK) return st;
  if (cache->batch == 0) return ND_OK;
  if (!q_host || !out_host || (!packed_in && (!k_new_host || !v_new_host))) return ND_ERR_INVALID_ARG;
  const int B = cache->batch, Hkv = cache->n_kv_heads, d = cache->head_dim;
  const HostStepLayout L = host_step_layout(B, n_q_heads, Hkv, d, cache->sink_cap + cache->ring_cap);
  if (!workspace || workspace_bytes < L.total || !aligned16(workspace)) return ND_ERR_WORKSPACE;
  if ((st = check_device(nullptr)) != ND_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  const size_t qb = size_t(B) * n_q_heads * d * 2, kb = size_t(B) * Hkv * d * 2;
  const size_t lb = size_t(B) * n_q_heads * sizeof(float);
  // device-addressable host buffers (NULL: not page-locked or not 16-byte
  // aligned -- staged instead)
  auto direct = [](const void *h) -> char * {
    void *dp = mapped_host(h);
    return dp && aligned16(dp) ? static_cast<char *>(dp) : nullptr;
  };
  cudaError_t e = cudaSuccess;
  // inputs: q, k_new, v_new (qb and kb are multiples of 128 bytes, so the
  // packed pieces stay 16-byte aligned)
  const char *qd, *kd, *vd;
  if (packed_in) {
    const char *in = direct(q_host);
    if (!in) {
      e = cudaMemcpyAsync(ws + L.q, q_host, qb + 2 * kb, cudaMemcpyHostToDevice, s);
      in = ws + L.q;
    }
    qd = in, kd = in + qb, vd = in + qb + kb;
  } else {
    const void *h[3] = {q_host, k_new_host, v_new_host};
    const size_t off[3] = {L.q, L.kn, L.vn}, len[3] = {qb, kb, kb};
    const char *dd[3];
    for (int i = 0; i < 3 && e == cudaSuccess; ++i) {
      dd[i] = direct(h[i]);
      if (!dd[i]) {
        e = cudaMemcpyAsync(ws + off[i], h[i], len[i], cudaMemcpyHostToDevice, s);
        dd[i] = ws + off[i];
      }
    }
    qd = dd[0], kd = dd[1], vd = dd[2];
  }
  if (e != cudaSuccess) return finish(e);
  // outputs: out and (optional) lse, written in place or staged
  const bool want_lse = packed_out || lse_host;
  char *od = direct(out_host);
  const bool out_direct = od != nullptr;
  float *ld = nullptr;
  bool lse_direct = false;
  if (packed_out) {
    if (!out_direct) od = ws + L.out;  // L.lse follows L.out: out | lse stay back to back
    ld = reinterpret_cast<float *>(od + qb);
    lse_direct = out_direct;
  } else {
    if (!out_direct) od = ws + L.out;
    if (lse_host) {
      char *lp = direct(lse_host);
      lse_direct = lp != nullptr;
      ld = reinterpret_cast<float *>(lse_direct ? lp : ws + L.lse);
    }
  }
  st = decode_step_device(qd, cache, kd, vd, n_q_heads, window, od, want_lse ? ld : nullptr, ws + L.split,
                          workspace_bytes - L.split, s);
  if (st != ND_OK) return st;
  if (!out_direct)
    e = cudaMemcpyAsync(out_host, od, packed_out ? qb + lb : qb, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && lse_host && !packed_out && !lse_direct)
    e = cudaMemcpyAsync(lse_host, ld, lb, cudaMemcpyDeviceToHost, s);
  return finish(e);
}

int nd_swa_sink_decode_step_host(const void *q_host, const nd_kv_cache *cache, const void *k_new_host,
                                 const void *v_new_host, int n_q_heads, int window, void *out_host,
                                 float *lse_host, void *workspace, size_t workspace_bytes,
                                 nd_stream_t stream) {
  return decode_step_host(q_host, cache, k_new_host, v_new_host, false, n_q_heads, window, out_host, lse_host,
                          false, workspace, workspace_bytes, stream);
}

int nd_swa_sink_decode_step_host_packed(const void *in_host, const nd_kv_cache *cache, int n_q_heads,
                                        int window, void *out_host, int with_lse, void *workspace,
                                        size_t workspace_bytes, nd_stream_t stream) {
  return decode_step_host(in_host, cache, nullptr, nullptr, true, n_q_heads, window, out_host, nullptr,
                          with_lse != 0, workspace, workspace_bytes, stream);
}

// Compressed decode step: rotated q at the front of the workspace, then the
// decode's split scratch.
static size_t compressed_q_bytes(int batch, int n_q_heads, int head_dim) {
  return round_up(size_t(batch) * n_q_heads * head_dim * 2, 256);
}

size_t nd_compressed_decode_step_workspace_size(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                                int max_slots) {
  if (batch <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_slots <= 0) return 0;
  return compressed_q_bytes(batch, n_q_heads, head_dim) +
         decode_workspace_bytes(batch, n_q_heads, head_dim, max_slots, n_kv_heads);
}

int nd_compressed_decode_step(const void *q, const nd_compressed_cache *cache, const void *k_new,
                              const void *v_new, int n_q_heads, int window, float rope_theta, void *out,
                              float *lse, void *workspace, size_t workspace_bytes, nd_stream_t stream) {
  if (!cache) return ND_ERR_INVALID_ARG;
  const nd_kv_cache *kv = &cache->kv;
  int st = validate_decode(q, kv, n_q_heads, window, out);
  if (st != ND_OK) return st;
  if (cache->block < 1 || cache->n_pinned < 0 || cache->n_pinned > kv->sink_cap) return ND_ERR_INVALID_ARG;
  if (kv->ring_cap < window) return ND_ERR_INVALID_ARG;  // the exact window must fit the ring
  if (kv->batch == 0) return ND_OK;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return ND_ERR_INVALID_ARG;
  if (!cache->k_sum || !cache->v_sum || !aligned16(cache->k_sum) || !aligned16(cache->v_sum))
    return ND_ERR_INVALID_ARG;
  const int B = kv->batch, d = kv->head_dim, max_slots = kv->sink_cap + kv->ring_cap;
  const size_t qb = compressed_q_bytes(B, n_q_heads, d);
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < qb + decode_workspace_bytes(B, n_q_heads, d, max_slots, kv->n_kv_heads))
    return ND_ERR_WORKSPACE;
  if ((st = check_device(nullptr)) != ND_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int *err = device_error_word();
  char *ws = static_cast<char *>(workspace);
  cudaError_t e = launch_compressed_append(*kv, cache->k_sum, cache->v_sum, cache->block, cache->n_pinned,
                                           window, q, n_q_heads, k_new, v_new, ws, rope_theta, err, s);
  if (e != cudaSuccess) return fail_cuda(e);
  return finish(launch_decode(ws, *kv, n_q_heads, window, out, lse, ws + qb, workspace_bytes - qb, err, s));
}

// Prefill workspace: the rotation buffers (when rope_theta != 0), then the
// tile records and plan (bf16 path).  Returns the offset of the plan.
static size_t prefill_rotation_bytes(nd_dtype dtype, int batch, int T, int n_q_heads, int n_kv_heads,
                                     int head_dim, float rope_theta) {
  const size_t esz = dtype == ND_F32 ? 4 : 2;
  size_t bytes = 0;
  if (rope_theta != 0.f) {
    // rotated q (fp32 path only: the bf16 kernel rotates q as it stages it),
    // rotated k, the angle table
    if (dtype == ND_F32) bytes += round_up(size_t(batch) * T * n_q_heads * head_dim * esz, 256);
    bytes += round_up(size_t(batch) * T * n_kv_heads * head_dim * esz, 256);
    bytes += round_up(rope_table_bytes(T, head_dim), 256);
  }
  return bytes;
}

// Pooled K and V the compressed bf16 prefill builds itself (block > 0,
// pooled_k = pooled_v = NULL), after the plan.
static size_t prefill_pooled_bytes(int batch, int T, int n_kv_heads, int head_dim, int block) {
  return block > 0 ? 2 * round_up(size_t(batch) * (T / block) * n_kv_heads * head_dim * 2, 256) : 0;
}

size_t nd_swa_sink_prefill_workspace_size(nd_dtype dtype, int batch, int T, int n_q_heads,
                                          int n_kv_heads, int head_dim, float rope_theta,
                                          int block) {
  if (batch <= 0 || T <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0) return 0;
  size_t bytes = prefill_rotation_bytes(dtype, batch, T, n_q_heads, n_kv_heads, head_dim, rope_theta);
  if (dtype == ND_F32) bytes += prefill_f32_partial_bytes(batch, T, n_q_heads, head_dim);
  if (dtype == ND_BF16)
    bytes += round_up(prefill_plan_bytes(batch, T, block), 256) +
             prefill_pooled_bytes(batch, T, n_kv_heads, head_dim, block);
  return bytes;
}

int nd_swa_sink_prefill_tiles(const void *workspace, int batch, int T, int n_q_heads, int n_kv_heads,
                              int head_dim, float rope_theta, int block, long long *tiles_out) {
  if (!tiles_out || batch < 0 || T < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || block < 0)
    return ND_ERR_INVALID_ARG;
  if (n_q_heads % n_kv_heads || (head_dim != 64 && head_dim != 128)) return ND_ERR_INVALID_ARG;
  *tiles_out = 0;
  if (size_t(batch) * T == 0) return ND_OK;
  if (!workspace || !aligned16(workspace)) return ND_ERR_WORKSPACE;
  int st = check_device(nullptr);
  if (st != ND_OK) return st;
  PrefillArgs a = {};
  a.dtype = ND_BF16;
  a.batch = batch;
  a.T = T;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.d = head_dim;
  a.block = block;
  const size_t off = prefill_rotation_bytes(ND_BF16, batch, T, n_q_heads, n_kv_heads, head_dim, rope_theta);
  long long n = 0;
  cudaError_t e = prefill_tile_count(a, static_cast<const char *>(workspace) + off, &n);
  if (e != cudaSuccess) return fail_cuda(e);
  *tiles_out = n;
  return ND_OK;
}

static int prefill_impl(const void *q, const void *k, const void *v, nd_dtype dtype, int batch, int T,
                        int n_q_heads, int n_kv_heads, int head_dim, const int32_t *seg_ids,
                        const uint8_t *sink, int window, float rope_theta, const void *pooled_k,
                        const void *pooled_v, int block, int n_pinned, void *out, float *lse,
                        void *workspace, size_t workspace_bytes, nd_stream_t stream) {
  if (dtype != ND_F32 && dtype != ND_BF16) return ND_ERR_INVALID_ARG;
  if (batch < 0 || T < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || window < 0 || block < 0)
    return ND_ERR_INVALID_ARG;
  if (n_q_heads % n_kv_heads) return ND_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128)
    return head_dim > 0 && head_dim % 2 == 0 ? ND_ERR_UNSUPPORTED : ND_ERR_INVALID_ARG;
  if (size_t(batch) * T == 0) return ND_OK;
  if (!q || !k || !v || !out) return ND_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ND_ERR_INVALID_ARG;
  const bool pool_inside = block > 0 && !pooled_k && !pooled_v;
  if (block > 0) {
    if (dtype != ND_BF16) return ND_ERR_UNSUPPORTED;
    if (seg_ids || sink || window < 1) return ND_ERR_INVALID_ARG;
    if (!pool_inside && (!pooled_k || !pooled_v || !aligned16(pooled_k) || !aligned16(pooled_v)))
      return ND_ERR_INVALID_ARG;
  }
  const size_t need = nd_swa_sink_prefill_workspace_size(dtype, batch, T, n_q_heads, n_kv_heads,
                                                         head_dim, rope_theta, block);
  if (need && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return ND_ERR_WORKSPACE;
  int st = check_device(nullptr);
  if (st != ND_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  PrefillArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.dtype = dtype;
  a.batch = batch;
  a.T = T;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.d = head_dim;
  a.seg_ids = seg_ids;
  a.sink = sink;
  a.window = window;
  a.pooled_k = block > 0 ? pooled_k : nullptr;
  a.pooled_v = block > 0 ? pooled_v : nullptr;
  a.block = block;
  a.out = out;
  a.lse = lse;
  a.n_pinned = n_pinned;

  char *ws = static_cast<char *>(workspace);
  const size_t esz = dtype == ND_F32 ? 4 : 2;
  const bool f32 = dtype == ND_F32;
  void *qr = nullptr, *kr = nullptr, *table = nullptr;
  if (rope_theta != 0.f) {
    if (f32) {  // the bf16 kernel rotates q as it stages it
      qr = ws;
      ws += round_up(size_t(batch) * T * n_q_heads * head_dim * esz, 256);
    }
    kr = ws;
    ws += round_up(size_t(batch) * T * n_kv_heads * head_dim * esz, 256);
    table = ws;
    ws += round_up(rope_table_bytes(T, head_dim), 256);
  }
  // bf16: the tile records and plan go first (an ordinary launch), the
  // rotation table beside them, then K's rotation (fused with the pooling
  // when the call pools) and the attention kernel, each a dependent launch
  // that waits for the kernel before it
  cudaError_t e = cudaSuccess;
  if (!f32) e = launch_prefill_tc_prep(a, ws, s);
  if (e == cudaSuccess && pool_inside) {
    char *pooled = ws + round_up(prefill_plan_bytes(batch, T, block), 256);
    const size_t pb = prefill_pooled_bytes(batch, T, n_kv_heads, head_dim, block) / 2;
    a.pooled_k = pooled;
    a.pooled_v = pooled + pb;
    e = launch_pool_rope(k, v, kr, pooled, pooled + pb, batch, T, n_kv_heads, head_dim, block, a.n_pinned,
                         rope_theta, table, /*chained=*/true, s);
    if (table) {
      a.k = kr;
      a.rope_cs = table;
    }
    if (e != cudaSuccess) return fail_cuda(e);
    return finish(launch_prefill_tc(a, ws, device_error_word(), s));
  }
  if (e == cudaSuccess && table) {
    e = launch_rope_qk(f32 ? q : nullptr, qr, f32 ? n_q_heads : 0, k, kr, n_kv_heads, batch, T, head_dim,
                       rope_theta, f32, table, /*chained=*/!f32, s);
    a.k = kr;
    if (f32) a.q = qr;
    else a.rope_cs = table;
  }
  if (e != cudaSuccess) return fail_cuda(e);
  if (f32)
    return finish(launch_prefill_f32(
        a, ws + prefill_rotation_bytes(dtype, batch, T, n_q_heads, n_kv_heads, head_dim, rope_theta), s));
  return finish(launch_prefill_tc(a, ws, device_error_word(), s));
}

// Chunked prefill workspace: gathered keys and values, segment ids, sink
// flags, the metadata snapshot, then the prefill's tile records and plan.
struct ChunkLayout {
  int R, Tk;
  size_t kk, vv, seg, sink, meta, plan, total;
};
static ChunkLayout chunk_layout(int batch, int chunk, int n_kv_heads, int head_dim, int sink_cap, int ring_cap,
                                int window) {
  ChunkLayout L;
  L.R = chunk_ring_rows(ring_cap, window);
  L.Tk = sink_cap + L.R + chunk;
  const size_t rows = size_t(batch) * L.Tk;
  L.kk = 0;
  L.vv = L.kk + round_up(rows * n_kv_heads * head_dim * 2, 256);
  L.seg = L.vv + round_up(rows * n_kv_heads * head_dim * 2, 256);
  L.sink = L.seg + round_up(rows * 4, 256);
  L.meta = L.sink + round_up(rows, 256);
  L.plan = L.meta + round_up(size_t(batch) * 16, 256);
  L.total = L.plan + round_up(prefill_plan_bytes(batch, L.Tk, 0), 256);
  return L;
}

size_t nd_swa_sink_chunk_prefill_workspace_size(int batch, int chunk, int n_q_heads, int n_kv_heads,
                                                int head_dim, int sink_cap, int ring_cap, int window) {
  if (batch <= 0 || chunk <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || sink_cap < 0 ||
      ring_cap <= 0 || window < 1)
    return 0;
  return chunk_layout(batch, chunk, n_kv_heads, head_dim, sink_cap, ring_cap, window).total;
}

int nd_swa_sink_chunk_prefill(const void *q, const void *k, const void *v, int chunk, const nd_kv_cache *cache,
                              int n_q_heads, int window, void *out, float *lse, void *workspace,
                              size_t workspace_bytes, nd_stream_t stream) {
  int st = validate_cache(cache);
  if (st != ND_OK) return st;
  if (chunk < 0 || window < 1 || n_q_heads <= 0 || n_q_heads % cache->n_kv_heads || cache->ring_cap <= 0)
    return ND_ERR_INVALID_ARG;
  if (cache->head_dim != 64 && cache->head_dim != 128) return ND_ERR_UNSUPPORTED;
  if (cache->batch == 0 || chunk == 0) return ND_OK;
  if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return ND_ERR_INVALID_ARG;
  const int B = cache->batch, d = cache->head_dim;
  const ChunkLayout L = chunk_layout(B, chunk, cache->n_kv_heads, d, cache->sink_cap, cache->ring_cap, window);
  if (!workspace || workspace_bytes < L.total || !aligned16(workspace)) return ND_ERR_WORKSPACE;
  if ((st = check_device(nullptr)) != ND_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int *err = device_error_word();
  char *ws = static_cast<char *>(workspace);
  int32_t *meta = reinterpret_cast<int32_t *>(ws + L.meta);
  cudaError_t e = launch_chunk_gather(*cache, k, v, chunk, window, ws + L.kk, ws + L.vv,
                                     reinterpret_cast<int32_t *>(ws + L.seg), reinterpret_cast<uint8_t *>(ws + L.sink),
                                     meta, err, s);
  if (e != cudaSuccess) return fail_cuda(e);
  PrefillArgs a;
  a.q = q;
  a.k = ws + L.kk;
  a.v = ws + L.vv;
  a.dtype = ND_BF16;
  a.batch = B;
  a.T = L.Tk;
  a.Hq = n_q_heads;
  a.Hkv = cache->n_kv_heads;
  a.d = d;
  a.seg_ids = reinterpret_cast<const int32_t *>(ws + L.seg);
  a.sink = reinterpret_cast<const uint8_t *>(ws + L.sink);
  a.window = window;
  a.pooled_k = a.pooled_v = nullptr;
  a.block = 0;
  a.out = out;
  a.lse = lse;
  a.q_off = cache->sink_cap + L.R;
  e = launch_prefill_tc_prep(a, ws + L.plan, s);
  if (e == cudaSuccess) e = launch_prefill_tc(a, ws + L.plan, err, s);
  if (e == cudaSuccess) e = launch_chunk_append(*cache, k, v, chunk, meta, s);
  return finish(e);
}

int nd_swa_sink_chunk_prefill_tiles(const void *workspace, int batch, int chunk, int n_q_heads, int n_kv_heads,
                                    int head_dim, int sink_cap, int ring_cap, int window, long long *tiles_out) {
  if (!tiles_out || batch < 0 || chunk < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || sink_cap < 0 ||
      ring_cap <= 0 || window < 1 || n_q_heads % n_kv_heads || (head_dim != 64 && head_dim != 128))
    return ND_ERR_INVALID_ARG;
  *tiles_out = 0;
  if (size_t(batch) * chunk == 0) return ND_OK;
  if (!workspace || !aligned16(workspace)) return ND_ERR_WORKSPACE;
  int st = check_device(nullptr);
  if (st != ND_OK) return st;
  const ChunkLayout L = chunk_layout(batch, chunk, n_kv_heads, head_dim, sink_cap, ring_cap, window);
  PrefillArgs a = {};
  a.dtype = ND_BF16;
  a.batch = batch;
  a.T = L.Tk;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.d = head_dim;
  a.q_off = sink_cap + L.R;
  long long n = 0;
  cudaError_t e = prefill_tile_count(a, static_cast<const char *>(workspace) + L.plan, &n);
  if (e != cudaSuccess) return fail_cuda(e);
  *tiles_out = n;
  return ND_OK;
}

int nd_set_prefill_epilogue_wait_limit(unsigned polls) {
  int st = check_device(nullptr);
  if (st != ND_OK) return st;
  return finish(set_epilogue_wait_limit(polls));
}

int nd_swa_sink_prefill(const void *q, const void *k, const void *v, nd_dtype dtype, int batch,
                        int T, int n_q_heads, int n_kv_heads, int head_dim,
                        const int32_t *seg_ids, const uint8_t *sink, int window, float rope_theta,
                        const void *pooled_k, const void *pooled_v, int block, void *out,
                        float *lse, void *workspace, size_t workspace_bytes, nd_stream_t stream) {
  return prefill_impl(q, k, v, dtype, batch, T, n_q_heads, n_kv_heads, head_dim, seg_ids, sink, window, rope_theta,
                      pooled_k, pooled_v, block, 0, out, lse, workspace, workspace_bytes, stream);
}

size_t nd_compressed_prefill_workspace_size(int batch, int T, int n_q_heads, int n_kv_heads, int head_dim,
                                            float rope_theta, int block) {
  if (block <= 0) return 0;
  return nd_swa_sink_prefill_workspace_size(ND_BF16, batch, T, n_q_heads, n_kv_heads, head_dim, rope_theta, block);
}

int nd_compressed_prefill(const void *q, const void *k, const void *v, int batch, int T, int n_q_heads,
                          int n_kv_heads, int head_dim, int window, int block, int n_pinned, float rope_theta,
                          void *out, float *lse, void *workspace, size_t workspace_bytes, nd_stream_t stream) {
  if (block < 1 || window < 1 || n_pinned < 0 || (T >= 0 && n_pinned > T)) return ND_ERR_INVALID_ARG;
  return prefill_impl(q, k, v, ND_BF16, batch, T, n_q_heads, n_kv_heads, head_dim, nullptr, nullptr, window,
                      rope_theta, nullptr, nullptr, block, n_pinned, out, lse, workspace, workspace_bytes, stream);
}

int nd_rope_apply(const void *x, void *y, int batch, int T, int n_heads, int head_dim,
                  float rope_theta, nd_stream_t stream) {
  if (batch < 0 || T < 0 || n_heads <= 0 || head_dim <= 0 || head_dim % 2) return ND_ERR_INVALID_ARG;
  if (head_dim > 256) return ND_ERR_UNSUPPORTED;
  if (size_t(batch) * T == 0) return ND_OK;
  if (!x || !y) return ND_ERR_INVALID_ARG;
  int st = check_device(nullptr);
  if (st != ND_OK) return st;
  return finish(launch_rope(x, y, batch, T, n_heads, head_dim, rope_theta,
                            reinterpret_cast<cudaStream_t>(stream)));
}

int nd_kv_compress_pool(const void *k, const void *v, int batch, int T, int n_heads, int head_dim,
                        int block, float rope_theta, void *pooled_k, void *pooled_v,
                        nd_stream_t stream) {
  if (batch < 0 || T < 0 || n_heads <= 0 || head_dim <= 0 || head_dim % 2 || block <= 0)
    return ND_ERR_INVALID_ARG;
  if (head_dim > 256) return ND_ERR_UNSUPPORTED;
  if (size_t(batch) * (T / block) == 0) return ND_OK;
  if (!k || !v || !pooled_k || !pooled_v) return ND_ERR_INVALID_ARG;
  int st = check_device(nullptr);
  if (st != ND_OK) return st;
  return finish(launch_compress_pool(k, v, batch, T, n_heads, head_dim, block, rope_theta, pooled_k,
                                     pooled_v, reinterpret_cast<cudaStream_t>(stream)));
}

size_t nd_kv_compress_pool_rope_workspace_size(int T, int head_dim, float rope_theta) {
  if (T <= 0 || head_dim <= 0 || rope_theta == 0.f) return 0;
  return round_up(rope_table_bytes(T, head_dim), 256);
}

int nd_kv_compress_pool_rope(const void *k, const void *v, int batch, int T, int n_heads, int head_dim, int block,
                             float rope_theta, void *k_rot, void *pooled_k, void *pooled_v, void *workspace,
                             size_t workspace_bytes, nd_stream_t stream) {
  if (batch < 0 || T < 0 || n_heads <= 0 || block <= 0) return ND_ERR_INVALID_ARG;
  if (head_dim <= 0 || head_dim % 16 || head_dim > 256)
    return head_dim > 0 && head_dim % 2 == 0 ? ND_ERR_UNSUPPORTED : ND_ERR_INVALID_ARG;
  if (size_t(batch) * T == 0) return ND_OK;
  const bool blocks = T / block > 0;  // pooled outputs are written only when there is a whole block
  if (!k || !v || (blocks && (!pooled_k || !pooled_v)) || (rope_theta != 0.f && !k_rot)) return ND_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || (blocks && (!aligned16(pooled_k) || !aligned16(pooled_v))) ||
      (k_rot && !aligned16(k_rot)))
    return ND_ERR_INVALID_ARG;
  const size_t need = nd_kv_compress_pool_rope_workspace_size(T, head_dim, rope_theta);
  if (need && (!workspace || workspace_bytes < need || !aligned16(workspace))) return ND_ERR_WORKSPACE;
  int st = check_device(nullptr);
  if (st != ND_OK) return st;
  return finish(launch_pool_rope(k, v, k_rot, pooled_k, pooled_v, batch, T, n_heads, head_dim, block, 0,
                                 rope_theta, workspace, /*chained=*/false, reinterpret_cast<cudaStream_t>(stream)));
}

int nd_kv_budget_window(const nd_model_cfg *cfg, int *budget_out, int *effective_out) {
  if (!cfg || !budget_out) return ND_ERR_INVALID_ARG;
  if (cfg->num_heads <= 0 || cfg->d_model < 0 || cfg->attn_dim < 0 || cfg->num_kv_heads < 0 ||
      cfg->num_layers < 0 || cfg->n_engram_sites < 0 || cfg->max_seq_len < 0 || cfg->kv_window < 0)
    return ND_ERR_INVALID_ARG;
  const int64_t kBudgetBytes = 11LL * 1024 * 1024 + 512LL * 1024;
  const int64_t kGroup = 32, kMin = 160;
  const int64_t head_dim = int64_t(cfg->attn_dim ? cfg->attn_dim : cfg->d_model) / cfg->num_heads;
  const int64_t kv = int64_t(cfg->num_kv_heads) * head_dim;
  const int64_t per_pos = int64_t(cfg->num_layers) * (2 * kv + 2 * (kv / kGroup) * 4) +
                          int64_t(cfg->n_engram_sites) * (cfg->d_model + kGroup * 4);
  if (per_pos <= 0) return ND_ERR_INVALID_ARG;
  int64_t w = (kBudgetBytes / per_pos) / kGroup * kGroup;
  if (w > cfg->max_seq_len) w = cfg->max_seq_len;
  if (w < kMin) w = kMin;
  *budget_out = int(w);
  if (effective_out)
    *effective_out = cfg->kv_window ? int(w < cfg->kv_window ? w : cfg->kv_window) : int(w);
  return ND_OK;
}

}  // extern "C"
