// nd_internal.h -- launch functions behind the C ABI (host side, C++).
// nd_api.cu validates arguments and then calls these; each enqueues kernels on
// `stream` and returns the CUDA error of its launches.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "nd.h"

namespace nd {

// Address of the current device's error word (see nd_device_errors()).
int *device_error_word();

// Records `e` as the calling thread's last CUDA error; returns ND_ERR_CUDA.
int fail_cuda(cudaError_t e);
// ND_OK if the current device is an sm_103 part, else ND_ERR_UNSUPPORTED (or
// ND_ERR_CUDA when the device query fails).
int check_device(int *dev_out);
// The argument checks of nd_swa_sink_decode (cache, heads, window, q, out),
// in its order; ND_OK also for an empty batch.
int validate_decode(const void *q, const nd_kv_cache *cache, int n_q_heads, int window, const void *out);

cudaError_t launch_kv_append_quant(const nd_kv_cache &c, const void *k_new, const void *v_new,
                                   int to_sink, int *err, cudaStream_t stream);

// Prefill -> cache handoff (nd_kv_cache_from_prefill): a planning kernel
// (one CTA per cache row) writes each row's kept tokens to `plan`
// (kv_fill_plan_ints ints per row), then a quantising kernel; dependent
// launches.
size_t kv_fill_plan_ints(int sink_cap, int ring_cap);
cudaError_t launch_kv_fill(const nd_kv_cache &c, const void *k, const void *v, int batch, int T,
                           const int32_t *seg_ids, const uint8_t *sink, const int32_t *src_row,
                           const int32_t *src_seg, int32_t *plan, int *err, cudaStream_t stream);

cudaError_t launch_kv_quant_rows(const void *x, int64_t n_rows, int head_dim, int8_t *codes,
                                 float *scales, cudaStream_t stream);

struct DecodePlan {
  int n_split;        // CTAs per (sequence, kv head)
  int slots_per_cta;  // multiple of 16
  int max_slots;      // upper bound of visible slots per sequence
};
DecodePlan plan_decode(int batch, int n_kv_heads, int max_slots, int head_dim);
size_t decode_workspace_bytes(int batch, int n_q_heads, int head_dim, int max_slots,
                              int n_kv_heads_hint);
// k_new / v_new non-NULL: fused step (ring append of the current token, then
// attention with it) in one clustered launch; cudaErrorInvalidConfiguration
// when the sequence's CTAs make a cluster larger than the fused step uses
// (decode_step_fuses() says which; the caller then appends and decodes in two
// launches).
cudaError_t launch_decode(const void *q, const nd_kv_cache &c, int n_q_heads, int window,
                          void *out, float *lse, void *ws, size_t ws_bytes, int *err,
                          cudaStream_t stream, const void *k_new = nullptr,
                          const void *v_new = nullptr);
bool decode_step_fuses(int batch, int n_kv_heads, int max_slots, int head_dim);

// Per sequence: rotate q into q_rot, append the token to the compressed
// cache (pinned slot or ring, block sums, a pooled slot when the token closes
// its block) and advance the metadata; a dependent launch.
cudaError_t launch_compressed_append(const nd_kv_cache &c, float *k_sum, float *v_sum, int block, int n_pinned,
                                     int window, const void *q, int Hq, const void *k_new, const void *v_new,
                                     void *q_rot, float theta, int *err, cudaStream_t stream);

// Chunked prefill against the cache: ring rows of the gathered key layout,
// the gather (cache -> bf16 keys / values, segment ids, sink flags, and a
// metadata snapshot [B][4]) and the chunk's ring append from that snapshot;
// dependent launches.
int chunk_ring_rows(int ring_cap, int window);
cudaError_t launch_chunk_gather(const nd_kv_cache &c, const void *k, const void *v, int Tc, int window, void *kk,
                                void *vv, int32_t *seg, uint8_t *sink, int32_t *meta, int *err, cudaStream_t stream);
cudaError_t launch_chunk_append(const nd_kv_cache &c, const void *k, const void *v, int Tc, const int32_t *meta,
                                cudaStream_t stream);

cudaError_t launch_rope(const void *x, void *y, int batch, int T, int n_heads, int head_dim,
                        float theta, cudaStream_t stream);

// Launch with programmatic stream serialization allowed: the kernel may be
// scheduled while the previous one on the stream runs, and must call
// pdl_wait() (nd_common.cuh) before it touches memory that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// theta^(-2i/head_dim) for i < head_dim/2, in double (head_dim <= 256).
constexpr int kMaxHalf = 128;
struct Freqs {
  double f[kMaxHalf];
};
Freqs make_freqs(int head_dim, float theta);

size_t rope_table_bytes(int T, int head_dim);
// Builds the (cos, sin) table of positions 0..T-1 into `table` (float2
// [T][head_dim/2]) and rotates q (Hq heads; q may be NULL with Hq = 0) and k.
// chained: the previous kernel on the stream is an ordinary launch of the
// same call that does not touch `table`; the table kernel then runs beside it
// and waits for it only before it exits (so its completion still implies that
// kernel's).  Otherwise the table kernel waits before it starts.
cudaError_t launch_rope_qk(const void *q, void *q_out, int Hq, const void *k, void *k_out, int Hkv,
                           int batch, int T, int head_dim, float theta, bool f32, void *table,
                           bool chained, cudaStream_t stream);

// The compressed prefill's fused pass: the angle table (theta != 0) into
// `table`, then one read of K and V writing K rotated at every position
// (k_rot; nothing when theta == 0) and the pooled blocks of positions pos0..
// ((T - pos0) / block of them, pooled K rotated at the midpoint).  chained as
// in launch_rope_qk.
cudaError_t launch_pool_rope(const void *k, const void *v, void *k_rot, void *pk, void *pv, int batch, int T,
                             int n_heads, int head_dim, int block, int pos0, float theta, void *table, bool chained,
                             cudaStream_t stream);

cudaError_t launch_compress_pool(const void *k, const void *v, int batch, int T, int n_heads,
                                 int head_dim, int block, float theta, void *pk, void *pv,
                                 cudaStream_t stream);

struct PrefillArgs {
  const void *q, *k, *v;  // after rotation, if any
  nd_dtype dtype;
  int batch, T, Hq, Hkv, d;
  const int32_t *seg_ids;  // may be NULL
  const uint8_t *sink;     // may be NULL
  int window;
  const void *pooled_k, *pooled_v;  // may be NULL
  int block;                        // 0 = no pooled columns
  void *out;
  float *lse;  // may be NULL
  // bf16 path: (cos, sin) table float2 [T][d/2] of the rotation; q is then
  // rotated inside the attention kernel (k arrives rotated).  NULL: q as is.
  const void *rope_cs = nullptr;
  // bf16 path: queries are key rows q_off .. T-1 (q, out and lse hold
  // T - q_off rows); 0 for an ordinary prefill
  int q_off = 0;
  // compressed variant: keys 0 .. n_pinned-1 pinned, pooled blocks tile the
  // positions after them ((T - n_pinned) / block of them)
  int n_pinned = 0;
};

size_t prefill_plan_bytes(int batch, int T, int block);
// fp32 prefill; small problems split their keys over several CTAs and merge
// the partial states in `partials` (prefill_f32_partial_bytes; 0 bytes and
// NULL otherwise)
size_t prefill_f32_partial_bytes(int batch, int T, int n_q_heads, int head_dim);
cudaError_t launch_prefill_f32(const PrefillArgs &a, void *partials, cudaStream_t stream);
// The tensor-core path in two launches: the tile records and plan (an
// ordinary launch, first of the call), then the attention kernel (a dependent
// launch: it waits for the kernel before it, which may be the rotation pass).
cudaError_t launch_prefill_tc_prep(const PrefillArgs &a, void *plan_ws, cudaStream_t stream);
cudaError_t launch_prefill_tc(const PrefillArgs &a, void *plan_ws, int *err, cudaStream_t stream);
// Poll limit of the tensor-core prefill epilogue's wait for a block's last
// PV on the current device (0 = the default bound); synchronous.
cudaError_t set_epilogue_wait_limit(unsigned polls);
// Products of a 128-row block with a 64-key tile that the attention kernel
// performs for the plan in plan_ws (synchronous read of the plan's counts).
cudaError_t prefill_tile_count(const PrefillArgs &a, const void *plan_ws, long long *tiles);

}  // namespace nd
