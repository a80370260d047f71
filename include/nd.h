/*
 * nd.h -- C ABI of libnd: sliding-window + KV-sink attention over a bounded
 * int8 group-32 KV cache, and the compressed-attention variant, for one
 * NVIDIA GB300 (sm_103a).
 *
 * The operations follow these web pages (cited by title and section):
 *  [N1] "256-token滑动窗口+KV sink：Needle 2工具钉住机制源码分析"
 *  [N2] "How the 256-Token Sliding Window Works with Tools as KV Sinks in Needle"
 *  [C3] "Compressed attention and the copy probe"
 *
 * Conventions for every entry point:
 *  - Tensor arguments are DEVICE pointers owned by the caller, contiguous,
 *    row-major, in the layout stated beside each argument.  bf16 tensors are
 *    passed as void* holding IEEE bfloat16 values.  Pointers must be 16-byte
 *    aligned.  The library keeps no pointer after a call returns.
 *  - Work is enqueued on the caller's stream (NULL = the legacy default
 *    stream) and runs asynchronously; the call returns once it is enqueued.
 *  - No entry point allocates device or host memory.  Scratch comes from a
 *    caller buffer sized by the matching *_workspace_size() query.
 *  - Every entry point returns an nd_status.  Argument errors are detected on
 *    the host before anything is enqueued and leave all buffers untouched.
 *    ND_ERR_CUDA means a launch failed; nd_last_cuda_error() returns the CUDA
 *    error code of the failing call on the calling thread.
 *  - No exception crosses the ABI.  The library is thread-safe as long as
 *    concurrent calls do not share output or workspace buffers.
 *  - Most kernels are programmatic dependent launches (each waits for the
 *    kernel before it on the stream, the caller's included, before it reads
 *    memory), and some let the next kernel on the stream be scheduled before
 *    they finish.  Ordinary
 *    launches, copies and events after a call see all of its results; a
 *    caller kernel launched with programmatic stream serialization must wait
 *    for its prerequisite grid (griddepcontrol.wait) before it reads them.
 */
#ifndef ND_H_
#define ND_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ND_API __attribute__((visibility("default")))
#else
#define ND_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA runtime header. */
typedef struct CUstream_st *nd_stream_t;

typedef enum {
  ND_OK = 0,
  ND_ERR_INVALID_ARG = 1,  /* a size, pointer, alignment or layout is invalid */
  ND_ERR_UNSUPPORTED = 2,  /* valid but not built: head_dim, dtype, device    */
  ND_ERR_CUDA = 3,         /* a CUDA launch failed; see nd_last_cuda_error()  */
  ND_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required      */
  ND_ERR_DEVICE = 5        /* a kernel reported a device-side error flag      */
} nd_status;

typedef enum { ND_F32 = 0, ND_BF16 = 1 } nd_dtype;

/* Library version string, e.g. "nd 0.1.0 sm_103a". */
ND_API const char *nd_version(void);

/* Human-readable name of a status code (never NULL). */
ND_API const char *nd_status_string(int status);

/* CUDA error code (cudaError_t as int) of the last failing CUDA call made by
 * this library on the calling thread; 0 if none. */
ND_API int nd_last_cuda_error(void);

/*
 * Device-side error word.  Kernels that wait on memory barriers give up after
 * a bounded number of polls and OR a flag into this word instead of hanging;
 * launches that read cache metadata flag out-of-range values the same way.
 * Reads (and, when clear != 0, resets) the word of the current device.  Blocks
 * until the device is idle.  Flags: 1 = a barrier wait timed out,
 * 2 = cache metadata out of range (the affected sequence was skipped).
 */
ND_API int nd_device_errors(int *flags_out, int clear);

/*
 * Failure-path hook for tests: the bf16 prefill's attention kernel waits
 * for each row block's last P*V before its epilogue reads the output; that
 * wait guards no copy in flight.  With polls > 0 the epilogue instead polls,
 * `polls` times without blocking, a barrier that nothing arrives on, so the
 * wait runs out on every CTA and raises device flag 1: the kernel then stops
 * issuing work, lets what is in flight land, frees its tensor memory and
 * exits, and the call's output is undefined.  0 restores the ordinary
 * bounded wait.  Applies to the current device from the next launch on;
 * blocks until earlier work on the legacy default stream is done.
 */
ND_API int nd_set_prefill_epilogue_wait_limit(unsigned polls);

/* ------------------------------------------------------------------------ */
/* Bounded KV cache                                                          */
/* ------------------------------------------------------------------------ */

/*
 * The bounded cache of [N1] "KV sink 如何「钉住」工具" and [N2] "KV Sinks for
 * Tools": pinned sink positions that are never evicted plus a ring holding the
 * most recent positions.  Storage is the int8 layout implied by the per-position
 * byte count of kv_budget_window ([N2] "Effective KV Window"): per token, per KV
 * head, head_dim int8 codes and one fp32 scale per 32 contiguous channels, for
 * K and for V.
 *
 *   k_codes, v_codes  int8  [batch][n_kv_heads][sink_cap + ring_cap][head_dim]
 *   k_scale, v_scale  fp32  [batch][n_kv_heads][sink_cap + ring_cap][head_dim/32]
 *   slot s <  sink_cap : sink slot s (the pinned prefix, position s)
 *   slot sink_cap + r  : ring slot r
 *   sink_len   int32 [batch]  valid sink slots
 *   ring_start int32 [batch]  ring slot of the oldest ring entry
 *   ring_len   int32 [batch]  valid ring entries (<= ring_cap)
 *   seq_len    int32 [batch]  tokens seen; the newest token has position
 *                             seq_len - 1 and the ring's entries, oldest
 *                             first, hold the ring_len positions ending there
 * All pointers are device pointers; the metadata lives on the device so a
 * decode loop can run without host synchronisation (and inside CUDA graphs).
 * head_dim must be a multiple of 32; the kernels are built for 64 and 128.
 */
typedef struct {
  int batch, n_kv_heads, head_dim, sink_cap, ring_cap;
  int8_t *k_codes;
  int8_t *v_codes;
  float *k_scale;
  float *v_scale;
  int32_t *sink_len;
  int32_t *ring_start;
  int32_t *ring_len;
  int32_t *seq_len;
} nd_kv_cache;

/*
 * Quantise one new bf16 token per sequence and append it to the cache
 * (fused quantise-and-append).
 *   k_new, v_new  bf16 [batch][n_kv_heads][head_dim]
 *   to_sink = 0   ring append: slot (ring_start + ring_len) mod ring_cap, or,
 *                 when the ring is full, the oldest slot (ring_start advances)
 *   to_sink = 1   sink append: slot sink_len; accepted only while ring_len == 0
 *                 and sink_len < sink_cap (the sink is a prefix).  A rejected
 *                 sink append writes nothing for that sequence and sets
 *                 device error flag 2.
 * Codec (one group = 32 contiguous channels of one token and head):
 *   amax = max |x|, scale = amax / 127 (fp32 IEEE divide),
 *   code = clamp(rint(x / scale), -127, 127) (fp32 IEEE divide, ties to even);
 *   amax == 0 gives scale 0 and zero codes.
 * seq_len advances by one for every accepted append.
 */
ND_API int nd_kv_append_quant(const nd_kv_cache *cache, const void *k_new,
                       const void *v_new, int to_sink, nd_stream_t stream);

/*
 * Bulk form of the same codec: quantise n_rows bf16 rows of head_dim channels.
 *   x       bf16 [n_rows][head_dim]
 *   codes   int8 [n_rows][head_dim]
 *   scales  fp32 [n_rows][head_dim/32]
 * Used to fill cache slots in bulk (for example after a prefill).
 */
ND_API int nd_kv_quant_rows(const void *x, int64_t n_rows, int head_dim,
                     int8_t *codes, float *scales, nd_stream_t stream);

/*
 * Prefill -> cache handoff: fills cache rows from the keys and values a
 * prefill computed, so decoding can continue after a packed prefill.  The
 * bounded cache of [N2] "KV Sinks for Tools" / [N1] "KV sink 如何「钉住」工具"
 * keeps a segment's pinned sink prefix and only its most recent positions;
 * cache row e receives the tokens of segment src_seg[e] of batch row
 * src_row[e] exactly as appending them one at a time, in position order, to
 * an empty cache row would (nd_kv_append_quant with to_sink = sink[b][t]):
 *   - while the ring is empty, a sink token goes to the next sink slot
 *     (rejected once sink_cap slots are used);
 *   - every other token goes to the ring, which keeps the newest ring_cap;
 *   - once the ring holds a token, sink tokens are rejected.
 * The row's codes, scales and metadata (sink_len, ring_start, ring_len,
 * seq_len) are then those of that sequence of appends; its other slots keep
 * whatever they held (they are not visible).  A rejected sink token is
 * dropped (not counted in seq_len) and sets device error flag 2.
 *   k, v     bf16 [batch][T][n_kv_heads][head_dim]: the keys as the decode
 *            will read them (already rotated, if the model rotates keys) and
 *            the values; n_kv_heads and head_dim are the cache's
 *   seg_ids  int32 [batch][T], or NULL (every position in one segment)
 *   sink     uint8 [batch][T], or NULL (no sink tokens)
 *   src_row, src_seg  int32 [cache->batch] device arrays; src_seg may be NULL
 *            when seg_ids is.  src_row[e] < 0 leaves cache row e untouched;
 *            src_row[e] >= batch or src_seg[e] <= 0 (padding) sets device
 *            error flag 2 and leaves it untouched.
 * Requires ring_cap > 0; head_dim 32, 64, 128 or 256.  The kept tokens'
 * plan lives in `workspace` (device, 16-byte aligned) of
 * nd_kv_cache_from_prefill_workspace_size(cache->batch, sink_cap, ring_cap)
 * bytes, else ND_ERR_WORKSPACE.
 */
ND_API size_t nd_kv_cache_from_prefill_workspace_size(int cache_batch, int sink_cap, int ring_cap);
ND_API int nd_kv_cache_from_prefill(const nd_kv_cache *cache, const void *k, const void *v,
                                    int batch, int T, const int32_t *seg_ids,
                                    const uint8_t *sink, const int32_t *src_row,
                                    const int32_t *src_seg, void *workspace,
                                    size_t workspace_bytes, nd_stream_t stream);

/*
 * One decode step ([N1] "256-token 滑动窗口：源码走读"): each sequence's query
 * sits at position seq_len - 1 and attends to every sink slot and to the ring
 * entries within `window` positions of it (recent = qpos - kpos < window; a
 * sink is kept at any distance).  The caller appends the current token before
 * calling, so the query sees its own key.  GQA: query head h reads KV head
 * h / (n_q_heads / n_kv_heads).  Softmax scale 1/sqrt(head_dim).
 *   q    bf16 [batch][n_q_heads][head_dim]  (already rotated, if the model
 *             uses a rotary embedding)
 *   out  bf16 [batch][n_q_heads][head_dim]
 *   lse  fp32 [batch][n_q_heads] natural-log softmax denominator, or NULL
 *   window >= 1.  n_q_heads / n_kv_heads must be 1..8.
 * A sequence with no visible key (empty cache) gets out = 0, lse = -inf.
 * Split-K partials go to the workspace, sized by
 * nd_swa_sink_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim,
 * sink_cap + ring_cap); the size may be 0 (no split).  The kernel walks every
 * physical slot of the cache and masks the ones the metadata marks invisible,
 * so its loads do not wait for the metadata.
 */
ND_API size_t nd_swa_sink_decode_workspace_size(int batch, int n_q_heads,
                                                int n_kv_heads, int head_dim,
                                                int max_slots);
ND_API int nd_swa_sink_decode(const void *q, const nd_kv_cache *cache, int n_q_heads,
                       int window, void *out, float *lse, void *workspace,
                       size_t workspace_bytes, nd_stream_t stream);

/*
 * One whole decode step: ring-append the current token (exactly as
 * nd_kv_append_quant with to_sink = 0) and attend with it (exactly as
 * nd_swa_sink_decode afterwards).  When a sequence's CTAs form a small
 * thread-block cluster (at most 4 of them: n_kv_heads x the split the decode
 * would use) both happen in one launch: the CTA that owns the new slot
 * quantises the token, writes it to the cache and uses it directly, and the
 * sequence's metadata is advanced after all of its CTAs have read it.
 * Otherwise the call makes the two launches itself.  Same arguments, layouts,
 * workspace and errors as the two calls; requires ring_cap > 0.
 *   k_new, v_new  bf16 [batch][n_kv_heads][head_dim]
 */
ND_API int nd_swa_sink_decode_step(const void *q, const nd_kv_cache *cache,
                                   const void *k_new, const void *v_new, int n_q_heads,
                                   int window, void *out, float *lse, void *workspace,
                                   size_t workspace_bytes, nd_stream_t stream);

/*
 * nd_swa_sink_decode_step with the step's inputs and outputs in host memory,
 * for a caller whose token and query live on the host: the call enqueues on
 * `stream` the step exactly as nd_swa_sink_decode_step, reading q, k_new and
 * v_new from the host and writing out (and lse, when lse_host is not NULL)
 * to it.  The host results are valid once the stream has passed the call
 * (synchronise the stream, or an event recorded after the call).
 * Page-locked, 16-byte aligned host buffers are read and written in place
 * by the step's kernels over the host link (no copies); other host memory
 * is staged in the workspace by one cudaMemcpyAsync per buffer each way
 * (synchronous for pageable memory).
 *   q_host, out_host        bf16 [batch][n_q_heads][head_dim], host memory
 *   k_new_host, v_new_host  bf16 [batch][n_kv_heads][head_dim], host memory
 *   lse_host                fp32 [batch][n_q_heads], host memory, or NULL
 * The device staging buffers and the decode's split scratch are carved from
 * `workspace` (device, 16-byte aligned), which must hold
 * nd_swa_sink_decode_step_host_workspace_size(batch, n_q_heads, n_kv_heads,
 * head_dim, sink_cap + ring_cap) bytes, else ND_ERR_WORKSPACE.  Other errors
 * as nd_swa_sink_decode_step; a NULL host pointer (lse_host excepted) is
 * ND_ERR_INVALID_ARG.
 */
ND_API size_t nd_swa_sink_decode_step_host_workspace_size(int batch, int n_q_heads,
                                                          int n_kv_heads, int head_dim,
                                                          int max_slots);
ND_API int nd_swa_sink_decode_step_host(const void *q_host, const nd_kv_cache *cache,
                                        const void *k_new_host, const void *v_new_host,
                                        int n_q_heads, int window, void *out_host,
                                        float *lse_host, void *workspace,
                                        size_t workspace_bytes, nd_stream_t stream);

/*
 * nd_swa_sink_decode_step_host with the step's host buffers packed (one
 * allocation each way: one page-locked lookup each, or one copy each for
 * memory that has to be staged):
 *   in_host   one host allocation holding, back to back,
 *             q     bf16 [batch][n_q_heads][head_dim],
 *             k_new bf16 [batch][n_kv_heads][head_dim],
 *             v_new bf16 [batch][n_kv_heads][head_dim]
 *   out_host  one host allocation holding out bf16 [batch][n_q_heads][head_dim]
 *             followed, when with_lse != 0, by lse fp32 [batch][n_q_heads]
 * (one allocation each: an access may not span two page-locked allocations
 * that merely sit next to each other).  Workspace, stream semantics and
 * errors as nd_swa_sink_decode_step_host; the workspace size is the same
 * query.
 */
ND_API int nd_swa_sink_decode_step_host_packed(const void *in_host, const nd_kv_cache *cache,
                                               int n_q_heads, int window, void *out_host,
                                               int with_lse, void *workspace,
                                               size_t workspace_bytes, nd_stream_t stream);

/*
 * nd_swa_sink_decode without a workspace argument.  The pages have no
 * counterpart: this is a library convenience for callers that cannot
 * allocate device memory -- a serving loop that must never call cudaMalloc
 * (it may synchronise the device and stall every stream), or a host runtime
 * that owns all device memory and passes a plugin only its inputs and
 * outputs.
 *
 * Computes exactly what nd_swa_sink_decode computes, with the same arguments
 * and results, and refuses what it refuses with the same status.  Its
 * split-K scratch is one fixed device array of ND_NOALLOC_SCRATCH_BYTES
 * (512 KiB) inside libnd, present on every device that loads the library
 * until the process exits.  The call allocates nothing and calls no
 * allocating routine.
 *  - Returns ND_ERR_WORKSPACE when the decode would need more scratch than
 *    ND_NOALLOC_SCRATCH_BYTES (nd_swa_sink_decode_workspace_size tells how
 *    much a shape needs); use nd_swa_sink_decode with a caller workspace then.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) and keeps it for later calls; make that first
 *    call before any stream capture on that device.  A failed lookup returns
 *    ND_ERR_CUDA (nd_last_cuda_error() has the code).  The kept address does
 *    not survive cudaDeviceReset: do not reset a device while the library is
 *    in use on it.
 *  - All calls on a device share the one array and each overwrites it, so
 *    calls whose kernels may overlap on the GPU (different streams without
 *    ordering between them) race; order them on one stream or use
 *    nd_swa_sink_decode with separate workspaces.
 */
#define ND_NOALLOC_SCRATCH_BYTES (512u << 10)
ND_API int nd_swa_sink_decode_noalloc(const void *q, const nd_kv_cache *cache,
                                      int n_q_heads, int window, void *out,
                                      float *lse, nd_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Compressed-attention decode                                               */
/* ------------------------------------------------------------------------ */

/*
 * The cache of compressed attention ([C3] "Two kinds of columns, pooled
 * blocks and exact recent keys", "Pool before rotating, not after"; priced
 * at inference in "So what happened ?": W exact positions plus one pooled
 * entry per block of `block` positions outside the window).  It is an
 * nd_kv_cache in the same int8 group-32 layout:
 *   sink slots [0, n_pinned)        pinned tokens 0 .. n_pinned-1, exact keys
 *                                   visible at any distance (the sink prefix
 *                                   of [N2] "KV Sinks for Tools"; 0 = the
 *                                   pages' compressed attention)
 *   sink slot n_pinned + j          pooled block j: positions
 *                                   n_pinned + j*block .. + block-1; key =
 *                                   mean of the unrotated keys rotated at
 *                                   n_pinned + j*block + block/2, value =
 *                                   mean of the values, each rounded to bf16
 *                                   and quantised with the cache codec
 *   ring (ring_cap >= window)       the exact keys (rotated at their
 *                                   positions) and values of the newest
 *                                   positions
 *   sink_len                        pinned tokens seen + pooled blocks
 *                                   visible to the newest query: block j is
 *                                   visible at query position p iff
 *                                   (j+1)*block <= p - window + 1 - n_pinned
 *   k_sum, v_sum  fp32 [batch][n_kv_heads][head_dim]: the running sums
 *                 (before rotation, in position order) of the block being
 *                 filled; nothing needs to be initialised
 * sink_cap must hold n_pinned + the number of blocks the sequence will
 * close; an empty cache has all four metadata arrays 0.
 */
typedef struct {
  nd_kv_cache kv;
  float *k_sum;
  float *v_sum;
  int block;     /* >= 1 */
  int n_pinned;  /* 0 .. kv.sink_cap */
} nd_compressed_cache;

/*
 * One decode step of compressed attention for every sequence: the token at
 * position p = seq_len (q, k_new, v_new before rotation, bf16) is appended --
 * pinned slot p while p < n_pinned, else the ring (nd_kv_append_quant's rule)
 * plus its block's sums, and when p is the last position of block j that
 * block is written to its pooled slot -- and the query, rotated at p, then
 * attends one softmax over [visible pooled blocks, pinned tokens, the ring
 * entries within `window` of p] (nd_swa_sink_decode on the cache).  With
 * n_pinned = 0 this is row p of the compressed attention of [C3], read from
 * int8 storage.  rope_theta 0 = no rotation.
 *   q        bf16 [batch][n_q_heads][head_dim]   (before rotation)
 *   k_new, v_new bf16 [batch][n_kv_heads][head_dim] (before rotation)
 *   out      bf16 [batch][n_q_heads][head_dim];  lse fp32 [batch][n_q_heads] or NULL
 * The rotated q and the decode's split scratch live in `workspace` (device,
 * 16-byte aligned) of nd_compressed_decode_step_workspace_size(batch,
 * n_q_heads, n_kv_heads, head_dim, sink_cap + ring_cap) bytes.  Requires
 * window >= 1, ring_cap >= window, head_dim 64 or 128, n_q_heads /
 * n_kv_heads 1..8.  A block that does not fit sink_cap, or a pinned token
 * beyond it, is not written and sets device error flag 2.
 */
ND_API size_t nd_compressed_decode_step_workspace_size(int batch, int n_q_heads, int n_kv_heads,
                                                       int head_dim, int max_slots);
ND_API int nd_compressed_decode_step(const void *q, const nd_compressed_cache *cache,
                                     const void *k_new, const void *v_new, int n_q_heads,
                                     int window, float rope_theta, void *out, float *lse,
                                     void *workspace, size_t workspace_bytes,
                                     nd_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Prefill                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * Prefill attention under make_causal_packing_mask ([N2] "KV Sinks for
 * Tools"): query t of row b attends key k iff
 *   seg_ids[b][t] == seg_ids[b][k] > 0 and k <= t and
 *   (window == 0 or t - k < window or sink[b][k] != 0)
 * (window == 0 switches the window term off; sink == NULL means no sinks).
 * GQA: query head h reads KV head h / (n_q_heads / n_kv_heads).  Softmax scale
 * 1/sqrt(head_dim).  Fully masked rows (padding, seg 0) get out = 0 and
 * lse = -inf.
 *
 *   q    [batch][T][n_q_heads][head_dim]    dtype
 *   k, v [batch][T][n_kv_heads][head_dim]   dtype
 *   seg_ids int32 [batch][T], or NULL (one segment, id 1)
 *   sink    uint8 [batch][T], or NULL
 *   out  [batch][T][n_q_heads][head_dim]    dtype
 *   lse  fp32 [batch][n_q_heads][T], or NULL
 *   rope_theta != 0 rotates q and k at their packed position t before the
 *     product (rotate-half pairs (i, i + head_dim/2), angle t*theta^(-2i/d)).
 *
 * Compressed variant ([C3] "Two kinds of columns" and "Pool before rotating,
 * not after"): when block > 0, pooled_k / pooled_v hold the T/block pooled
 * blocks from nd_kv_compress_pool ([batch][T/block][n_kv_heads][head_dim],
 * pooled K already rotated at its block midpoint) and every query attends
 * one softmax over the columns [pooled blocks j visible iff
 * (j+1)*block <= t - window + 1, exact keys k <= t with t - k < window].  The
 * compressed variant requires seg_ids == NULL, sink == NULL and window >= 1.
 * pooled_k and pooled_v may both be NULL: the call then pools K and V itself
 * (exactly as nd_kv_compress_pool, into its workspace) in one pass over K
 * and V that also rotates K (nd_kv_compress_pool_rope).
 *
 * dtype ND_F32 runs on CUDA cores in fp32; ND_BF16 runs on the tensor cores
 * (bf16 operands, fp32 accumulation).  head_dim 64 or 128.
 *
 * workspace: device memory of at least nd_swa_sink_prefill_workspace_size()
 * bytes, 16-byte aligned, owned by the caller and scratch between calls: the
 * rotated copies when rope_theta != 0 (q too on the fp32 path) and the angle
 * table; bf16: the tile records and tile plan (nd_swa_sink_prefill_tiles
 * reads the plan back), and the pooled blocks when the call pools; fp32
 * problems of at most 256 sixteen-row CTAs (batch x n_q_heads x
 * ceil(T / 16)): the partial softmax states of the four CTAs that share each
 * row tile's keys.  A size of 0 means no workspace is needed (NULL allowed).
 */
ND_API size_t nd_swa_sink_prefill_workspace_size(nd_dtype dtype, int batch, int T,
                                          int n_q_heads, int n_kv_heads,
                                          int head_dim, float rope_theta,
                                          int block);
ND_API int nd_swa_sink_prefill(const void *q, const void *k, const void *v,
                        nd_dtype dtype, int batch, int T, int n_q_heads,
                        int n_kv_heads, int head_dim, const int32_t *seg_ids,
                        const uint8_t *sink, int window, float rope_theta,
                        const void *pooled_k, const void *pooled_v, int block,
                        void *out, float *lse, void *workspace,
                        size_t workspace_bytes, nd_stream_t stream);

/*
 * Compressed-attention prefill with a pinned prefix (the compressed
 * attention of [C3] "Two kinds of columns" with the sink prefix of [N2]
 * "KV Sinks for Tools"; the library's reading, the same as
 * nd_compressed_decode_step's): keys 0 .. n_pinned-1 are exact keys visible
 * to every later query; the pooled blocks tile the positions after them
 * (block j = positions n_pinned + j*block .. + block-1, its key the mean of
 * the unrotated keys rotated at n_pinned + j*block + block/2) and are visible
 * to query t iff (j+1)*block <= t - window + 1 - n_pinned; the other keys are
 * exact within the window (t - k < window, k <= t).  n_pinned = 0 is
 * nd_swa_sink_prefill's compressed variant with pooled_k = pooled_v = NULL.
 * The call pools K and V itself (fused with K's rotation, into the
 * workspace).  q, k, v, out, lse as nd_swa_sink_prefill (bf16, before
 * rotation; rope_theta 0 = none); window >= 1, block >= 1,
 * 0 <= n_pinned <= T; head_dim 64 or 128.
 */
ND_API size_t nd_compressed_prefill_workspace_size(int batch, int T, int n_q_heads,
                                                   int n_kv_heads, int head_dim,
                                                   float rope_theta, int block);
ND_API int nd_compressed_prefill(const void *q, const void *k, const void *v, int batch, int T,
                                 int n_q_heads, int n_kv_heads, int head_dim, int window,
                                 int block, int n_pinned, float rope_theta, void *out,
                                 float *lse, void *workspace, size_t workspace_bytes,
                                 nd_stream_t stream);

/*
 * Chunked prefill against the bounded cache: a chunk of `chunk` new tokens
 * per sequence, at positions p0 .. p0+chunk-1 where p0 = seq_len, attends
 * under the decode mask of [N1] "256-token 滑动窗口：源码走读" (causal, and a
 * sink at any distance or qpos - kpos < window) to the cached sink and ring
 * entries and to the chunk's own keys -- the rows p0.. of a prefill over the
 * whole sequence, computed from the cache instead of the evicted prefix.
 * Then the chunk's tokens are ring-appended to the cache (exactly as `chunk`
 * calls of nd_kv_append_quant with to_sink = 0), so the next chunk or decode
 * step continues from it.
 *   q     bf16 [batch][chunk][n_q_heads][head_dim]  (rotated at their
 *   k, v  bf16 [batch][chunk][n_kv_heads][head_dim]  positions, if the model
 *                                                    rotates q and k)
 *   out   bf16 [batch][chunk][n_q_heads][head_dim]
 *   lse   fp32 [batch][n_q_heads][chunk], or NULL
 * The cached keys are dequantised (code * scale) and rounded to bf16 for the
 * tensor cores; the chunk's keys are used as given.  GQA as the prefill.
 * Requires window >= 1, ring_cap > 0, head_dim 64 or 128; the workspace
 * (device, 16-byte aligned) holds nd_swa_sink_chunk_prefill_workspace_size()
 * bytes (the gathered bf16 keys and values of sink_cap + min(ring_cap,
 * window-1) + chunk positions per sequence, and the tile plan).
 */
ND_API size_t nd_swa_sink_chunk_prefill_workspace_size(int batch, int chunk, int n_q_heads,
                                                       int n_kv_heads, int head_dim, int sink_cap,
                                                       int ring_cap, int window);
ND_API int nd_swa_sink_chunk_prefill(const void *q, const void *k, const void *v, int chunk,
                                     const nd_kv_cache *cache, int n_q_heads, int window,
                                     void *out, float *lse, void *workspace,
                                     size_t workspace_bytes, nd_stream_t stream);
/* The tile products nd_swa_sink_chunk_prefill's attention kernel performed
 * in its last call on `workspace` (as nd_swa_sink_prefill_tiles; the
 * arguments are those of the call and of its cache). */
ND_API int nd_swa_sink_chunk_prefill_tiles(const void *workspace, int batch, int chunk,
                                           int n_q_heads, int n_kv_heads, int head_dim,
                                           int sink_cap, int ring_cap, int window,
                                           long long *tiles_out);

/*
 * Work the bf16 prefill's attention kernel performed: after an
 * nd_swa_sink_prefill call with dtype ND_BF16 and these arguments has run on
 * `workspace` (the call's own workspace, not yet reused), writes to
 * *tiles_out the number of products of a 128-row query block with a 64-key
 * tile the kernel computed -- the tiles its plan kept, read from the plan in
 * the workspace (so this synchronises with the device).  Each such product
 * is 4 * 128 * 64 * head_dim flops (QK^T and PV).
 */
ND_API int nd_swa_sink_prefill_tiles(const void *workspace, int batch, int T, int n_q_heads,
                                     int n_kv_heads, int head_dim, float rope_theta, int block,
                                     long long *tiles_out);

/*
 * Rotary embedding (rotate-half) of x at positions 0..T-1 of each row, the
 * rotation [C3] "Pool before rotating, not after" applies to q and k.
 *   x, y  bf16 [batch][T][n_heads][head_dim]  (y may equal x: in place)
 * Angles: theta^(-2i/head_dim) and t * theta^(-2i/head_dim) reduced modulo
 * 2*pi are computed in double; the sine and cosine of the reduced angle and
 * the rotation itself in fp32, rounded once to bf16.
 */
ND_API int nd_rope_apply(const void *x, void *y, int batch, int T, int n_heads,
                  int head_dim, float rope_theta, nd_stream_t stream);

/*
 * Block pooling with midpoint rotation ([C3] "Pool before rotating, not
 * after"): pooled_k[j] = mean(k[j*block .. j*block+block-1]) rotated at
 * position min(j*block + block/2, T-1); pooled_v[j] = the mean of v (not
 * rotated).  Means are accumulated in fp32.  rope_theta == 0: no rotation.
 *   k, v                bf16 [batch][T][n_heads][head_dim]  (before rotation)
 *   pooled_k, pooled_v  bf16 [batch][T/block][n_heads][head_dim]
 */
ND_API int nd_kv_compress_pool(const void *k, const void *v, int batch, int T,
                        int n_heads, int head_dim, int block, float rope_theta,
                        void *pooled_k, void *pooled_v, nd_stream_t stream);

/*
 * Block pooling and K's rotation in one pass over K and V, as the compressed
 * prefill needs them ([C3] "Pool before rotating, not after"): writes
 *   k_rot               bf16 [batch][T][n_heads][head_dim]: k rotated at its
 *                       position (exactly as nd_rope_apply); not written and
 *                       may be NULL when rope_theta == 0
 *   pooled_k, pooled_v  exactly as nd_kv_compress_pool
 * The (cos, sin) table of positions 0..T-1 is built in `workspace` (device,
 * 16-byte aligned) of nd_kv_compress_pool_rope_workspace_size() bytes (0
 * when rope_theta == 0).  head_dim a multiple of 16, at most 256.
 */
ND_API size_t nd_kv_compress_pool_rope_workspace_size(int T, int head_dim, float rope_theta);
ND_API int nd_kv_compress_pool_rope(const void *k, const void *v, int batch, int T, int n_heads,
                                    int head_dim, int block, float rope_theta, void *k_rot,
                                    void *pooled_k, void *pooled_v, void *workspace,
                                    size_t workspace_bytes, nd_stream_t stream);

/* ------------------------------------------------------------------------ */
/* KV budget window (host only)                                              */
/* ------------------------------------------------------------------------ */

/*
 * kv_budget_window and effective_kv_window of [N2] "Effective KV Window:
 * Bounding the Cache Size" with the constants of [N1] "256 这个窗口宽度从哪来"
 * (budget 11 MiB + 512 KiB, group 32, minimum window 160):
 *   head_dim = (attn_dim or d_model) / num_heads     (attn_dim 0 = unset)
 *   kv       = num_kv_heads * head_dim
 *   per_pos  = num_layers * (2 kv + 2 (kv/32) * 4) + n_engram_sites * (d_model + 128)
 *   budget   = max(160, min(((11.5 MiB / per_pos) / 32) * 32, max_seq_len))
 *   effective = kv_window ? min(budget, kv_window) : budget
 * Exact integer arithmetic on the host; no device is touched.
 * Returns ND_ERR_INVALID_ARG for a NULL pointer, num_heads <= 0, negative
 * fields, or per_pos == 0.
 */
typedef struct {
  int d_model, attn_dim, num_heads, num_kv_heads, num_layers, n_engram_sites,
      max_seq_len, kv_window;
} nd_model_cfg;

ND_API int nd_kv_budget_window(const nd_model_cfg *cfg, int *budget_out,
                        int *effective_out);

#ifdef __cplusplus
}
#endif

#endif /* ND_H_ */
