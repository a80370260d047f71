// chunk_prefill.cu -- prefill of a chunk of new tokens against the bounded
// int8 cache, then the chunk's append to the cache.
//
// A sequence whose cache holds its pinned sink prefix and its newest ring
// entries continues with a chunk of Tc tokens at positions p0 .. p0+Tc-1
// (p0 = seq_len): query p0 + t attends, under the decode mask of
// "256-token滑动窗口+KV sink：Needle 2工具钉住机制源码分析" ("256-token 滑动窗口：
// 源码走读") -- a sink at any distance, otherwise qpos - kpos < window, causal
// -- to the cached keys and to the chunk's own keys.  The same computation as
// a prefill over the whole sequence for those rows, with the evicted
// positions gone (they are outside every chunk row's window).
//
// How: a gather kernel lays each sequence's keys out as one bf16 key
// sequence [sink slots | the newest min(ring_cap, window-1) ring entries in
// position order | the chunk] with segment ids (0 for empty slots) and sink
// flags, dequantising the cache (code * scale, rounded to bf16).  Key index
// distances then equal position distances between ring entries and chunk
// tokens, and sinks carry their flag, so the tensor-core prefill kernel's
// packed mask (same segment, causal, window or sink) is exactly the decode
// mask; it runs with queries = the chunk's rows only.  Finally the chunk's
// tokens are ring-appended to the cache (nd_kv_append_quant's rule, only the
// newest ring_cap of them need writing).
#include "nd_common.cuh"
#include "nd_internal.h"

namespace nd {

namespace {

struct GatherParams {
  nd_kv_cache c;
  const uint16_t *k, *v;  // chunk [B][Tc][Hkv][D]
  int Tc, R;              // chunk tokens, ring rows in the layout
  uint16_t *kk, *vv;      // [B][Tk][Hkv][D], Tk = sink_cap + R + Tc
  int32_t *seg;           // [B][Tk]
  uint8_t *sink;          // [B][Tk]
  int32_t *meta;          // [B][4] snapshot: sink_len, ring_start, ring_len, seq_len
  int *err;
};

// grid (row blocks of 8 key rows, B); each warp writes 256/D (key row, head,
// K or V) rows per step, a lane 8 channels of one row.
template <int D>
__global__ void __launch_bounds__(256) chunk_gather_kernel(const GatherParams p) {
  const nd_kv_cache &c = p.c;
  const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = c.sink_cap, Tk = S + p.R + p.Tc, Hkv = c.n_kv_heads, nslot = c.sink_cap + c.ring_cap;
  pdl_wait();
  const int sl = c.sink_len[b], rs = c.ring_start[b], rl = c.ring_len[b], sq = c.seq_len[b];
  const bool sane = sl >= 0 && sl <= S && rl >= 0 && rl <= c.ring_cap && rs >= 0 && rs < c.ring_cap;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    p.meta[4 * b + 0] = sane ? sl : 0;
    p.meta[4 * b + 1] = sane ? rs : 0;
    p.meta[4 * b + 2] = sane ? rl : 0;
    p.meta[4 * b + 3] = sane ? sq : -1;  // -1: skip the append
    if (!sane) raise_device_error(p.err, ND_DEVERR_METADATA);
  }
  const int row0 = blockIdx.x * 8;
  // segment ids and sink flags of this block's rows
  if (threadIdx.x < 8 && row0 + threadIdx.x < Tk) {
    const int i = row0 + threadIdx.x;
    int sg = 0, sk = 0;
    if (i < S) {
      sg = sane && i < sl;
      sk = sg;
    } else if (i < S + p.R) {
      const int r = S + p.R - i;  // position p0 - r
      sg = sane && r <= rl;
    } else {
      sg = 1;
    }
    p.seg[size_t(b) * Tk + i] = sg;
    p.sink[size_t(b) * Tk + i] = uint8_t(sk);
  }
  // rows of this block: (key row i, head h, K or V); a lane moves 8
  // channels (16 bytes of bf16), RPI rows per warp-iteration, kU
  // iterations' loads in flight before any is converted
  constexpr int RPI = 256 / D, kU = 4, kLanesPerRow = D / 8;
  const int sub = lane / kLanesPerRow, ch = (lane % kLanesPerRow) * 8;
  const int n_rows = 8 * Hkv * 2;
  for (int r0 = warp * RPI * kU; r0 < n_rows; r0 += 8 * RPI * kU) {
    int kind[kU];  // 0: zeros, 1: cached codes, 2: chunk copy, -1: past the end
    uint2 cw[kU];
    float sc[kU];
    uint4 cv[kU];
    size_t dst[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int r = r0 + u * RPI + sub;
      const int i = row0 + r / (2 * Hkv), h = (r >> 1) % Hkv;
      const bool is_v = r & 1;
      kind[u] = -1;
      if (r >= n_rows || i >= Tk) continue;
      dst[u] = ((size_t(b) * Tk + i) * Hkv + h) * D + ch;
      int slot = -1;
      if (i < S) {
        if (sane && i < sl) slot = i;
      } else if (i < S + p.R) {
        const int rr = S + p.R - i;
        if (sane && rr <= rl) slot = S + (rs + rl - rr) % c.ring_cap;
      } else {
        kind[u] = 2;
        cv[u] = *reinterpret_cast<const uint4 *>((is_v ? p.v : p.k) +
                                                 ((size_t(b) * p.Tc + (i - S - p.R)) * Hkv + h) * D + ch);
        continue;
      }
      kind[u] = slot >= 0 ? 1 : 0;
      if (slot >= 0) {
        const size_t row = (size_t(b) * Hkv + h) * nslot + slot;
        cw[u] = *reinterpret_cast<const uint2 *>((is_v ? c.v_codes : c.k_codes) + row * D + ch);
        sc[u] = (is_v ? c.v_scale : c.k_scale)[row * (D / 32) + ch / 32];
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int r = r0 + u * RPI + sub;
      if (kind[u] < 0) continue;
      uint16_t *out = ((r & 1) ? p.vv : p.kk) + dst[u];
      uint4 o = make_uint4(0u, 0u, 0u, 0u);
      if (kind[u] == 2) {
        o = cv[u];
      } else if (kind[u] == 1) {
        const uint32_t w2[2] = {cw[u].x, cw[u].y};
        uint32_t pk[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t wd = w2[q / 2];
          const int sh = (q & 1) * 16;
          const float lo = float(int8_t((wd >> sh) & 0xffu)) * sc[u];
          const float hi = float(int8_t((wd >> (sh + 8)) & 0xffu)) * sc[u];
          pk[q] = pack_bf16x2(lo, hi);
        }
        o = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      *reinterpret_cast<uint4 *>(out) = o;
    }
  }
}

constexpr int kAppendTokens = 2;  // chunk tokens per append CTA

struct AppendParams {
  nd_kv_cache c;
  const uint16_t *k, *v;  // chunk [B][Tc][Hkv][D]
  int Tc;
  const int32_t *meta;    // the snapshot taken before the chunk
};

// grid (pairs of tokens of the newest min(Tc, ring_cap), B): a warp per
// (token, head, K or V) quantises one row into its ring slot; block 0 of a
// sequence then advances its metadata (from the snapshot, so no block reads
// metadata another one has written).
template <int D>
__global__ void __launch_bounds__(256) chunk_append_kernel(const AppendParams p) {
  constexpr int CPL = D / 32;
  const nd_kv_cache &c = p.c;
  const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = c.n_kv_heads, nslot = c.sink_cap + c.ring_cap, cap = c.ring_cap;
  pdl_wait();
  const int rs = p.meta[4 * b + 1], rl = p.meta[4 * b + 2], sq = p.meta[4 * b + 3];
  if (sq < 0) return;
  const int first = p.Tc > cap ? p.Tc - cap : 0;  // older chunk tokens are overwritten within the chunk
  const int t0 = first + blockIdx.x * kAppendTokens;
  for (int item = warp; item < kAppendTokens * Hkv * 2; item += blockDim.x >> 5) {
    const int t = t0 + item / (2 * Hkv), h = (item >> 1) % Hkv;
    const bool is_v = item & 1;
    if (t >= p.Tc) continue;
    const int slot = c.sink_cap + (rs + rl + t) % cap;
    const uint16_t *src = (is_v ? p.v : p.k) + ((size_t(b) * p.Tc + t) * Hkv + h) * D + lane * CPL;
    float x[CPL];
    if constexpr (CPL == 4) {
      const uint2 w = *reinterpret_cast<const uint2 *>(src);
      x[0] = bf16_lo(w.x), x[1] = bf16_hi(w.x), x[2] = bf16_lo(w.y), x[3] = bf16_hi(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t *>(src);
      x[0] = bf16_lo(w), x[1] = bf16_hi(w);
    }
    int code[CPL];
    const float scale = quant_lanes<CPL>(x, code);
    const size_t row = (size_t(b) * Hkv + h) * nslot + slot;
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < CPL; ++e) packed |= uint32_t(code[e] & 0xff) << (8 * e);
    int8_t *codes = (is_v ? c.v_codes : c.k_codes) + row * D;
    if constexpr (CPL == 4) reinterpret_cast<uint32_t *>(codes)[lane] = packed;
    else reinterpret_cast<uint16_t *>(codes)[lane] = uint16_t(packed);
    if (lane % (32 / CPL) == 0) (is_v ? c.v_scale : c.k_scale)[row * (D / 32) + lane / (32 / CPL)] = scale;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const int total = rl + p.Tc;
    c.ring_len[b] = total < cap ? total : cap;
    c.ring_start[b] = (rs + (total > cap ? total - cap : 0)) % cap;
    c.seq_len[b] = sq + p.Tc;
  }
}

}  // namespace

int chunk_ring_rows(int ring_cap, int window) { return ring_cap < window - 1 ? ring_cap : window - 1; }

cudaError_t launch_chunk_gather(const nd_kv_cache &c, const void *k, const void *v, int Tc, int window, void *kk,
                                void *vv, int32_t *seg, uint8_t *sink, int32_t *meta, int *err, cudaStream_t stream) {
  GatherParams p;
  p.c = c;
  p.k = static_cast<const uint16_t *>(k);
  p.v = static_cast<const uint16_t *>(v);
  p.Tc = Tc;
  p.R = chunk_ring_rows(c.ring_cap, window);
  p.kk = static_cast<uint16_t *>(kk);
  p.vv = static_cast<uint16_t *>(vv);
  p.seg = seg;
  p.sink = sink;
  p.meta = meta;
  p.err = err;
  const int Tk = c.sink_cap + p.R + Tc;
  const dim3 grid((Tk + 7) / 8, c.batch);
  if (c.head_dim == 64) return launch_pdl(chunk_gather_kernel<64>, grid, dim3(256), 0, stream, p);
  if (c.head_dim == 128) return launch_pdl(chunk_gather_kernel<128>, grid, dim3(256), 0, stream, p);
  return cudaErrorInvalidValue;
}

cudaError_t launch_chunk_append(const nd_kv_cache &c, const void *k, const void *v, int Tc, const int32_t *meta,
                                cudaStream_t stream) {
  AppendParams p;
  p.c = c;
  p.k = static_cast<const uint16_t *>(k);
  p.v = static_cast<const uint16_t *>(v);
  p.Tc = Tc;
  p.meta = meta;
  const int n = Tc < c.ring_cap ? Tc : c.ring_cap;
  const dim3 grid((n + kAppendTokens - 1) / kAppendTokens, c.batch);
  if (c.head_dim == 64) return launch_pdl(chunk_append_kernel<64>, grid, dim3(256), 0, stream, p);
  if (c.head_dim == 128) return launch_pdl(chunk_append_kernel<128>, grid, dim3(256), 0, stream, p);
  return cudaErrorInvalidValue;
}

}  // namespace nd
