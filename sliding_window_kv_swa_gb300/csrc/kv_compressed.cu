// kv_compressed.cu -- decode step of compressed attention over a bounded,
// incrementally pooled int8 cache.
//
// "Compressed attention and the copy probe", sections "Two kinds of columns,
// pooled blocks and exact recent keys" and "Pool before rotating, not after":
// a query at position p attends one softmax over [pooled blocks j visible iff
// (j+1)*block <= p - W + 1, exact keys p-W+1 .. p]; a pooled key is the mean of
// its block's keys before rotation, rotated once at the block midpoint
// j*block + block/2; pooled values are plain means.  Section "So what
// happened ?" prices this cache at inference: W exact positions plus one per
// block outside the window instead of every position.
//
// The cache is an nd_kv_cache: its sink region holds n_pinned pinned tokens
// (the sink prefix of "KV Sinks for Tools", exact keys visible at any
// distance; 0 for the pages' compressed attention) followed by pooled block j
// in slot n_pinned + j; its ring holds the exact window.  A pooled block,
// once visible, stays visible for every later query, so the visible pooled
// blocks are a growing prefix of the sink region and sink_len counts them:
// the ordinary decode kernel then computes the compressed attention as is.
//
// One step (this file): per sequence, the token at position p = seq_len --
//   pinned (p < n_pinned): rotated K and V quantised into sink slot p;
//   else: rotated K and V quantised into the ring (the append rule), and the
//         token's unrotated K and V added to the fp32 sums of its block;
//         when p closes block j (its last token), the means (sum / block,
//         IEEE divide) are formed, K's rotated at the midpoint, both rounded
//         to bf16 and quantised into slot n_pinned + j -- the block is
//         written as soon as it is complete and becomes visible (sink_len
//         grows) once (j+1)*block <= p' - W + 1 - n_pinned at a later p';
// q is rotated at p into the workspace; then the decode kernel attends.
// Rotation and quantisation use the same angles (rot_cs), rounding
// (rope_pair, bf16) and codec as the rotary, pooling and append kernels, so
// the ring and the pooled slots hold bit for bit what those produce.
#include "nd_common.cuh"
#include "nd_internal.h"

namespace nd {

namespace {

struct CompressedParams {
  nd_kv_cache c;
  float *k_sum, *v_sum;  // [batch][n_kv_heads][D]
  int block, n_pinned, window, Hq;
  const uint16_t *q, *k_new, *v_new;
  uint16_t *q_rot;  // [batch][Hq][D]
  int *err;
  Freqs fr;
};

// One CTA per sequence; warp items: (KV head, K or V) rows, then q heads.
template <int D>
__global__ void __launch_bounds__(512) compressed_append_kernel(const CompressedParams p) {
  constexpr int CPL = D / 32;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const nd_kv_cache &c = p.c;
  // s_meta: 0 position, 1 exact slot (-1: skip), 2 pooled slot (-1: none),
  //         3 new ring_start, 4 new ring_len, 5 new sink_len, 6 block
  //         flags (bit 0: first token of its block, bit 1: closes it)
  __shared__ int s_meta[8];
  // (cos, sin) at the token's position and at its block's midpoint, built
  // once per CTA (the double-precision reduction is off every row's chain)
  __shared__ float2 s_cs[2][D / 2];
  pdl_wait();
  // Each warp's first kPre items read their inputs (the new token's row, the
  // block's running sums, a query row) now, so those loads overlap the
  // metadata read and the angle setup below instead of following them.
  const int Hkv = c.n_kv_heads, nslot = c.sink_cap + c.ring_cap;
  const int n_items = 2 * Hkv + p.Hq;
  const int c0 = lane * CPL;
  constexpr int kPre = 4;
  auto load = [&](const uint16_t *src, float *x) {
    if constexpr (CPL == 4) {
      const uint2 w = reinterpret_cast<const uint2 *>(src)[lane];
      x[0] = bf16_lo(w.x), x[1] = bf16_hi(w.x), x[2] = bf16_lo(w.y), x[3] = bf16_hi(w.y);
    } else {
      const uint32_t w = reinterpret_cast<const uint32_t *>(src)[lane];
      x[0] = bf16_lo(w), x[1] = bf16_hi(w);
    }
  };
  auto fetch = [&](int item, float *x, float *sum) {
    if (item >= 2 * Hkv) {
      load(p.q + (size_t(b) * p.Hq + (item - 2 * Hkv)) * D, x);
      return;
    }
    const size_t pair = size_t(b) * Hkv + (item >> 1);
    const bool is_v = item & 1;
    load((is_v ? p.v_new : p.k_new) + pair * D, x);
    const float *sp = (is_v ? p.v_sum : p.k_sum) + pair * D + c0;
#pragma unroll
    for (int e = 0; e < CPL; ++e) sum[e] = sp[e];
  };
  float px[kPre][CPL], ps[kPre][CPL];
#pragma unroll
  for (int t = 0; t < kPre; ++t)
    if (warp + t * nw < n_items) fetch(warp + t * nw, px[t], ps[t]);
  if (threadIdx.x == 0) {
    const int sl = c.sink_len[b], rs = c.ring_start[b], rl = c.ring_len[b], pos = c.seq_len[b];
    const bool sane = sl >= 0 && sl <= c.sink_cap && rl >= 0 && rl <= c.ring_cap && rs >= 0 &&
                      rs < c.ring_cap && pos >= 0;
    int exact = -1, pooled = -1, nrs = rs, nrl = rl, mode = 0, nsl = sl;
    if (!sane) {
      raise_device_error(p.err, ND_DEVERR_METADATA);
    } else if (pos < p.n_pinned) {
      if (pos < c.sink_cap) exact = pos;
      else raise_device_error(p.err, ND_DEVERR_METADATA);
    } else {
      exact = c.sink_cap + (rl < c.ring_cap ? (rs + rl) % c.ring_cap : rs);
      if (rl == c.ring_cap) nrs = (rs + 1) % c.ring_cap;
      else nrl = rl + 1;
      const int r = (pos - p.n_pinned) % p.block, j = (pos - p.n_pinned) / p.block;
      mode = r == 0 ? 1 : 0;
      if (r == p.block - 1) {
        mode |= 2;
        if (p.n_pinned + j < c.sink_cap) pooled = p.n_pinned + j;
        else raise_device_error(p.err, ND_DEVERR_METADATA);
      }
    }
    if (exact >= 0) {
      // visible after this token: the pinned tokens seen, then the pooled
      // blocks j with (j+1)*block <= pos - W + 1 - n_pinned
      const int lim = pos - p.window + 1 - p.n_pinned;
      const int n_blk = lim >= p.block ? lim / p.block : 0;
      nsl = min(pos + 1, p.n_pinned) + n_blk;
      nsl = min(nsl, c.sink_cap);
    }
    s_meta[0] = pos;
    s_meta[1] = exact;
    s_meta[2] = pooled;
    s_meta[3] = nrs;
    s_meta[4] = nrl;
    s_meta[5] = nsl;
    s_meta[6] = mode;
  }
  __syncthreads();
  const int pos = s_meta[0], exact = s_meta[1], pooled = s_meta[2], mode = s_meta[6];
  if (exact < 0) return;
  const bool pinned = pos < p.n_pinned;
  const int mid = pinned ? 0 : p.n_pinned + ((pos - p.n_pinned) / p.block) * p.block + p.block / 2;
  for (int i = threadIdx.x; i < D; i += blockDim.x)
    s_cs[i / (D / 2)][i % (D / 2)] = rot_cs(double(i < D / 2 ? pos : mid), p.fr.f[i % (D / 2)]);
  __syncthreads();
  // this lane's channel pairs: lanes 0-15 hold x_i, lanes 16-31 the partner
  // x_{i + D/2} of the same pairs (lane ^ 16)
  const int i0 = c0 % (D / 2);
  const bool hi = lane >= 16;
  auto rotate = [&](float *x, int which) {  // which: 0 at the position, 1 at the block midpoint
    float partner[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) partner[e] = __shfl_xor_sync(0xffffffffu, x[e], 16);
#pragma unroll
    for (int e = 0; e < CPL; ++e) {
      const float2 cs = s_cs[which][i0 + e];
      float ya, yb;
      if (hi) {
        rope_pair(partner[e], x[e], cs.x, cs.y, ya, yb);
        x[e] = yb;
      } else {
        rope_pair(x[e], partner[e], cs.x, cs.y, ya, yb);
        x[e] = ya;
      }
    }
  };
  auto store_quant = [&](const float *x, int8_t *codes, float *scales) {
    int code[CPL];
    const float scale = quant_lanes<CPL>(x, code);
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < CPL; ++e) packed |= uint32_t(code[e] & 0xff) << (8 * e);
    if constexpr (CPL == 4) reinterpret_cast<uint32_t *>(codes)[lane] = packed;
    else reinterpret_cast<uint16_t *>(codes)[lane] = uint16_t(packed);
    if (lane % (32 / CPL) == 0) scales[lane / (32 / CPL)] = scale;
  };
  // item: its inputs x (the row) and sum (the block's running sums), fetched
  auto process = [&](int item, const float *x_in, const float *sum_in) {
    if (item >= 2 * Hkv) {  // a query head: rotated at pos, rounded to bf16
      const int h = item - 2 * Hkv;
      const size_t off = (size_t(b) * p.Hq + h) * D;
      float x[CPL];
#pragma unroll
      for (int e = 0; e < CPL; ++e) x[e] = x_in[e];
      rotate(x, 0);
      if constexpr (CPL == 4)
        reinterpret_cast<uint2 *>(p.q_rot + off)[lane] = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
      else
        reinterpret_cast<uint32_t *>(p.q_rot + off)[lane] = pack_bf16x2(x[0], x[1]);
      return;
    }
    const int h = item >> 1;
    const bool is_v = item & 1;
    const size_t pair = size_t(b) * Hkv + h;
    float x[CPL], raw[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) raw[e] = x[e] = x_in[e];
    // the exact key (rotated at pos, rounded to bf16) or value
    if (!is_v) {
      rotate(x, 0);
#pragma unroll
      for (int e = 0; e < CPL; ++e) x[e] = round_bf16(x[e]);
    }
    store_quant(x, (is_v ? c.v_codes : c.k_codes) + (pair * nslot + exact) * D,
                (is_v ? c.v_scale : c.k_scale) + (pair * nslot + exact) * (D / 32));
    if (pinned) return;
    // the block's running sums (fp32, in position order, before rotation)
    float *sum = (is_v ? p.v_sum : p.k_sum) + pair * D + c0;
    float acc[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) acc[e] = (mode & 1) ? raw[e] : sum_in[e] + raw[e];
    if (!(mode & 2)) {
#pragma unroll
      for (int e = 0; e < CPL; ++e) sum[e] = acc[e];
      return;
    }
    // the block is complete: its mean, K rotated at the block midpoint
    const float fb = float(p.block);
#pragma unroll
    for (int e = 0; e < CPL; ++e) acc[e] = __fdiv_rn(acc[e], fb);
    if (!is_v) rotate(acc, 1);
#pragma unroll
    for (int e = 0; e < CPL; ++e) acc[e] = round_bf16(acc[e]);
    if (pooled >= 0)
      store_quant(acc, (is_v ? c.v_codes : c.k_codes) + (pair * nslot + pooled) * D,
                  (is_v ? c.v_scale : c.k_scale) + (pair * nslot + pooled) * (D / 32));
  };
#pragma unroll
  for (int t = 0; t < kPre; ++t)
    if (warp + t * nw < n_items) process(warp + t * nw, px[t], ps[t]);
  for (int item = warp + kPre * nw; item < n_items; item += nw) {
    float x[CPL], sum[CPL];
    fetch(item, x, sum);
    process(item, x, sum);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!pinned) {
      c.ring_start[b] = s_meta[3];
      c.ring_len[b] = s_meta[4];
    }
    c.sink_len[b] = s_meta[5];
    c.seq_len[b] = pos + 1;
  }
}

}  // namespace

cudaError_t launch_compressed_append(const nd_kv_cache &c, float *k_sum, float *v_sum, int block, int n_pinned,
                                     int window, const void *q, int Hq, const void *k_new, const void *v_new,
                                     void *q_rot, float theta, int *err, cudaStream_t stream) {
  CompressedParams p;
  p.c = c;
  p.k_sum = k_sum;
  p.v_sum = v_sum;
  p.block = block;
  p.n_pinned = n_pinned;
  p.window = window;
  p.Hq = Hq;
  p.q = static_cast<const uint16_t *>(q);
  p.k_new = static_cast<const uint16_t *>(k_new);
  p.v_new = static_cast<const uint16_t *>(v_new);
  p.q_rot = static_cast<uint16_t *>(q_rot);
  p.err = err;
  p.fr = make_freqs(c.head_dim, theta);
  if (theta == 0.f)  // no rotation: every angle 0 (cos 1, sin 0: rope_pair is exact)
    for (int i = 0; i < kMaxHalf; ++i) p.fr.f[i] = 0.0;
  const dim3 grid(c.batch), blk(512);
  if (c.head_dim == 64) return launch_pdl(compressed_append_kernel<64>, grid, blk, 0, stream, p);
  if (c.head_dim == 128) return launch_pdl(compressed_append_kernel<128>, grid, blk, 0, stream, p);
  return cudaErrorInvalidValue;
}

}  // namespace nd
