// kv_quant.cu -- int8 group-32 KV codec kernels: fused quantise-and-append into
// the bounded cache, and bulk row quantisation.
//
// Storage follows the per-position byte count of kv_budget_window in "How the
// 256-Token Sliding Window Works with Tools as KV Sinks in Needle", section
// "Effective KV Window: Bounding the Cache Size": int8 codes plus one fp32
// scale per 32 contiguous channels, for K and for V.  The ring/sink placement
// follows "KV Sinks for Tools" (pinned prefix never evicted, recent window
// kept).  Codec: scale = amax/127, code = clamp(rint(x/scale), +-127), both
// divisions IEEE fp32, so codes are reproducible bit for bit.
//
// Memory-bound and tiny (one token per sequence); one warp quantises one
// (token, head) row: lane l holds channels [l*CPL, l*CPL+CPL), a group of 32
// channels spans 32/CPL lanes, and the group absmax is a shuffle reduction.
#include "nd_common.cuh"
#include "nd_internal.h"

namespace nd {

namespace {

template <int CPL>
struct RowIO;

template <>
struct RowIO<1> {
  __device__ static void load(const uint16_t *src, int lane, float *x) {
    x[0] = __uint_as_float(uint32_t(src[lane]) << 16);
  }
  __device__ static void store(int8_t *dst, int lane, const int *c) {
    dst[lane] = int8_t(c[0]);
  }
};
template <>
struct RowIO<2> {
  __device__ static void load(const uint16_t *src, int lane, float *x) {
    uint32_t w = reinterpret_cast<const uint32_t *>(src)[lane];
    x[0] = bf16_lo(w);
    x[1] = bf16_hi(w);
  }
  __device__ static void store(int8_t *dst, int lane, const int *c) {
    reinterpret_cast<uint16_t *>(dst)[lane] = uint16_t((c[0] & 0xff) | ((c[1] & 0xff) << 8));
  }
};
template <>
struct RowIO<4> {
  __device__ static void load(const uint16_t *src, int lane, float *x) {
    uint2 w = reinterpret_cast<const uint2 *>(src)[lane];
    x[0] = bf16_lo(w.x);
    x[1] = bf16_hi(w.x);
    x[2] = bf16_lo(w.y);
    x[3] = bf16_hi(w.y);
  }
  __device__ static void store(int8_t *dst, int lane, const int *c) {
    reinterpret_cast<uint32_t *>(dst)[lane] = uint32_t(c[0] & 0xff) | (uint32_t(c[1] & 0xff) << 8) |
                                              (uint32_t(c[2] & 0xff) << 16) |
                                              (uint32_t(c[3] & 0xff) << 24);
  }
};
template <>
struct RowIO<8> {
  __device__ static void load(const uint16_t *src, int lane, float *x) {
    uint4 w = reinterpret_cast<const uint4 *>(src)[lane];
    uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16_lo(ws[i]);
      x[2 * i + 1] = bf16_hi(ws[i]);
    }
  }
  __device__ static void store(int8_t *dst, int lane, const int *c) {
    uint2 o;
    o.x = uint32_t(c[0] & 0xff) | (uint32_t(c[1] & 0xff) << 8) | (uint32_t(c[2] & 0xff) << 16) |
          (uint32_t(c[3] & 0xff) << 24);
    o.y = uint32_t(c[4] & 0xff) | (uint32_t(c[5] & 0xff) << 8) | (uint32_t(c[6] & 0xff) << 16) |
          (uint32_t(c[7] & 0xff) << 24);
    reinterpret_cast<uint2 *>(dst)[lane] = o;
  }
};

// Quantise one row of 32*CPL bf16 channels held by a full warp.
template <int CPL>
__device__ __forceinline__ void quant_row(const uint16_t *src, int8_t *codes, float *scales,
                                          int lane) {
  constexpr int kLanesPerGroup = 32 / CPL;
  float x[CPL];
  RowIO<CPL>::load(src, lane, x);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < CPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int off = kLanesPerGroup / 2; off >= 1; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = __fdiv_rn(amax, 127.0f), inv = __frcp_rn(scale);
  int c[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    float r = 0.f;
    if (amax != 0.f) r = fminf(fmaxf(codec_rint(x[i], scale, inv), -127.f), 127.f);
    c[i] = int(r);
  }
  RowIO<CPL>::store(codes, lane, c);
  if (lane % kLanesPerGroup == 0) scales[lane / kLanesPerGroup] = scale;
}

template <int CPL>
__global__ void __launch_bounds__(256) kv_append_quant_kernel(nd_kv_cache c, const uint16_t *k_new,
                                                              const uint16_t *v_new, int to_sink,
                                                              int *err) {
  constexpr int D = 32 * CPL;
  const int b = blockIdx.x;
  __shared__ int s_slot;
  if (threadIdx.x == 0) {
    int sl = c.sink_len[b], rs = c.ring_start[b], rl = c.ring_len[b];
    int slot = -1;
    bool sane = sl >= 0 && sl <= c.sink_cap && rl >= 0 && rl <= c.ring_cap && rs >= 0 &&
                rs < (c.ring_cap > 0 ? c.ring_cap : 1);
    if (!sane) {
      raise_device_error(err, ND_DEVERR_METADATA);
    } else if (to_sink) {
      if (rl == 0 && sl < c.sink_cap) slot = sl;
      else raise_device_error(err, ND_DEVERR_METADATA);
    } else if (c.ring_cap > 0) {
      int r = rl < c.ring_cap ? (rs + rl) % c.ring_cap : rs;
      slot = c.sink_cap + r;
    }
    s_slot = slot;
  }
  __syncthreads();
  const int slot = s_slot;
  if (slot < 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nslot = c.sink_cap + c.ring_cap;
  for (int item = warp; item < 2 * c.n_kv_heads; item += blockDim.x >> 5) {
    const int h = item >> 1;
    const bool is_v = item & 1;
    const size_t row = (size_t(b) * c.n_kv_heads + h) * nslot + slot;
    const uint16_t *src = (is_v ? v_new : k_new) + (size_t(b) * c.n_kv_heads + h) * D;
    quant_row<CPL>(src, (is_v ? c.v_codes : c.k_codes) + row * D,
                   (is_v ? c.v_scale : c.k_scale) + row * (D / 32), lane);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (to_sink) {
      c.sink_len[b] += 1;
    } else if (c.ring_len[b] < c.ring_cap) {
      c.ring_len[b] += 1;
    } else {
      c.ring_start[b] = (c.ring_start[b] + 1) % c.ring_cap;
    }
    c.seq_len[b] += 1;
  }
}

template <int CPL>
__global__ void __launch_bounds__(256) kv_quant_rows_kernel(const uint16_t *x, int64_t n_rows,
                                                            int8_t *codes, float *scales) {
  constexpr int D = 32 * CPL;
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n_rows;
       r += warps)
    quant_row<CPL>(x + r * D, codes + r * D, scales + r * (D / 32), lane);
}

// ------------------------------------------------------------------ prefill -> cache
// Quantise RPI = 256/D rows of D channels per warp-iteration: lane l holds 8
// channels (16 bytes) of row l / (D/8); a 32-channel group spans 4 lanes (a
// group never straddles two rows, so every lane of a group has the same row).
// Same arithmetic as quant_row (IEEE divides, rint, clamp), so the same codes.
// Every lane of the warp must call it (the group absmax is a shuffle).
__device__ __forceinline__ uint2 quant8(const uint4 w, float &scale) {
  float x[8];
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16_lo(u[i]);
    x[2 * i + 1] = bf16_hi(u[i]);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  scale = __fdiv_rn(amax, 127.0f);
  if (amax == 0.f) return make_uint2(0u, 0u);
  const float inv = __frcp_rn(scale);
  // Round-to-integer by adding and subtracting 1.5 * 2^23 (the classic
  // "magic number" rounding): for |p| < 2^22 the sum t has a unit ulp, so it
  // is p rounded to the nearest integer (ties to even, as rint), and t's low
  // mantissa byte is that integer's two's-complement byte -- the code.  The
  // decision to trust p is codec_rint's; outside its tie band, with a normal
  // scale, |p| <= 127 * (1 + 3 * 2^-24) < 127.5, so the code needs no clamp.
  // Inside the band the IEEE quotient decides (and is clamped), as there.
  uint32_t wd[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float p = __fmul_rn(x[i], inv);
    const float t = __fadd_rn(p, 12582912.0f);
    const float r = __fsub_rn(t, 12582912.0f);
    wd[i] = __float_as_uint(t);
    if (!(fabsf(fabsf(__fsub_rn(p, r)) - 0.5f) > 1e-4f && scale >= 1e-30f))
      wd[i] = uint32_t(int(fminf(fmaxf(rintf(__fdiv_rn(x[i], scale)), -127.f), 127.f)));
  }
  // byte 0 of each word, four to a register
  const uint32_t lo = prmt(prmt(wd[0], wd[1], 0x0040u), prmt(wd[2], wd[3], 0x0040u), 0x5410u);
  const uint32_t hi = prmt(prmt(wd[4], wd[5], 0x0040u), prmt(wd[6], wd[7], 0x0040u), 0x5410u);
  return make_uint2(lo, hi);
}

constexpr int kFillTokens = 16;     // kept tokens per quantising CTA
constexpr int kFillThreads = 256;
constexpr int kPlanThreads = 1024;  // one planning CTA per cache row

struct FillParams {
  nd_kv_cache c;
  const uint16_t *k, *v;  // [batch][T][Hkv][D]
  int batch, T;
  const int32_t *seg_ids;  // may be NULL
  const uint8_t *sink;     // may be NULL
  const int32_t *src_row, *src_seg;
  int32_t *plan;  // per cache row: [0] kept tokens (-1: row untouched), then (position, slot) pairs
  int plan_stride;
  int *err;
};

// Plan of cache row e (one CTA): the tokens of segment src_seg[e] of batch
// row src_row[e], in position order, under the append rule -- while the ring
// is empty a sink token goes to the next sink slot (rejected once the sink
// region is full); every other token goes to the ring, and once the ring has
// a token, sink tokens are rejected.  Two walks over the batch row, four
// positions per thread per pass: totals and the first ring token's rank,
// then every token's rank; the kept tokens' (position, slot) pairs go to the
// plan, the row's metadata to the cache.  A row of at most one pass keeps
// its flags and prefix sums in registers for the second walk.
__global__ void __launch_bounds__(kPlanThreads) kv_fill_plan_kernel(const FillParams p) {
  constexpr int NW = kPlanThreads / 32, kPer = 4, kPass = kPer * kPlanThreads;
  __shared__ int s_wsum[NW][2];
  __shared__ int s_first_r;
  const nd_kv_cache &c = p.c;
  const int e = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t *plan = p.plan + size_t(e) * p.plan_stride;
  pdl_wait();
  const int b = p.src_row[e];
  const int seg = p.seg_ids ? p.src_seg[e] : 1;
  if (b < 0 || b >= p.batch || seg <= 0) {  // row left untouched
    if (tid == 0) {
      plan[0] = -1;
      if (b >= 0) raise_device_error(p.err, ND_DEVERR_METADATA);
    }
    return;
  }
  if (tid == 0) s_first_r = 0x7fffffff;
  __syncthreads();
  const int32_t *sg = p.seg_ids ? p.seg_ids + size_t(b) * p.T : nullptr;
  const uint8_t *sk = p.sink ? p.sink + size_t(b) * p.T : nullptr;
  // a thread's four positions are consecutive: one 16-byte load of their
  // segment ids and one 4-byte load of their sink flags where the row allows
  const bool vec = (p.T % kPer) == 0 && (reinterpret_cast<uintptr_t>(p.seg_ids) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(p.sink) & 3) == 0;
  auto load_flags = [&](int base, bool *in, bool *snk) {
    const int t0 = base + kPer * tid;
    if (vec && t0 + kPer <= p.T) {
      int sv[kPer] = {seg, seg, seg, seg};
      if (sg) {
        const int4 q = *reinterpret_cast<const int4 *>(sg + t0);
        sv[0] = q.x, sv[1] = q.y, sv[2] = q.z, sv[3] = q.w;
      }
      const uint32_t f = sk ? *reinterpret_cast<const uint32_t *>(sk + t0) : 0u;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        in[j] = sv[j] == seg;
        snk[j] = in[j] && ((f >> (8 * j)) & 0xffu) != 0u;
      }
      return;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int t = t0 + j;
      in[j] = t < p.T && (!sg || sg[t] == seg);
      snk[j] = in[j] && sk && sk[t];
    }
  };
  // block-wide exclusive prefix of (a, s) over threads; totals in ta, ts
  auto block_scan = [&](int a, int s, int &ea, int &es, int &ta, int &ts) {
    int ia = a, is = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int ya = __shfl_up_sync(0xffffffffu, ia, off), ys = __shfl_up_sync(0xffffffffu, is, off);
      if (lane >= off) ia += ya, is += ys;
    }
    if (lane == 31) s_wsum[warp][0] = ia, s_wsum[warp][1] = is;
    __syncthreads();
    ea = ia - a, es = is - s, ta = 0, ts = 0;
#pragma unroll 8
    for (int w = 0; w < NW; ++w) {
      if (w < warp) ea += s_wsum[w][0], es += s_wsum[w][1];
      ta += s_wsum[w][0], ts += s_wsum[w][1];
    }
    __syncthreads();  // s_wsum is reused by the next call
  };
  // a row of at most kPass positions is one pass: its flags and prefix sums
  // serve the second walk as they are
  const bool one_pass = p.T <= kPass;
  bool in1[kPer], snk1[kPer];
  int ea1 = 0, es1 = 0;
  int tot_seg = 0, tot_snk = 0;
  for (int base = 0; base < p.T; base += kPass) {
    bool in[kPer], snk[kPer];
    load_flags(base, in, snk);
    int a = 0, s = 0, first_local = -1;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (in[j] && !snk[j] && first_local < 0) first_local = a;
      a += in[j];
      s += snk[j];
    }
    int ea, es, ta, ts;
    block_scan(a, s, ea, es, ta, ts);
    if (one_pass) {
#pragma unroll
      for (int j = 0; j < kPer; ++j) in1[j] = in[j], snk1[j] = snk[j];
      ea1 = ea, es1 = es;
    }
    if (first_local >= 0) atomicMin(&s_first_r, tot_seg + ea + first_local);
    tot_seg += ta;
    tot_snk += ts;
  }
  __syncthreads();
  // the rank of the first ring token = the segment's tokens before it (all
  // sinks); no ring token: every token of the segment
  const int f = s_first_r == 0x7fffffff ? tot_seg : s_first_r;
  const int n_sink = min(f, c.sink_cap);  // accepted sink tokens
  const int n_ring = tot_seg - tot_snk;   // ring tokens
  const int kept_ring = min(n_ring, c.ring_cap);
  const int i0 = n_ring - kept_ring;      // oldest ring token kept
  if (tid == 0) {
    c.sink_len[e] = n_sink;
    c.ring_len[e] = kept_ring;
    c.ring_start[e] = n_ring > c.ring_cap ? n_ring % c.ring_cap : 0;
    c.seq_len[e] = n_sink + n_ring;
    plan[0] = n_sink + kept_ring;
    if (tot_snk > n_sink) raise_device_error(p.err, ND_DEVERR_METADATA);  // rejected sink tokens
  }
  int carry_seg = 0, carry_snk = 0;
  for (int base = 0; base < p.T; base += kPass) {
    bool in[kPer], snk[kPer];
    int ea, es, ta, ts;
    if (one_pass) {
#pragma unroll
      for (int j = 0; j < kPer; ++j) in[j] = in1[j], snk[j] = snk1[j];
      ea = ea1, es = es1, ta = tot_seg, ts = tot_snk;
    } else {
      load_flags(base, in, snk);
      int a = 0, s = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) a += in[j], s += snk[j];
      block_scan(a, s, ea, es, ta, ts);
    }
    int rank = carry_seg + ea, rsnk = carry_snk + es;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (!in[j]) continue;
      int kept = -1, slot = 0;
      if (rank < n_sink) {
        kept = rank;
        slot = rank;
      } else if (!snk[j]) {
        const int i = rank - rsnk;  // ring index of this token
        if (i >= i0) {
          kept = n_sink + i - i0;
          slot = c.sink_cap + i % c.ring_cap;
        }
      }
      if (kept >= 0) {
        plan[1 + 2 * kept] = base + kPer * tid + j;
        plan[2 + 2 * kept] = slot;
      }
      rank += 1;
      rsnk += snk[j];
    }
    carry_seg += ta;
    carry_snk += ts;
  }
}

// Quantise kept tokens [16*blockIdx.x, +16) of cache row blockIdx.y from its
// plan: rows (token, head, K or V), RPI = 256/D rows per warp-iteration, four
// iterations' loads in flight.
template <int D>
__global__ void __launch_bounds__(kFillThreads) kv_fill_kernel(const FillParams p) {
  constexpr int NW = kFillThreads / 32;
  const nd_kv_cache &c = p.c;
  const int e = blockIdx.y, c0 = blockIdx.x * kFillTokens;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  __shared__ int s_pos[kFillTokens], s_slot[kFillTokens];
  const int32_t *plan = p.plan + size_t(e) * p.plan_stride;
  const int n_kept = plan[0];
  if (c0 >= n_kept) return;  // also the untouched rows (-1)
  const int b = p.src_row[e];
  // this CTA's (position, slot) pairs, so no row's load waits on the plan
  if (threadIdx.x < kFillTokens && c0 + int(threadIdx.x) < n_kept) {
    s_pos[threadIdx.x] = plan[1 + 2 * (c0 + threadIdx.x)];
    s_slot[threadIdx.x] = plan[2 + 2 * (c0 + threadIdx.x)];
  }
  __syncthreads();
  constexpr int RPI = 256 / D, kUnroll = 4;
  const int n_tok = min(kFillTokens, n_kept - c0), Hkv = c.n_kv_heads;
  const int n_rows = n_tok * Hkv * 2, nslot = c.sink_cap + c.ring_cap;
  const int sub = lane / (D / 8);
  // row r = (token j, head h, K or V) = 2 (j Hkv + h) + (r & 1).  With two
  // or more rows per warp-iteration (RPI even) a lane's rows advance by
  // whole (token, head) pairs and keep their K/V side, so each lane divides
  // once per iteration and steps its (j, h) from there.
  for (int r0 = warp * RPI * kUnroll; r0 < n_rows; r0 += NW * RPI * kUnroll) {
    uint4 w[kUnroll];
    int rows[kUnroll], slots[kUnroll], heads[kUnroll];
    int j = 0, h = 0;
    if constexpr (RPI >= 2) {
      const int pair0 = (r0 >> 1) + (sub >> 1);
      j = pair0 / Hkv;
      h = pair0 - j * Hkv;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int r = r0 + u * RPI + sub;
      if constexpr (RPI == 1) {  // (head_dim 256: one row per iteration)
        j = (r >> 1) / Hkv;
        h = (r >> 1) - j * Hkv;
      }
      rows[u] = r;
      heads[u] = h;
      w[u] = make_uint4(0, 0, 0, 0);
      slots[u] = 0;
      if (r < n_rows) {
        const int t = s_pos[j];
        slots[u] = s_slot[j];
        const uint16_t *src = ((r & 1) ? p.v : p.k) + ((size_t(b) * p.T + t) * Hkv + h) * D;
        w[u] = *reinterpret_cast<const uint4 *>(src + (lane % (D / 8)) * 8);
      }
      if constexpr (RPI >= 2) {
        h += RPI / 2;  // this lane's next row: RPI/2 pairs on, same side
        while (h >= Hkv) {
          h -= Hkv;
          ++j;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      // every lane takes part in the shuffles; rows past the end are not stored
      float scale;
      const uint2 q8 = quant8(w[u], scale);
      const int r = rows[u];
      if (r < n_rows) {
        const int h = heads[u], ch = (lane % (D / 8)) * 8;
        const bool is_v = r & 1;
        const size_t row = (size_t(e) * Hkv + h) * nslot + slots[u];
        *reinterpret_cast<uint2 *>((is_v ? c.v_codes : c.k_codes) + row * D + ch) = q8;
        if ((lane & 3) == 0) (is_v ? c.v_scale : c.k_scale)[row * (D / 32) + ch / 32] = scale;
      }
    }
  }
}

}  // namespace

size_t kv_fill_plan_ints(int sink_cap, int ring_cap) {
  return (size_t(1) + 2 * size_t(sink_cap + ring_cap) + 3) / 4 * 4;  // 16-byte rows
}

cudaError_t launch_kv_fill(const nd_kv_cache &c, const void *k, const void *v, int batch, int T,
                           const int32_t *seg_ids, const uint8_t *sink, const int32_t *src_row,
                           const int32_t *src_seg, int32_t *plan, int *err, cudaStream_t stream) {
  FillParams p;
  p.c = c;
  p.k = static_cast<const uint16_t *>(k);
  p.v = static_cast<const uint16_t *>(v);
  p.batch = batch;
  p.T = T;
  p.seg_ids = seg_ids;
  p.sink = sink;
  p.src_row = src_row;
  p.src_seg = src_seg;
  p.plan = plan;
  p.plan_stride = int(kv_fill_plan_ints(c.sink_cap, c.ring_cap));
  p.err = err;
  cudaError_t e = launch_pdl(kv_fill_plan_kernel, dim3(c.batch), dim3(kPlanThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  const int slots = c.sink_cap + c.ring_cap;
  const dim3 grid((slots + kFillTokens - 1) / kFillTokens, c.batch);
  switch (c.head_dim) {
    case 32: return launch_pdl(kv_fill_kernel<32>, grid, dim3(kFillThreads), 0, stream, p);
    case 64: return launch_pdl(kv_fill_kernel<64>, grid, dim3(kFillThreads), 0, stream, p);
    case 128: return launch_pdl(kv_fill_kernel<128>, grid, dim3(kFillThreads), 0, stream, p);
    case 256: return launch_pdl(kv_fill_kernel<256>, grid, dim3(kFillThreads), 0, stream, p);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_kv_append_quant(const nd_kv_cache &c, const void *k_new, const void *v_new,
                                   int to_sink, int *err, cudaStream_t stream) {
  const uint16_t *kn = static_cast<const uint16_t *>(k_new);
  const uint16_t *vn = static_cast<const uint16_t *>(v_new);
  dim3 grid(c.batch), block(256);
  switch (c.head_dim) {
    case 32: kv_append_quant_kernel<1><<<grid, block, 0, stream>>>(c, kn, vn, to_sink, err); break;
    case 64: kv_append_quant_kernel<2><<<grid, block, 0, stream>>>(c, kn, vn, to_sink, err); break;
    case 128: kv_append_quant_kernel<4><<<grid, block, 0, stream>>>(c, kn, vn, to_sink, err); break;
    case 256: kv_append_quant_kernel<8><<<grid, block, 0, stream>>>(c, kn, vn, to_sink, err); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_kv_quant_rows(const void *x, int64_t n_rows, int head_dim, int8_t *codes,
                                 float *scales, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  const uint16_t *xs = static_cast<const uint16_t *>(x);
  int64_t blocks = (n_rows + 7) / 8;
  int grid = int(blocks < 152 * 16 ? blocks : 152 * 16);
  switch (head_dim) {
    case 32: kv_quant_rows_kernel<1><<<grid, 256, 0, stream>>>(xs, n_rows, codes, scales); break;
    case 64: kv_quant_rows_kernel<2><<<grid, 256, 0, stream>>>(xs, n_rows, codes, scales); break;
    case 128: kv_quant_rows_kernel<4><<<grid, 256, 0, stream>>>(xs, n_rows, codes, scales); break;
    case 256: kv_quant_rows_kernel<8><<<grid, 256, 0, stream>>>(xs, n_rows, codes, scales); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace nd
