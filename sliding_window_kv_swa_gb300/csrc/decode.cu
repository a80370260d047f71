// decode.cu -- one decode step over the bounded int8 cache (sink slots + ring
// window), split-K over slots, with a combine kernel for the splits.
//
// What is computed: the decode mask of "256-token滑动窗口+KV sink：Needle 2工具钉住
// 机制源码分析", section "256-token 滑动窗口：源码走读": the query at position
// seq_len-1 keeps a cached key iff it is a sink or qpos - kpos < window; GQA
// head h reads KV head h / G.  Keys and values are code * scale with one fp32
// scale per 32 channels ("How the 256-Token Sliding Window Works with Tools as
// KV Sinks in Needle", section "Effective KV Window").
//
// How: HBM-bound (about 7 flop per byte at G = 4).  Each CTA streams a slice of
// the visible slots of one (sequence, KV head) straight from global memory
// (8-byte and 4-byte loads that fill whole 32-byte sectors), converts codes to
// fp16 in registers with byte permutes (exact for |code| <= 127), and lets
// warp-level m16n8k16 tensor-core MMAs do the dot products, so the per-byte
// ALU work is the conversion alone:
//   QK : D[head][slot]   = q(fp16, rows = heads) x codes^T, one MMA pair per
//        32-channel group so each group's partial is scaled by its own fp32
//        scale; q is pre-scaled by a power of two so its fp16 copy is exact.
//   PV : D[chan][head]   = codes^T(rows = channels) x P'^T, P' = p * v_scale,
//        also pre-scaled by a per-group power of two (no fp16 subnormals).
// The QK accumulator layout equals the PV B-operand layout, so
// probabilities never leave registers.  Online softmax per head uses quad
// shuffles; the four warps of a CTA are merged through shared memory.
#include "nd_common.cuh"
#include "nd_internal.h"

namespace nd {

namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kStep = 16;            // slots per warp iteration (one MMA k-step)
constexpr int kTargetCtas = 152 * 4;  // enough CTAs to fill every SM

struct DecodeParams {
  const uint16_t *q;
  nd_kv_cache c;
  int Hq, G, window;
  int n_split, slots_per_cta;
  uint16_t *out;
  float *lse;
  float *ws_ml;  // [B*Hkv][n_split][G][2]   (m in log2 units, l)
  float *ws_o;   // [B*Hkv][n_split][G][D]
  int *err;
};

__device__ __forceinline__ int ilog2_floor(float x) {  // x > 0, finite
  int e = int((__float_as_uint(x) >> 23) & 0xff) - 127;
  if (e == -127) {  // subnormal
    e = -127 + (31 - __clz(__float_as_uint(x) & 0x7fffff)) - 22;
  }
  return e;
}

// 2^e for e in [-126, 127]
__device__ __forceinline__ float exp2i(int e) {
  e = max(-126, min(127, e));
  return __uint_as_float(uint32_t(e + 127) << 23);
}

template <int D>
__global__ void __launch_bounds__(kThreads, D == 128 ? 3 : 4) decode_kernel(const DecodeParams p) {
  constexpr int NG = D / 32;  // scale groups per row
  const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const nd_kv_cache &c = p.c;
  const int G = p.G;
  const int nslot = c.sink_cap + c.ring_cap;
  const size_t pair = size_t(b) * c.n_kv_heads + hkv;

  __shared__ int s_meta[4];
  __shared__ unsigned s_vmax[NG];
  __shared__ float s_m[kWarps][8], s_l[kWarps][8];
  __shared__ float s_o[kWarps][8][D];
  __shared__ float s_qmax[8];

  if (threadIdx.x == 0) {
    int sl = c.sink_len[b], rs = c.ring_start[b], rl = c.ring_len[b];
    bool sane = sl >= 0 && sl <= c.sink_cap && rl >= 0 && rl <= c.ring_cap && rs >= 0 &&
                (c.ring_cap == 0 || rs < c.ring_cap);
    int total = 0, rs_eff = 0;
    if (!sane) {
      raise_device_error(p.err, ND_DEVERR_METADATA);
      sl = 0;
    } else {
      int n_vis = rl < p.window ? rl : p.window;
      int i0 = rl - n_vis;  // oldest visible ring entry (logical)
      rs_eff = c.ring_cap ? (rs + i0) % c.ring_cap : 0;
      total = sl + n_vis;
    }
    s_meta[0] = sl;
    s_meta[1] = rs_eff;
    s_meta[2] = total;
  }
  if (threadIdx.x < NG) s_vmax[threadIdx.x] = 0u;
  if (threadIdx.x < 8) s_qmax[threadIdx.x] = 0.f;
  __syncthreads();
  const int sink_len = s_meta[0], rs_eff = s_meta[1], total = s_meta[2];
  const int v_begin = split * p.slots_per_cta;
  const int v_end = min(v_begin + p.slots_per_cta, total);

  // virtual visible index -> physical slot
  auto phys = [&](int v) -> int {
    if (v < sink_len) return v;
    int r = rs_eff + (v - sink_len);
    if (r >= c.ring_cap) r -= c.ring_cap;
    return c.sink_cap + r;
  };

  const int8_t *kc = c.k_codes + pair * nslot * D;
  const int8_t *vc = c.v_codes + pair * nslot * D;
  const float *ks = c.k_scale + pair * nslot * NG;
  const float *vs = c.v_scale + pair * nslot * NG;

  // ---- per-group max of the value scales over this CTA's slots (for the
  //      power-of-two pre-scale of P'), and per-head max |q|.
  {
    float vmax[NG];
#pragma unroll
    for (int i = 0; i < NG; ++i) vmax[i] = 0.f;
    for (int v = v_begin + threadIdx.x; v < v_end; v += kThreads) {
      const float *row = vs + size_t(phys(v)) * NG;
#pragma unroll
      for (int i = 0; i < NG; ++i) vmax[i] = fmaxf(vmax[i], row[i]);
    }
#pragma unroll
    for (int i = 0; i < NG; ++i) {
      float m = vmax[i];
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) atomicMax(&s_vmax[i], __float_as_uint(m));
    }
    // |q| max per head: warp w handles heads w, w + 4
    for (int h = warp; h < G; h += kWarps) {
      const uint16_t *qh = p.q + (size_t(b) * p.Hq + hkv * G + h) * D;
      float m = 0.f;
      for (int ch = lane; ch < D; ch += 32) m = fmaxf(m, fabsf(__uint_as_float(uint32_t(qh[ch]) << 16)));
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) s_qmax[h] = m;
    }
  }
  __syncthreads();

  // ---- q fragments (A operand of QK), channel permutation per group:
  //      thread t owns channels 32*grp + 8t .. +7; k-step s uses 4s .. 4s+3.
  uint32_t qa[NG][2][2];
  float head_coef = 0.f;  // 2^-Eq * log2(e) / sqrt(D), for head g
  {
    const bool row_ok = g < G;
    float qm = row_ok ? s_qmax[g] : 0.f;
    int eq = qm > 0.f ? 14 - ilog2_floor(qm) : 0;
    float up = exp2i(eq);
    head_coef = exp2i(-eq) * (1.4426950408889634f * rsqrtf(float(D)));
    const uint16_t *qh = p.q + (size_t(b) * p.Hq + hkv * G + (row_ok ? g : 0)) * D;
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
      uint4 w = row_ok ? *reinterpret_cast<const uint4 *>(qh + 32 * grp + 8 * t) : make_uint4(0, 0, 0, 0);
      uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        qa[grp][s][0] = pack_half2(bf16_lo(ws[2 * s]) * up, bf16_hi(ws[2 * s]) * up);
        qa[grp][s][1] = pack_half2(bf16_lo(ws[2 * s + 1]) * up, bf16_hi(ws[2 * s + 1]) * up);
      }
    }
  }
  float vup[NG], vdown[NG];
#pragma unroll
  for (int grp = 0; grp < NG; ++grp) {
    float vm = __uint_as_float(s_vmax[grp]);
    int ev = vm > 0.f ? 14 - ilog2_floor(vm) : 0;
    vup[grp] = exp2i(ev);
    vdown[grp] = exp2i(-ev);
  }

  // ---- main loop: warp w takes k-steps w, w+4, ...
  float o[NG][2][4];
#pragma unroll
  for (int grp = 0; grp < NG; ++grp)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[grp][tt][i] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;

  for (int base = v_begin + warp * kStep; base < v_end; base += kWarps * kStep) {
    // slots this thread touches: K rows (tile j, slot g) and the score / V
    // columns 2t, 2t+1, 8+2t, 9+2t.
    const int vk0 = base + g, vk1 = base + 8 + g;
    const int vcol[4] = {base + 2 * t, base + 2 * t + 1, base + 8 + 2 * t, base + 9 + 2 * t};
    const int pk0 = phys(vk0 < v_end ? vk0 : base), pk1 = phys(vk1 < v_end ? vk1 : base);
    int pc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pc[i] = phys(vcol[i] < v_end ? vcol[i] : base);

    uint2 kw[2][NG];
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
      kw[0][grp] = *reinterpret_cast<const uint2 *>(kc + size_t(pk0) * D + 32 * grp + 8 * t);
      kw[1][grp] = *reinterpret_cast<const uint2 *>(kc + size_t(pk1) * D + 32 * grp + 8 * t);
    }
    uint32_t vw[4][NG];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int grp = 0; grp < NG; ++grp)
        vw[i][grp] = *reinterpret_cast<const uint32_t *>(vc + size_t(pc[i]) * D + 32 * grp + 4 * g);
    float ksc[4][NG], vsc[4][NG];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (NG == 4) {
        float4 a = *reinterpret_cast<const float4 *>(ks + size_t(pc[i]) * NG);
        float4 bb = *reinterpret_cast<const float4 *>(vs + size_t(pc[i]) * NG);
        ksc[i][0] = a.x; ksc[i][1] = a.y; ksc[i][2] = a.z; ksc[i][3] = a.w;
        vsc[i][0] = bb.x; vsc[i][1] = bb.y; vsc[i][2] = bb.z; vsc[i][3] = bb.w;
      } else {
#pragma unroll
        for (int grp = 0; grp < NG; ++grp) {
          ksc[i][grp] = ks[size_t(pc[i]) * NG + grp];
          vsc[i][grp] = vs[size_t(pc[i]) * NG + grp];
        }
      }
    }

    // ---- QK: scores for head g at columns 2t, 2t+1 of tiles 0 and 1
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) {
        float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
        const uint32_t w0 = kw[j][grp].x ^ 0x80808080u, w1 = kw[j][grp].y ^ 0x80808080u;
        mma_f16_16816(d0, d1, d2, d3, qa[grp][0][0], 0u, qa[grp][0][1], 0u,
                      codes_to_half2(w0, kSelBytes01), codes_to_half2(w0, kSelBytes23));
        mma_f16_16816(d0, d1, d2, d3, qa[grp][1][0], 0u, qa[grp][1][1], 0u,
                      codes_to_half2(w1, kSelBytes01), codes_to_half2(w1, kSelBytes23));
        sc[2 * j] = fmaf(ksc[2 * j][grp], d0, sc[2 * j]);
        sc[2 * j + 1] = fmaf(ksc[2 * j + 1][grp], d1, sc[2 * j + 1]);
      }
    }
    // ---- online softmax for head g (log2 domain)
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      sc[i] = (vcol[i] < v_end && g < G) ? sc[i] * head_coef : -INFINITY;
      mx = fmaxf(mx, sc[i]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);
    const float alpha = (m_new == -INFINITY) ? 1.f : ex2(m_run - m_new);
    float pr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pr[i] = (m_new == -INFINITY) ? 0.f : ex2(sc[i] - m_new);
    l_run = l_run * alpha + (pr[0] + pr[1]) + (pr[2] + pr[3]);
    m_run = m_new;
    // rescale O: this thread's O columns are heads 2t and 2t+1
    const float a_lo = __shfl_sync(0xffffffffu, alpha, (2 * t) * 4);
    const float a_hi = __shfl_sync(0xffffffffu, alpha, (2 * t + 1) * 4);
#pragma unroll
    for (int grp = 0; grp < NG; ++grp)
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        o[grp][tt][0] *= a_lo;
        o[grp][tt][1] *= a_hi;
        o[grp][tt][2] *= a_lo;
        o[grp][tt][3] *= a_hi;
      }
    // ---- PV: per group, B = P'^T (slot x head), A = V^T (channel x slot)
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
      const float u = vup[grp];
      const uint32_t b0 = pack_half2(pr[0] * (vsc[0][grp] * u), pr[1] * (vsc[1][grp] * u));
      const uint32_t b1 = pack_half2(pr[2] * (vsc[2][grp] * u), pr[3] * (vsc[3][grp] * u));
      const uint32_t x01 = prmt(vw[0][grp], vw[1][grp], 0x5140u) ^ 0x80808080u;
      const uint32_t x23 = prmt(vw[0][grp], vw[1][grp], 0x7362u) ^ 0x80808080u;
      const uint32_t y01 = prmt(vw[2][grp], vw[3][grp], 0x5140u) ^ 0x80808080u;
      const uint32_t y23 = prmt(vw[2][grp], vw[3][grp], 0x7362u) ^ 0x80808080u;
      // tile 0: rows g <-> channel 4g, rows g+8 <-> channel 4g+1
      mma_f16_16816(o[grp][0][0], o[grp][0][1], o[grp][0][2], o[grp][0][3],
                    codes_to_half2(x01, kSelBytes01), codes_to_half2(x01, kSelBytes23),
                    codes_to_half2(y01, kSelBytes01), codes_to_half2(y01, kSelBytes23), b0, b1);
      // tile 1: rows g <-> channel 4g+2, rows g+8 <-> channel 4g+3
      mma_f16_16816(o[grp][1][0], o[grp][1][1], o[grp][1][2], o[grp][1][3],
                    codes_to_half2(x23, kSelBytes01), codes_to_half2(x23, kSelBytes23),
                    codes_to_half2(y23, kSelBytes01), codes_to_half2(y23, kSelBytes23), b0, b1);
    }
  }

  // ---- merge: quad-sum l, then the four warps through shared memory
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  if (t == 0 && g < 8) {
    s_m[warp][g] = m_run;
    s_l[warp][g] = l_run;
  }
#pragma unroll
  for (int grp = 0; grp < NG; ++grp)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
      const int ch0 = 32 * grp + 4 * g + 2 * tt;  // row g; row g+8 is ch0 + 1
      s_o[warp][2 * t][ch0] = o[grp][tt][0] * vdown[grp];
      s_o[warp][2 * t + 1][ch0] = o[grp][tt][1] * vdown[grp];
      s_o[warp][2 * t][ch0 + 1] = o[grp][tt][2] * vdown[grp];
      s_o[warp][2 * t + 1][ch0 + 1] = o[grp][tt][3] * vdown[grp];
    }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
    const int h = idx / D, ch = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][h]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = ex2(s_m[w][h] - M);
        L += f * s_l[w][h];
        O += f * s_o[w][h][ch];
      }
    }
    if (p.n_split == 1) {
      const size_t row = size_t(b) * p.Hq + hkv * G + h;
      const float val = L > 0.f ? O / L : 0.f;
      p.out[row * D + ch] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
      if (ch == 0 && p.lse)
        p.lse[row] = L > 0.f ? (M + __log2f(L)) * 0.6931471805599453f : -INFINITY;
    } else {
      const size_t part = (pair * p.n_split + split) * G + h;
      p.ws_o[part * D + ch] = O;
      if (ch == 0) {
        p.ws_ml[part * 2] = M;
        p.ws_ml[part * 2 + 1] = L;
      }
    }
  }
}

// Merge the split-K partials of one (sequence, query head) per block.
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodeParams p) {
  const int row = blockIdx.x;  // b * Hq + h
  const int b = row / p.Hq, hq = row % p.Hq;
  const int hkv = hq / p.G, h = hq % p.G;
  const size_t pair = size_t(b) * p.c.n_kv_heads + hkv;
  const int ch = threadIdx.x;
  float M = -INFINITY;
  for (int s = 0; s < p.n_split; ++s)
    M = fmaxf(M, p.ws_ml[((pair * p.n_split + s) * p.G + h) * 2]);
  float L = 0.f, O = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < p.n_split; ++s) {
      const size_t part = (pair * p.n_split + s) * p.G + h;
      const float f = ex2(p.ws_ml[part * 2] - M);
      L += f * p.ws_ml[part * 2 + 1];
      O += f * p.ws_o[part * D + ch];
    }
  }
  const float val = L > 0.f ? O / L : 0.f;
  p.out[size_t(row) * D + ch] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
  if (ch == 0 && p.lse) p.lse[row] = L > 0.f ? (M + __log2f(L)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace

DecodePlan plan_decode(int batch, int n_kv_heads, int max_slots) {
  DecodePlan pl;
  const long pairs = long(batch) * n_kv_heads;
  const int ksteps = (max_slots + kStep - 1) / kStep;
  long want = pairs > 0 ? (kTargetCtas + pairs - 1) / pairs : 1;
  long cap = (ksteps + kWarps - 1) / kWarps;  // at least one k-step per warp
  long ns = want < cap ? want : cap;
  if (ns < 1) ns = 1;
  pl.n_split = int(ns);
  pl.slots_per_cta = int((ksteps + ns - 1) / ns) * kStep;
  if (pl.slots_per_cta == 0) pl.slots_per_cta = kStep;
  pl.max_slots = max_slots;
  return pl;
}

size_t decode_workspace_bytes(int batch, int n_q_heads, int head_dim, int max_slots,
                              int n_kv_heads_hint) {
  DecodePlan pl = plan_decode(batch, n_kv_heads_hint, max_slots);
  if (pl.n_split <= 1) return 0;
  return size_t(batch) * n_q_heads * pl.n_split * (head_dim + 2) * sizeof(float);
}

cudaError_t launch_decode(const void *q, const nd_kv_cache &c, int n_q_heads, int window,
                          void *out, float *lse, void *ws, size_t ws_bytes, int *err,
                          cudaStream_t stream) {
  const int max_slots = c.sink_cap + (c.ring_cap < window ? c.ring_cap : window);
  DecodePlan pl = plan_decode(c.batch, c.n_kv_heads, max_slots);
  DecodeParams p;
  p.q = static_cast<const uint16_t *>(q);
  p.c = c;
  p.Hq = n_q_heads;
  p.G = n_q_heads / c.n_kv_heads;
  p.window = window;
  p.n_split = pl.n_split;
  p.slots_per_cta = pl.slots_per_cta;
  p.out = static_cast<uint16_t *>(out);
  p.lse = lse;
  p.ws_ml = nullptr;
  p.ws_o = nullptr;
  p.err = err;
  if (pl.n_split > 1) {
    const size_t parts = size_t(c.batch) * n_q_heads * pl.n_split;
    if (ws == nullptr || ws_bytes < parts * (c.head_dim + 2) * sizeof(float))
      return cudaErrorInvalidValue;
    p.ws_o = static_cast<float *>(ws);
    p.ws_ml = p.ws_o + parts * c.head_dim;
  }
  dim3 grid(pl.n_split, c.n_kv_heads, c.batch);
  if (c.head_dim == 128) {
    decode_kernel<128><<<grid, kThreads, 0, stream>>>(p);
    if (pl.n_split > 1) decode_combine_kernel<128><<<c.batch * n_q_heads, 128, 0, stream>>>(p);
  } else if (c.head_dim == 64) {
    decode_kernel<64><<<grid, kThreads, 0, stream>>>(p);
    if (pl.n_split > 1) decode_combine_kernel<64><<<c.batch * n_q_heads, 64, 0, stream>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace nd
