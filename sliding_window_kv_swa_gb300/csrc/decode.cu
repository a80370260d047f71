// decode.cu -- one decode step over the bounded int8 cache (sink slots + ring
// window), with an optional split-K over slots and a combine kernel.
//
// What is computed: the decode mask of "256-token滑动窗口+KV sink：Needle 2工具钉住
// 机制源码分析", section "256-token 滑动窗口：源码走读": the query at position
// seq_len-1 keeps a cached key iff it is a sink or qpos - kpos < window; GQA
// head h reads KV head h / G.  Keys and values are code * scale with one fp32
// scale per 32 channels ("How the 256-Token Sliding Window Works with Tools as
// KV Sinks in Needle", section "Effective KV Window").
//
// How: HBM-bound (about 7 flop per byte at G = 4).  A CTA owns one (sequence,
// KV head) -- or a slice of its visible slots when there are too few sequences
// to fill the GPU -- and each warp walks 16-slot steps of it:
//   copy : every lane issues 16-byte cp.async copies of K codes, V codes and
//          scales for the step three (or four) steps ahead into the warp's own shared
//          stages (XOR-swizzled 16-byte chunks, so the fragment reads below
//          are bank-conflict free); no registers are tied up by loads in
//          flight, and the warp never waits on other warps.
//   math : codes become fp16 with byte permutes (exact for |code| <= 127) and
//          warp-level m16n8k16 tensor-core MMAs do the dot products, so the
//          per-byte ALU work is the conversion alone.
//          QK : D[head][slot] = q(fp16, rows = heads) x codes^T, one MMA pair
//               per 32-channel group so each group's fp32 scale multiplies its
//               own partial; q is pre-scaled by a power of two (exact).
//          PV : D[chan][head] = codes^T(rows = channels) x P'^T with
//               P' = p * v_scale, pre-scaled per group by a power of two that
//               only ever decreases (no fp16 overflow or subnormals).
//          The QK accumulator layout equals the PV B-operand layout, so
//          probabilities never leave registers; the online softmax uses quad
//          shuffles.
//   merge: the warps of a CTA merge through shared memory; split CTAs write
//          (max, sum, O) partials that a combine kernel merges.
// The kernel is a dependent launch: it may be scheduled while the previous
// kernel on the stream runs, and waits for it before its first global read.
// q, k_new / v_new and out / lse may be page-locked host memory (the
// host-buffer step passes its buffers in place): every access to them is an
// ordinary load or store.
#include <atomic>

#include "nd_common.cuh"
#include "nd_internal.h"

namespace nd {

namespace {

constexpr int kStep = 16;    // slots per warp step (one MMA k-step)
constexpr int kTargetCtas = 152;
constexpr float kLazyLog2 = 8.f;  // p is taken against a max at most 2^8 below the true one
// Largest cluster the fused step uses.  Clusters are co-scheduled on one GPC;
// at 8 CTAs that costs the large-batch step more than the saved launch.
constexpr int kMaxFusedCluster = 4;

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
  // fused step: the current token, appended to the ring before attending
  // (NULL: plain decode).  The launch is then a thread-block cluster over one
  // sequence's (split, KV head) CTAs.
  const uint16_t *k_new, *v_new;
};

// Cluster barrier halves: every thread arrives once it no longer needs the
// sequence's cache metadata; a wait returns once every non-exited thread of
// the cluster has arrived.
// Relaxed: the arrival only says that this CTA has read the sequence's
// metadata, and those reads have already returned (their values reached
// shared memory before the block-wide barrier that precedes the arrival), so
// no ordering of this thread's other memory traffic is needed -- a release
// would make every thread wait for its cache copies in flight (measured:
// 3% of the fused step).
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// Quantise one bf16 row of D channels held by a full warp (lane l has
// channels [l*CPL, l*CPL + CPL)) with the cache codec -- scale = amax/127,
// code = clamp(rint(x/scale), +-127), IEEE fp32 divides -- the same
// arithmetic as the append kernel, so the codes agree bit for bit.
template <int D>
__device__ __forceinline__ void quant_row_regs(uint2 w, int lane, int *code, float &scale) {
  constexpr int CPL = D / 32, kLanesPerGroup = 32 / CPL;
  float x[CPL];
  if constexpr (CPL == 4) {
    x[0] = bf16_lo(w.x), x[1] = bf16_hi(w.x), x[2] = bf16_lo(w.y), x[3] = bf16_hi(w.y);
  } else {
    x[0] = bf16_lo(w.x), x[1] = bf16_hi(w.x);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < CPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int off = kLanesPerGroup / 2; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  scale = __fdiv_rn(amax, 127.0f);
  const float inv = __frcp_rn(scale);
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    float r = 0.f;
    if (amax != 0.f) r = fminf(fmaxf(codec_rint(x[i], scale, inv), -127.f), 127.f);
    code[i] = int(r);
  }
}

// This lane's channels (D/32 of them, bf16) of one token row.
template <int D>
__device__ __forceinline__ uint2 load_row_words(const uint16_t *src, int lane) {
  if constexpr (D / 32 == 4) return reinterpret_cast<const uint2 *>(src)[lane];
  else return make_uint2(reinterpret_cast<const uint32_t *>(src)[lane], 0u);
}

template <int D>
struct Stage {
  static constexpr int kCodes = kStep * D;              // bytes of K (or V) codes per step
  static constexpr int kScales = kStep * (D / 32) * 4;  // bytes of K (or V) scales per step
  static constexpr int kBytes = 2 * kCodes + 2 * kScales;
};

__device__ __forceinline__ int ilog2_floor(float x) {  // x > 0, finite
  int e = int((__float_as_uint(x) >> 23) & 0xff) - 127;
  if (e == -127) e = -127 + (31 - __clz(__float_as_uint(x) & 0x7fffff)) - 22;  // subnormal
  return e;
}

// 2^e for e in [-126, 127]
__device__ __forceinline__ float exp2i(int e) {
  e = max(-126, min(127, e));
  return __uint_as_float(uint32_t(e + 127) << 23);
}

// Byte offset inside a stage: 16-byte chunks XOR-swizzled by the 128-byte
// line index, a bijection inside every 128-byte line.
__device__ __forceinline__ uint32_t swz(uint32_t a) { return a ^ (((a >> 7) & 7u) << 4); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ float ldsf(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a) : "memory");
  return v;
}
// The NG group scales of one slot, which sit together in the stage (16 or 8
// bytes).  At head_dim 128 one 16-byte load replaces four 4-byte loads for
// each of the eight K and V scale rows a thread reads per step (the kernel
// is issue-bound there: 4-5 points of HBM at B128-B512); at head_dim 64 the
// two 4-byte loads stay, since the 8-byte form adds a spill to the 96-register
// builds.
template <int NG>
__device__ __forceinline__ void lds_scales(uint32_t a, float *s) {
  if constexpr (NG == 4) {
    const float4 v = lds128f(a);
    s[0] = v.x, s[1] = v.y, s[2] = v.z, s[3] = v.w;
  } else {
    s[0] = ldsf(a);
    s[1] = ldsf(a + 4);
  }
}

// ST: cp.async stages per warp (ST - 1 steps in flight).  d = 128 has two
// builds: 4 stages at three CTAs per SM, and 5 stages at two CTAs per SM for
// grids of at most four CTAs per SM, where the bytes each CTA keeps in flight
// matter more than how many CTAs an SM holds.
template <int D, int NW, int ST>
__global__ void __launch_bounds__(NW * 32, D == 128 ? (ST == 4 ? 3 : 2) : (NW == 4 ? 5 : 1))
    decode_kernel(const DecodeParams p) {
  constexpr int kStages = ST;
  constexpr int NG = D / 32;  // scale groups per row
  using S = Stage<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ int s_meta[8];

  const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const nd_kv_cache &c = p.c;
  const int G = p.G;
  const int nslot = c.sink_cap + c.ring_cap;
  const size_t pair = size_t(b) * c.n_kv_heads + hkv;

  // The launch allows programmatic dependent launch: this grid may be
  // scheduled while the previous kernel on the stream is still running.
  // Nothing above reads global memory; the wait returns once that kernel
  // has completed and its writes (the cache, its metadata, q) are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const bool fused = p.k_new != nullptr;
  // the appended token, read now so its latency hides behind the metadata
  // read (only the warp that owns the new slot uses it).  At d = 128 the two
  // live registers cost the large-batch decode more than the early read
  // saves, so there the owning warp reads it when it needs it.
  uint2 k_row = make_uint2(0u, 0u), v_row = make_uint2(0u, 0u);
  if (D == 64 && fused) {
    k_row = load_row_words<D>(p.k_new + pair * D, lane);
    v_row = load_row_words<D>(p.v_new + pair * D, lane);
  }
  if (threadIdx.x == 0) {
    int sl = c.sink_len[b], rs = c.ring_start[b], rl = c.ring_len[b];
    const bool sane = sl >= 0 && sl <= c.sink_cap && rl >= 0 && rl <= c.ring_cap && rs >= 0 &&
                      (c.ring_cap == 0 || rs < c.ring_cap);
    int n_vis = 0, rs_eff = 0, new_slot = -1;
    if (!sane) {
      raise_device_error(p.err, ND_DEVERR_METADATA);
      sl = 0;
    } else {
      if (fused) {
        // ring append of the current token: the slot after the newest, or
        // the oldest one (which advances the ring start) when the ring is full
        new_slot = c.sink_cap + (rl < c.ring_cap ? (rs + rl) % c.ring_cap : rs);
        if (rl == c.ring_cap) rs = (rs + 1) % c.ring_cap;
        else ++rl;
        s_meta[4] = rs;
        s_meta[5] = rl;
        s_meta[6] = c.seq_len[b] + 1;
      }
      n_vis = rl < p.window ? rl : p.window;
      const int i0 = rl - n_vis;  // oldest visible ring entry (logical)
      rs_eff = c.ring_cap ? (rs + i0) % c.ring_cap : 0;
    }
    s_meta[0] = sl;
    s_meta[1] = rs_eff;
    s_meta[2] = n_vis;
    s_meta[3] = new_slot;
  }

  // ---- q: its loads go out now, its fragments are built once the cache
  //      copies below are on their way.  Thread t owns channels
  //      32*grp + 8t .. +7 of head g; k-step s uses 4s .. 4s+3.
  uint4 w[NG];
  {
    const bool row_ok = g < G;
    const uint16_t *qh = p.q + (size_t(b) * p.Hq + hkv * G + (row_ok ? g : 0)) * D;
#pragma unroll
    for (int grp = 0; grp < NG; ++grp)
      w[grp] = row_ok ? *reinterpret_cast<const uint4 *>(qh + 32 * grp + 8 * t) : make_uint4(0, 0, 0, 0);
  }
  // The CTA walks physical slots [v_begin, v_end) of the pair -- sink region,
  // then ring -- in storage order: the softmax does not depend on slot order,
  // so the copies start before the metadata read lands, and the metadata only
  // masks slots that are not visible.
  const int v_begin = split * p.slots_per_cta;
  const int v_end = min(v_begin + p.slots_per_cta, nslot);

  const int8_t *kc = c.k_codes + pair * nslot * D;
  const int8_t *vc = c.v_codes + pair * nslot * D;
  const float *ks = c.k_scale + pair * nslot * NG;
  const float *vs = c.v_scale + pair * nslot * NG;

  const uint32_t my_stages = smem_u32(smem) + warp * kStages * S::kBytes;
  // step n of this warp covers virtual slots base(n) .. base(n)+15
  const int first = v_begin + warp * kStep;
  const int n_steps = v_end > first ? (v_end - first + NW * kStep - 1) / (NW * kStep) : 0;
  auto base_of = [&](int n) { return first + n * NW * kStep; };

  // Every lane copies its share of one step: 16-byte chunks of K and V codes
  // and one scale row (K or V) of one slot.  One commit group per step
  // (empty past the end) keeps the group count uniform.
  // this lane's 16-byte chunks of a step: rows lane/(D/16) + k*(32*16/D),
  // column chunk lane % (D/16); fixed for every step
  constexpr int kChunks = kStep * D / 16, kPerLane = kChunks / 32, kRowStride = 32 * 16 / D;
  const int my_row0 = lane / (D / 16), my_ch = lane % (D / 16);
  // this lane's sources at slot 0 (a whole step adds base rows)
  const int8_t *kc_lane = kc + size_t(my_row0) * D + my_ch * 16;
  const int8_t *vc_lane = vc + size_t(my_row0) * D + my_ch * 16;
  const float *sc_lane = ((lane >> 4) ? vs : ks) + size_t(lane & 15) * NG;
  auto issue = [&](int n) {
    if (n < n_steps) {
      const int base = base_of(n);
      const uint32_t st = my_stages + (n % kStages) * S::kBytes;
      // a whole step (no slot past the range) needs no per-slot clamp; at
      // head_dim 64 the extra lane pointers would spill in the 96-register
      // builds, so there every step takes the clamped form below
      if (D == 128 && base + kStep <= v_end) {
        const size_t boff = size_t(base) * D;
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) {
          const uint32_t off = swz(uint32_t((my_row0 + k * kRowStride) * D + my_ch * 16));
          cp_async16(st + off, kc_lane + boff + k * kRowStride * D);
          cp_async16(st + S::kCodes + off, vc_lane + boff + k * kRowStride * D);
        }
        const uint32_t dst = st + 2 * S::kCodes + (lane >> 4) * S::kScales + (lane & 15) * NG * 4;
        if constexpr (NG == 4) cp_async16(dst, sc_lane + size_t(base) * NG);
        else cp_async8(dst, sc_lane + size_t(base) * NG);
        cp_async_commit();
        return;
      }
#pragma unroll
      for (int k = 0; k < kPerLane; ++k) {
        const int row = my_row0 + k * kRowStride;
        const int ps = base + row < v_end ? base + row : base;
        const uint32_t off = swz(uint32_t(row * D + my_ch * 16));
        const size_t goff = size_t(ps) * D + my_ch * 16;
        cp_async16(st + off, kc + goff);
        cp_async16(st + S::kCodes + off, vc + goff);
      }
      {
        const int row = lane & 15, which = lane >> 4;
        const int v = base + row;
        const int ps = v < v_end ? v : base;
        const uint32_t dst = st + 2 * S::kCodes + which * S::kScales + row * NG * 4;
        const float *src = (which ? vs : ks) + size_t(ps) * NG;
        if constexpr (NG == 4) cp_async16(dst, src);
        else cp_async8(dst, src);
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int n = 0; n < kStages - 1; ++n) issue(n);
  uint32_t qa[NG][2][2];
  float head_coef;  // 2^-Eq * log2(e) / sqrt(D), for head g
  {
    float qm = 0.f;
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
      const uint32_t ws[4] = {w[grp].x, w[grp].y, w[grp].z, w[grp].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) qm = fmaxf(qm, fmaxf(fabsf(bf16_lo(ws[i])), fabsf(bf16_hi(ws[i]))));
    }
    qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, 1));
    qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, 2));
    const int eq = qm > 0.f ? 14 - ilog2_floor(qm) : 0;
    const float up = exp2i(eq);
    head_coef = exp2i(-eq) * (1.4426950408889634f * rsqrtf(float(D)));
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
      const uint32_t ws[4] = {w[grp].x, w[grp].y, w[grp].z, w[grp].w};
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        qa[grp][s][0] = pack_half2(bf16_lo(ws[2 * s]) * up, bf16_hi(ws[2 * s]) * up);
        qa[grp][s][1] = pack_half2(bf16_lo(ws[2 * s + 1]) * up, bf16_hi(ws[2 * s + 1]) * up);
      }
    }
  }
  __syncthreads();  // the metadata is in
  const int sink_len = s_meta[0], rs_eff = s_meta[1], n_vis = s_meta[2], new_slot = s_meta[3];
  if (fused) cluster_arrive();  // this CTA is done reading the sequence's metadata
  // visible: a filled sink slot, or a ring slot inside the window's arc
  auto visible = [&](int ps) -> bool {
    if (ps >= v_end) return false;
    if (ps < c.sink_cap) return ps < sink_len;
    int d = ps - c.sink_cap - rs_eff;
    if (d < 0) d += c.ring_cap;
    return d < n_vis;
  };

  float o[NG][2][4];
#pragma unroll
  for (int grp = 0; grp < NG; ++grp)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[grp][tt][i] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // m_run: the max p is taken against (log2 units)
  int e_acc = 127;  // power-of-two pre-scale of P' (never increases; 127 = unset)

  for (int n = 0; n < n_steps; ++n) {
    issue(n + kStages - 1);
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const int base = base_of(n);
    const uint32_t st = my_stages + (n % kStages) * S::kBytes;
    if (fused && new_slot >= base && new_slot < base + kStep && new_slot < v_end) {
      // this warp owns the appended slot: quantise the token, store it in the
      // cache, and put it into the stage over the stale copy
      const int row = new_slot - base;
      constexpr int CPL = D / 32, kLanesPerGroup = 32 / CPL;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        int code[CPL];
        float scale;
        const uint2 row_w = D == 64 ? (which ? v_row : k_row)
                                    : load_row_words<D>((which ? p.v_new : p.k_new) + pair * D, lane);
        quant_row_regs<D>(row_w, lane, code, scale);
        uint32_t packed = 0;
#pragma unroll
        for (int i = 0; i < CPL; ++i) packed |= uint32_t(code[i] & 0xff) << (8 * i);
        int8_t *gcodes = (which ? c.v_codes : c.k_codes) + (pair * nslot + new_slot) * D;
        float *gscale = (which ? c.v_scale : c.k_scale) + (pair * nslot + new_slot) * NG;
        const uint32_t scodes = st + which * S::kCodes + swz(uint32_t(row * D + lane * CPL));
        if constexpr (CPL == 4) {
          reinterpret_cast<uint32_t *>(gcodes)[lane] = packed;
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(scodes), "r"(packed) : "memory");
        } else {
          reinterpret_cast<uint16_t *>(gcodes)[lane] = uint16_t(packed);
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(scodes), "h"(uint16_t(packed)) : "memory");
        }
        if (lane % kLanesPerGroup == 0) {
          const int grp = lane / kLanesPerGroup;
          gscale[grp] = scale;
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(st + 2 * S::kCodes + which * S::kScales +
                                                       (row * NG + grp) * 4),
                       "f"(scale)
                       : "memory");
        }
      }
      __syncwarp();
    }
    const int col[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
    // whole step visible (a filled sink run, or a full ring) -- the common
    // case -- or per slot
    const bool all_vis = base + kStep <= v_end &&
                         (base + kStep <= sink_len || (base >= c.sink_cap && n_vis == c.ring_cap));
    bool vis[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) vis[i] = all_vis || visible(base + col[i]);

    // ---- QK: scores for head g at columns 2t, 2t+1 of tiles 0 and 1
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int row = 8 * j + g;
      float ks0[NG], ks1[NG];  // K scales of this thread's two columns
      lds_scales<NG>(st + 2 * S::kCodes + (8 * j + 2 * t) * NG * 4, ks0);
      lds_scales<NG>(st + 2 * S::kCodes + (8 * j + 2 * t + 1) * NG * 4, ks1);
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) {
        const uint2 kw = lds64(st + swz(uint32_t(row * D + 32 * grp + 8 * t)));
        float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
        const uint32_t w0 = kw.x ^ 0x80808080u, w1 = kw.y ^ 0x80808080u;
        mma_f16_16816(d0, d1, d2, d3, qa[grp][0][0], 0u, qa[grp][0][1], 0u,
                      codes_to_half2(w0, kSelBytes01), codes_to_half2(w0, kSelBytes23));
        mma_f16_16816(d0, d1, d2, d3, qa[grp][1][0], 0u, qa[grp][1][1], 0u,
                      codes_to_half2(w1, kSelBytes01), codes_to_half2(w1, kSelBytes23));
        sc[2 * j] = fmaf(ks0[grp], d0, sc[2 * j]);
        sc[2 * j + 1] = fmaf(ks1[grp], d1, sc[2 * j + 1]);
      }
    }
    // ---- online softmax for head g (log2 domain)
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      sc[i] = (vis[i] && g < G) ? sc[i] * head_coef : -INFINITY;
      mx = fmaxf(mx, sc[i]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    // lazy max: p is taken against m_run, which moves (and O is rescaled)
    // only when a score exceeds it by more than 2^kLazyLog2, so p <= 2^8
    const bool need = mx > m_run + kLazyLog2;
    const float m_new = need ? mx : m_run;
    const float alpha = need ? (m_run == -INFINITY ? 0.f : ex2(m_run - m_new)) : 1.f;
    float pr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pr[i] = (m_new == -INFINITY) ? 0.f : ex2(sc[i] - m_new);
    l_run = l_run * alpha + (pr[0] + pr[1]) + (pr[2] + pr[3]);
    m_run = m_new;
    // V scales of the step, and one exponent for all groups that keeps
    // p * v_scale * 2^e below 2^15 (p <= 2^8); the accumulator keeps the
    // smallest exponent seen so far
    float vsc[NG][4];
    float vm = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float vs_i[NG];
      lds_scales<NG>(st + 2 * S::kCodes + S::kScales + col[i] * NG * 4, vs_i);
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) vsc[grp][i] = vs_i[grp];
    }
#pragma unroll
    for (int grp = 0; grp < NG; ++grp)
#pragma unroll
      for (int i = 0; i < 4; ++i) vm = fmaxf(vm, vis[i] ? vsc[grp][i] : 0.f);
    vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 1));
    vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 2));
    const int e_step = vm > 0.f ? 14 - int(kLazyLog2) - ilog2_floor(vm) : 127;
    const bool shrink_e = e_step < e_acc;
    // rescale O (this thread's columns are heads 2t and 2t+1) only when a
    // head's max moved or the exponent shrank: warp-uniform, and rare
    if (__any_sync(0xffffffffu, need || shrink_e)) {
      const float shrink = shrink_e ? (e_acc == 127 ? 0.f : exp2i(e_step - e_acc)) : 1.f;
      const float f_lo = __shfl_sync(0xffffffffu, alpha, (2 * t) * 4) * shrink;
      const float f_hi = __shfl_sync(0xffffffffu, alpha, (2 * t + 1) * 4) * shrink;
#pragma unroll
      for (int grp = 0; grp < NG; ++grp)
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
          o[grp][tt][0] *= f_lo;
          o[grp][tt][1] *= f_hi;
          o[grp][tt][2] *= f_lo;
          o[grp][tt][3] *= f_hi;
        }
      if (shrink_e) e_acc = e_step;
    }
    // (while no scale has been seen, every visible scale is 0 and u is moot)
    const float u = e_acc == 127 ? 1.f : exp2i(e_acc);
    float pu[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pu[i] = vis[i] ? pr[i] * u : 0.f;
    // ---- PV per group: B = P'^T (slot x head), A = V^T (channel x slot)
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
      // masked slots contribute 0 (their scale may be anything, even non-finite)
      const uint32_t b0 = pack_half2(vis[0] ? pu[0] * vsc[grp][0] : 0.f, vis[1] ? pu[1] * vsc[grp][1] : 0.f);
      const uint32_t b1 = pack_half2(vis[2] ? pu[2] * vsc[grp][2] : 0.f, vis[3] ? pu[3] * vsc[grp][3] : 0.f);
      uint32_t vw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        vw[i] = lds32(st + S::kCodes + swz(uint32_t(col[i] * D + 32 * grp + 4 * g)));
      const uint32_t x01 = prmt(vw[0], vw[1], 0x5140u) ^ 0x80808080u;
      const uint32_t x23 = prmt(vw[0], vw[1], 0x7362u) ^ 0x80808080u;
      const uint32_t y01 = prmt(vw[2], vw[3], 0x5140u) ^ 0x80808080u;
      const uint32_t y23 = prmt(vw[2], vw[3], 0x7362u) ^ 0x80808080u;
      // tile 0: rows g <-> channel 4g, rows g+8 <-> channel 4g+1
      mma_f16_16816(o[grp][0][0], o[grp][0][1], o[grp][0][2], o[grp][0][3],
                    codes_to_half2(x01, kSelBytes01), codes_to_half2(x01, kSelBytes23),
                    codes_to_half2(y01, kSelBytes01), codes_to_half2(y01, kSelBytes23), b0, b1);
      // tile 1: rows g <-> channel 4g+2, rows g+8 <-> channel 4g+3
      mma_f16_16816(o[grp][1][0], o[grp][1][1], o[grp][1][2], o[grp][1][3],
                    codes_to_half2(x23, kSelBytes01), codes_to_half2(x23, kSelBytes23),
                    codes_to_half2(y23, kSelBytes01), codes_to_half2(y23, kSelBytes23), b0, b1);
    }
    __syncwarp();  // every lane is done with this stage before it is refilled
  }
  cp_async_wait<0>();

  // With one CTA per SM (d = 64, 20 warps) the next kernel's CTAs may be
  // scheduled from here on; where several CTAs share an SM, early-placed CTAs
  // of the next step crowd unevenly, so there the trigger stays implicit (exit).
  if (D == 64 && NW == 20) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // ---- merge: quad-sum l, then the warps through shared memory (the stage
  //      buffers are free once every warp is past its loop)
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  __syncthreads();
  float *s_o = reinterpret_cast<float *>(smem);  // [NW][8][D]
  float *s_m = s_o + NW * 8 * D;                 // [NW][8]
  float *s_l = s_m + NW * 8;                     // [NW][8]
  if (t == 0) {
    s_m[warp * 8 + g] = m_run;
    s_l[warp * 8 + g] = l_run;
  }
  const float down = e_acc == 127 ? 0.f : exp2i(-e_acc);
#pragma unroll
  for (int grp = 0; grp < NG; ++grp) {
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
      const int ch0 = 32 * grp + 4 * g + 2 * tt;  // row g; row g+8 is ch0 + 1
      float *w0 = s_o + (warp * 8 + 2 * t) * D;
      float *w1 = s_o + (warp * 8 + 2 * t + 1) * D;
      w0[ch0] = o[grp][tt][0] * down;
      w1[ch0] = o[grp][tt][1] * down;
      w0[ch0 + 1] = o[grp][tt][2] * down;
      w1[ch0 + 1] = o[grp][tt][3] * down;
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
    const int h = idx / D, ch = idx % D;
    float M = -INFINITY;
    for (int w = 0; w < NW; ++w) M = fmaxf(M, s_m[w * 8 + h]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < NW; ++w) {
        const float f = ex2(s_m[w * 8 + h] - M);
        L += f * s_l[w * 8 + h];
        O += f * s_o[(w * 8 + h) * D + ch];
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
  if (fused && split == 0 && hkv == 0) {
    // the cluster barrier completes once every CTA of the sequence has read
    // its metadata (threads that have exited count as arrived); then the first
    // CTA publishes the appended state.  The others leave without waiting.
    cluster_wait();
    if (threadIdx.x == 0 && new_slot >= 0) {
      c.ring_start[b] = s_meta[4];
      c.ring_len[b] = s_meta[5];
      c.seq_len[b] = s_meta[6];
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

// Warps per CTA: 20 at head_dim 64 (one CTA per SM covers a whole short
// sequence in one or two steps per warp), 4 at head_dim 128 (two or three CTAs
// per SM, by ring depth).  Grids of many (sequence, KV head) pairs at head_dim
// 64 take a 4-warp build at five CTAs per SM instead (kManyPairs64): each
// warp then walks more steps and a CTA's merge spans 4 warps, not 20.
constexpr int warps_for(int D) { return D == 64 ? 20 : 4; }
constexpr long kManyPairs64 = 4L * kTargetCtas;

template <int D, int NW, int ST>
size_t decode_smem_bytes() {
  const size_t stages = size_t(NW) * ST * Stage<D>::kBytes;
  const size_t merge = size_t(NW) * 8 * D * 4 + 2 * size_t(NW) * 8 * 4;
  return stages > merge ? stages : merge;
}

template <int D, int ST, int NW = warps_for(D)>
cudaError_t launch_d(const DecodeParams &p, dim3 grid, cudaStream_t stream) {
  const size_t smem = decode_smem_bytes<D, NW, ST>();
  auto kern = decode_kernel<D, NW, ST>;
  // the shared-memory opt-in once per device (a per-launch call is host
  // time on every decode step)
  static std::atomic<unsigned long long> smem_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (!bit || !(smem_set.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    smem_set.fetch_or(bit, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.k_new) {
    // one cluster per sequence: its (split, KV head) CTAs
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = grid.x;
    attr[1].val.clusterDim.y = grid.y;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  if (p.n_split > 1) decode_combine_kernel<D><<<p.c.batch * p.Hq, D, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

DecodePlan plan_decode(int batch, int n_kv_heads, int max_slots, int head_dim) {
  DecodePlan pl;
  const long pairs = long(batch) * n_kv_heads;
  const int steps = (max_slots + kStep - 1) / kStep;
  const int nw = warps_for(head_dim);
  long ns = 1;
  // One CTA per (sequence, KV head) while that fills at least half the SMs;
  // otherwise split the slots so every SM gets work (at least one step per warp).
  if (pairs * 2 < kTargetCtas) {
    const long want = (kTargetCtas + pairs - 1) / (pairs > 0 ? pairs : 1);
    const long cap = (steps + nw - 1) / nw;
    ns = want < cap ? want : cap;
    if (ns < 1) ns = 1;
  }
  pl.n_split = int(ns);
  pl.slots_per_cta = int((steps + ns - 1) / ns) * kStep;
  if (pl.slots_per_cta == 0) pl.slots_per_cta = kStep;
  pl.max_slots = max_slots;
  return pl;
}

bool decode_step_fuses(int batch, int n_kv_heads, int max_slots, int head_dim) {
  return plan_decode(batch, n_kv_heads, max_slots, head_dim).n_split * n_kv_heads <= kMaxFusedCluster;
}

size_t decode_workspace_bytes(int batch, int n_q_heads, int head_dim, int max_slots, int n_kv_heads) {
  DecodePlan pl = plan_decode(batch, n_kv_heads, max_slots, head_dim);
  if (pl.n_split <= 1) return 0;
  return size_t(batch) * n_q_heads * pl.n_split * (head_dim + 2) * sizeof(float);
}

cudaError_t launch_decode(const void *q, const nd_kv_cache &c, int n_q_heads, int window,
                          void *out, float *lse, void *ws, size_t ws_bytes, int *err,
                          cudaStream_t stream, const void *k_new, const void *v_new) {
  const int max_slots = c.sink_cap + c.ring_cap;  // every physical slot is walked
  DecodePlan pl = plan_decode(c.batch, c.n_kv_heads, max_slots, c.head_dim);
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
  p.k_new = static_cast<const uint16_t *>(k_new);
  p.v_new = static_cast<const uint16_t *>(v_new);
  if (k_new && pl.n_split * c.n_kv_heads > kMaxFusedCluster) return cudaErrorInvalidConfiguration;
  if (pl.n_split > 1) {
    const size_t parts = size_t(c.batch) * n_q_heads * pl.n_split;
    if (ws == nullptr || ws_bytes < parts * (c.head_dim + 2) * sizeof(float))
      return cudaErrorInvalidValue;
    p.ws_o = static_cast<float *>(ws);
    p.ws_ml = p.ws_o + parts * c.head_dim;
  }
  dim3 grid(pl.n_split, c.n_kv_heads, c.batch);
  if (c.head_dim == 128) {
    // deeper rings when the grid is small (at most four CTAs per SM):
    // measured +4 points of HBM at 256 and 512 CTAs, -2 to -4 at 1024 and up
    const long ctas = long(grid.x) * grid.y * grid.z;
    return ctas <= 4L * kTargetCtas ? launch_d<128, 5>(p, grid, stream) : launch_d<128, 4>(p, grid, stream);
  }
  if (c.head_dim == 64) {
    const long ctas = long(grid.x) * grid.y * grid.z;
    return ctas >= kManyPairs64 ? launch_d<64, 4, 4>(p, grid, stream) : launch_d<64, 4>(p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace nd
