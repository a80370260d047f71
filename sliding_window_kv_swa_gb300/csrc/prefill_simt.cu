// prefill_simt.cu -- prefill attention on CUDA cores in fp32.
//
// The mask is make_causal_packing_mask of "How the 256-Token Sliding Window
// Works with Tools as KV Sinks in Needle", section "KV Sinks for Tools":
// same segment (id > 0), causal, and (no window, or within the window, or a
// sink key).  With pooled columns it is compressed_mask of "Compressed
// attention and the copy probe", section "Two kinds of columns": pooled block j
// visible iff (j+1)*block <= q - window + 1, then the causal sliding window.
//
// This is the path for fp32 inputs (parity at 1e-4 rules out reduced-precision
// tensor-core inputs).  One CTA takes 16 query rows of one (sequence, query
// head); eight threads share a row and split the head dimension (short
// dot-product chains, two partial sums each, and four times the CTAs of a
// two-threads-per-row layout for the small problems this path serves).  Key
// tiles of 64 are staged in shared memory; a tile is skipped when no row of
// the CTA can see any of its keys (causal bound, window bound without sinks,
// or disjoint segment-id ranges).  Online softmax in the log2 domain.
#include "nd_common.cuh"
#include "nd_internal.h"

#include <climits>

namespace nd {

namespace {

constexpr int kTpr = 8;  // threads per query row
constexpr int kRows = 16, kKeys = 64, kThreads = kRows * kTpr;

template <typename E>
__device__ __forceinline__ float ld_elem(const E *p, size_t i);
template <>
__device__ __forceinline__ float ld_elem<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld_elem<uint16_t>(const uint16_t *p, size_t i) {
  return __uint_as_float(uint32_t(p[i]) << 16);
}
template <typename E>
__device__ __forceinline__ void st_elem(E *p, size_t i, float x);
template <>
__device__ __forceinline__ void st_elem<float>(float *p, size_t i, float x) { p[i] = x; }
template <>
__device__ __forceinline__ void st_elem<uint16_t>(uint16_t *p, size_t i, float x) {
  p[i] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

template <typename E, int D>
__global__ void __launch_bounds__(kThreads) prefill_simt_kernel(const PrefillArgs a) {
  constexpr int H2 = D / kTpr;  // channels per thread
  extern __shared__ float smem[];
  float *sk = smem;                 // [kKeys][D]
  float *sv = sk + kKeys * D;       // [kKeys][D]
  __shared__ int s_seg[kKeys];
  __shared__ unsigned char s_sink[kKeys];
  __shared__ int s_qseg_lo, s_qseg_hi;

  const int qt = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
  const int T = a.T, G = a.Hq / a.Hkv, hk = hq / G;
  const int r = threadIdx.x / kTpr, part = threadIdx.x % kTpr;  // part: this thread's channel slice
  const int q0 = qt * kRows;
  const int q = q0 + r;
  const bool row_ok = q < T;
  const int q_last = min(q0 + kRows, T) - 1;
  const E *Q = static_cast<const E *>(a.q);
  const E *K = static_cast<const E *>(a.k);
  const E *V = static_cast<const E *>(a.v);
  const int W = a.window;
  const int my_seg = (a.seg_ids && row_ok) ? a.seg_ids[size_t(b) * T + q] : (row_ok ? 1 : 0);

  if (threadIdx.x == 0) {
    s_qseg_lo = INT_MAX;
    s_qseg_hi = INT_MIN;
  }
  __syncthreads();
  if (part == 0 && row_ok && my_seg > 0) {
    atomicMin(&s_qseg_lo, my_seg);
    atomicMax(&s_qseg_hi, my_seg);
  }

  const float qscale = 1.4426950408889634f * rsqrtf(float(D));
  float qr[H2], o[H2];
#pragma unroll
  for (int c = 0; c < H2; ++c) {
    qr[c] = row_ok ? ld_elem(Q, ((size_t(b) * T + q) * a.Hq + hq) * D + part * H2 + c) * qscale : 0.f;
    o[c] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  __syncthreads();
  const int qseg_lo = s_qseg_lo, qseg_hi = s_qseg_hi;

  // One pass over a column source: pooled (src = 1) or exact keys (src = 0).
  auto run = [&](int src, int n_cols) {
    const E *KK = src ? static_cast<const E *>(a.pooled_k) : K;
    const E *VV = src ? static_cast<const E *>(a.pooled_v) : V;
    const int TK = src ? (T / a.block) : T;
    int col_end;  // exclusive bound on useful columns for this CTA
    if (src) {
      // largest j with (j+1)*block <= q_last - W + 1
      int lim = q_last - W + 1;
      col_end = lim >= a.block ? min(lim / a.block, n_cols) : 0;
    } else {
      col_end = q_last + 1;
    }
    for (int k0 = 0; k0 < col_end; k0 += kKeys) {
      // ---- tile metadata and skip test (exact keys only)
      if (!src) {
        if (threadIdx.x < kKeys) {
          const int k = k0 + threadIdx.x;
          s_seg[threadIdx.x] = (k < T) ? (a.seg_ids ? a.seg_ids[size_t(b) * T + k] : 1) : 0;
          s_sink[threadIdx.x] = (k < T && a.sink) ? a.sink[size_t(b) * T + k] : 0;
        }
        __syncthreads();
        int any_sink = 0, lo = INT_MAX, hi = INT_MIN;
        for (int i = 0; i < kKeys; ++i) {
          if (s_seg[i] > 0) {
            lo = min(lo, s_seg[i]);
            hi = max(hi, s_seg[i]);
          }
          any_sink |= s_sink[i];
        }
        const bool in_window = (W == 0) || (k0 + kKeys - 1 >= q0 - W + 1);
        const bool seg_overlap = lo <= qseg_hi && hi >= qseg_lo;
        if (!seg_overlap || (!in_window && !any_sink)) {
          __syncthreads();
          continue;
        }
      }
      // ---- stage K and V tile (fp32): 16-byte loads, a thread's loads all
      //      issued before its shared-memory stores
      if constexpr (sizeof(E) == 4) {
        constexpr int kVec = kKeys * D / 4, kPer = kVec / kThreads;
        float4 kx[kPer], vx[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int idx = threadIdx.x + u * kThreads;
          const int kk = idx / (D / 4), c4 = idx % (D / 4);
          const int k = k0 + kk;
          kx[u] = vx[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (k < TK) {
            const size_t off = ((size_t(b) * TK + k) * a.Hkv + hk) * D + 4 * c4;
            kx[u] = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(KK) + off);
            vx[u] = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(VV) + off);
          }
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int idx = threadIdx.x + u * kThreads;
          reinterpret_cast<float4 *>(sk)[idx] = kx[u];
          reinterpret_cast<float4 *>(sv)[idx] = vx[u];
        }
      } else {
        for (int idx = threadIdx.x; idx < kKeys * D; idx += kThreads) {
          const int kk = idx / D, c = idx % D;
          const int k = k0 + kk;
          float kv = 0.f, vv = 0.f;
          if (k < TK) {
            const size_t off = ((size_t(b) * TK + k) * a.Hkv + hk) * D + c;
            kv = ld_elem(KK, off);
            vv = ld_elem(VV, off);
          }
          sk[idx] = kv;
          sv[idx] = vv;
        }
      }
      __syncthreads();
      // four keys per step: four independent dot products, then one max,
      // one rescale and four exponentials (the online softmax's serial
      // chain is a quarter as long)
      constexpr int kStepKeys = 4;
      for (int kk0 = 0; kk0 < kKeys; kk0 += kStepKeys) {
        float sv4[kStepKeys];
        bool vis4[kStepKeys];
#pragma unroll
        for (int u = 0; u < kStepKeys; ++u) {
          const int kk = kk0 + u, k = k0 + kk;
          if (src) {
            vis4[u] = row_ok && k < n_cols && (k + 1) * a.block <= q - W + 1;
          } else {
            vis4[u] = row_ok && k <= q && my_seg > 0 && s_seg[kk] == my_seg &&
                      (W == 0 || q - k < W || s_sink[kk]);
          }
          const float *kr = sk + kk * D + part * H2;
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int c = 0; c < H2; c += 2) {
            s0 = fmaf(qr[c], kr[c], s0);
            s1 = fmaf(qr[c + 1], kr[c + 1], s1);
          }
          sv4[u] = s0 + s1;
        }
#pragma unroll
        for (int off = 1; off < kTpr; off <<= 1)
#pragma unroll
          for (int u = 0; u < kStepKeys; ++u) sv4[u] += __shfl_xor_sync(0xffffffffu, sv4[u], off);
        float mx = m;
#pragma unroll
        for (int u = 0; u < kStepKeys; ++u)
          if (vis4[u]) mx = fmaxf(mx, sv4[u]);
        if (mx == -INFINITY) continue;  // nothing visible yet
        if (mx > m) {
          const float f = ex2(m - mx);  // m = -inf: f = 0
          l *= f;
#pragma unroll
          for (int c = 0; c < H2; ++c) o[c] *= f;
          m = mx;
        }
#pragma unroll
        for (int u = 0; u < kStepKeys; ++u) {
          if (!vis4[u]) continue;
          const float pr = ex2(sv4[u] - m);
          l += pr;
          const float *vr = sv + (kk0 + u) * D + part * H2;
#pragma unroll
          for (int c = 0; c < H2; ++c) o[c] = fmaf(pr, vr[c], o[c]);
        }
      }
      __syncthreads();
    }
  };

  if (a.block > 0) run(1, T / a.block);
  run(0, T);

  if (row_ok) {
    E *O = static_cast<E *>(a.out);
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < H2; ++c)
      st_elem(O, ((size_t(b) * T + q) * a.Hq + hq) * D + part * H2 + c, o[c] * inv);
    if (a.lse && part == 0)
      a.lse[(size_t(b) * a.Hq + hq) * T + q] =
          l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
  }
}

template <typename E, int D>
cudaError_t launch_simt(const PrefillArgs &a, cudaStream_t stream) {
  const size_t smem = size_t(2) * kKeys * D * sizeof(float);
  auto kern = prefill_simt_kernel<E, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((a.T + kRows - 1) / kRows, a.Hq, a.batch);
  kern<<<grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

// fp32 inputs on CUDA cores (bf16 inputs always take the tensor-core kernel).
cudaError_t launch_prefill_f32(const PrefillArgs &a, cudaStream_t stream) {
  if (size_t(a.batch) * a.T == 0) return cudaSuccess;
  if (a.dtype != ND_F32) return cudaErrorInvalidValue;
  if (a.d == 64) return launch_simt<float, 64>(a, stream);
  if (a.d == 128) return launch_simt<float, 128>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace nd
