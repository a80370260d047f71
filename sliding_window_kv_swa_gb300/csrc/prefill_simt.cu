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
// tensor-core inputs).  One CTA takes 64 query rows of one (sequence, query
// head); two threads share a row and split the head dimension.  Key tiles of
// 64 are staged in shared memory; a tile is skipped when no row of the CTA can
// see any of its keys (causal bound, window bound without sinks, or disjoint
// segment-id ranges).  Online softmax in the log2 domain.
#include "nd_common.cuh"
#include "nd_internal.h"

#include <climits>

namespace nd {

namespace {

constexpr int kRows = 64, kKeys = 64, kThreads = 128;

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
  constexpr int H2 = D / 2;
  extern __shared__ float smem[];
  float *sk = smem;                 // [kKeys][D]
  float *sv = sk + kKeys * D;       // [kKeys][D]
  __shared__ int s_seg[kKeys];
  __shared__ unsigned char s_sink[kKeys];
  __shared__ int s_qseg_lo, s_qseg_hi;

  const int qt = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
  const int T = a.T, G = a.Hq / a.Hkv, hk = hq / G;
  const int r = threadIdx.x >> 1, half = threadIdx.x & 1;
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
  if (half == 0 && row_ok && my_seg > 0) {
    atomicMin(&s_qseg_lo, my_seg);
    atomicMax(&s_qseg_hi, my_seg);
  }

  const float qscale = 1.4426950408889634f * rsqrtf(float(D));
  float qr[H2], o[H2];
#pragma unroll
  for (int c = 0; c < H2; ++c) {
    qr[c] = row_ok ? ld_elem(Q, ((size_t(b) * T + q) * a.Hq + hq) * D + half * H2 + c) * qscale : 0.f;
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
      // ---- stage K and V tile (fp32)
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
      __syncthreads();
      for (int kk = 0; kk < kKeys; ++kk) {
        const int k = k0 + kk;
        bool vis;
        if (src) {
          vis = row_ok && k < n_cols && (k + 1) * a.block <= q - W + 1;
        } else {
          vis = row_ok && k <= q && my_seg > 0 && s_seg[kk] == my_seg &&
                (W == 0 || q - k < W || s_sink[kk]);
        }
        const float *kr = sk + kk * D + half * H2;
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < H2; ++c) s = fmaf(qr[c], kr[c], s);
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        if (!vis) continue;
        if (s > m) {
          const float f = ex2(m - s);
          l *= f;
#pragma unroll
          for (int c = 0; c < H2; ++c) o[c] *= f;
          m = s;
        }
        const float pr = ex2(s - m);
        l += pr;
        const float *vr = sv + kk * D + half * H2;
#pragma unroll
        for (int c = 0; c < H2; ++c) o[c] = fmaf(pr, vr[c], o[c]);
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
      st_elem(O, ((size_t(b) * T + q) * a.Hq + hq) * D + half * H2 + c, o[c] * inv);
    if (a.lse && half == 0)
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
