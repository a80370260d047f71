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
// tiles of 64 are copied into shared memory with cp.async, the next tile's
// copies in flight while the current one is used; a tile is skipped when no
// row of the CTA can see any of its keys (causal bound, window bound without
// sinks, or disjoint segment-id ranges, found by warp reductions).  Eight
// keys per online-softmax step, in the log2 domain.  A problem of at most
// 256 such CTAs, which leaves most SMs idle and each CTA walking every key
// tile of its rows in turn, splits each row tile's key tiles over four CTAs
// and merges their softmax states (max, sum, weighted values) in a second
// pass.
#include "nd_common.cuh"
#include "nd_internal.h"

#include <climits>

namespace nd {

namespace {

constexpr int kTpr = 8;  // threads per query row
constexpr int kRows = 16, kKeys = 64, kThreads = kRows * kTpr;

__device__ __forceinline__ void cp_async16z(uint32_t dst, const void *src, bool valid) {
  // 16 bytes, or zeros (source size 0) for a key past the end
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Small problems split each row tile's keys over kSplit CTAs (split s takes
// key tiles s, s + kSplit, ...); each writes its rows' partial softmax state
// (max, sum, weighted values) and simt_combine_kernel merges them.
template <int D, int kSplit>
__global__ void __launch_bounds__(kThreads) prefill_simt_kernel(const PrefillArgs a, float *partials) {
  constexpr int H2 = D / kTpr;  // channels per thread
  constexpr int kTile = kKeys * D;  // floats of one K (or V) tile
  extern __shared__ __align__(16) float smem[];
  // two stages of [K tile][V tile]: the next tile's copies land while this
  // one is used
  __shared__ int s_seg[kKeys];
  __shared__ unsigned char s_sink[kKeys];
  __shared__ int s_red[3][2];
  __shared__ int s_qseg_lo, s_qseg_hi;

  const int qt = blockIdx.x, hq = blockIdx.y, b = blockIdx.z / kSplit, split = blockIdx.z % kSplit;
  const int T = a.T, G = a.Hq / a.Hkv, hk = hq / G;
  const int r = threadIdx.x / kTpr, part = threadIdx.x % kTpr;  // part: this thread's channel slice
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = qt * kRows;
  const int q = q0 + r;
  const bool row_ok = q < T;
  const int q_last = min(q0 + kRows, T) - 1;
  const float *Q = static_cast<const float *>(a.q);
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
    qr[c] = row_ok ? Q[((size_t(b) * T + q) * a.Hq + hq) * D + part * H2 + c] * qscale : 0.f;
    o[c] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  __syncthreads();
  const int qseg_lo = s_qseg_lo, qseg_hi = s_qseg_hi;
  const uint32_t sbase = smem_u32(smem);

  // One pass over a column source: pooled (src = 1) or exact keys (src = 0).
  auto run = [&](int src, int n_cols) {
    const float *KK = static_cast<const float *>(src ? a.pooled_k : a.k);
    const float *VV = static_cast<const float *>(src ? a.pooled_v : a.v);
    const int TK = src ? (T / a.block) : T;
    int col_end;  // exclusive bound on useful columns for this CTA
    if (src) {
      // largest j with (j+1)*block <= q_last - W + 1
      int lim = q_last - W + 1;
      col_end = lim >= a.block ? min(lim / a.block, n_cols) : 0;
    } else {
      col_end = q_last + 1;
    }
    const int n_tiles = (col_end + kKeys - 1) / kKeys;
    // this CTA's tiles: split, split + kSplit, ...; the i-th of them uses
    // stage i & 1
    const int n_mine = n_tiles > split ? (n_tiles - split + kSplit - 1) / kSplit : 0;
    // a thread copies 16-byte chunks idx = tid + u*kThreads of each tile
    auto stage = [&](int i) {
      const int k0 = (split + i * kSplit) * kKeys;
      const uint32_t dk = sbase + uint32_t((i & 1) * 2 * kTile) * 4, dv = dk + kTile * 4;
      constexpr int kPer = kTile / 4 / kThreads;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int idx = threadIdx.x + u * kThreads;
        const int kk = idx / (D / 4), c4 = idx % (D / 4);
        const int k = k0 + kk;
        const bool ok = k < TK;
        const size_t off = ((size_t(b) * TK + (ok ? k : 0)) * a.Hkv + hk) * D + 4 * c4;
        cp_async16z(dk + idx * 16, KK + off, ok);
        cp_async16z(dv + idx * 16, VV + off, ok);
      }
    };
    if (n_mine > 0) stage(0);
    cp_async_commit_group();
    for (int i = 0; i < n_mine; ++i) {
      const int k0 = (split + i * kSplit) * kKeys;
      // the next tile's copies go out first (one commit group per tile,
      // empty past the last)
      if (i + 1 < n_mine) stage(i + 1);
      cp_async_commit_group();
      // this tile's copies land before anything else: a skipped tile's
      // buffer takes the copies of tile t + 2 next
      cp_async_wait_group<1>();
      // ---- tile metadata and skip test (exact keys only): the tile's
      //      segment-id range and sink presence by warp reductions
      if (!src) {
        int sg = 0, sk = 0;
        if (threadIdx.x < kKeys) {
          const int k = k0 + threadIdx.x;
          sg = (k < T) ? (a.seg_ids ? a.seg_ids[size_t(b) * T + k] : 1) : 0;
          sk = (k < T && a.sink) ? a.sink[size_t(b) * T + k] : 0;
          s_seg[threadIdx.x] = sg;
          s_sink[threadIdx.x] = (unsigned char)sk;
          const int lo = __reduce_min_sync(0xffffffffu, sg > 0 ? sg : INT_MAX);
          const int hi = __reduce_max_sync(0xffffffffu, sg > 0 ? sg : INT_MIN);
          const int any = __reduce_or_sync(0xffffffffu, unsigned(sk)) != 0u;
          if (lane == 0) {
            s_red[0][warp] = lo;
            s_red[1][warp] = hi;
            s_red[2][warp] = any;
          }
        }
        __syncthreads();
        const int lo = min(s_red[0][0], s_red[0][1]), hi = max(s_red[1][0], s_red[1][1]);
        const bool any_sink = (s_red[2][0] | s_red[2][1]) != 0;
        const bool in_window = (W == 0) || (k0 + kKeys - 1 >= q0 - W + 1);
        const bool seg_overlap = lo <= qseg_hi && hi >= qseg_lo;
        if (!seg_overlap || (!in_window && !any_sink)) {
          __syncthreads();  // (the metadata is rewritten for the next tile)
          continue;
        }
      }
      __syncthreads();  // every thread's copies of this tile are visible
      const float *sk = smem + (i & 1) * 2 * kTile, *sv = sk + kTile;
      // eight keys per step: eight independent dot products, one shuffle
      // tree for all eight, then one max, one rescale and eight exponentials
      constexpr int kStepKeys = 8;
      for (int kk0 = 0; kk0 < kKeys; kk0 += kStepKeys) {
        float sc[kStepKeys];
        bool vis[kStepKeys];
#pragma unroll
        for (int u = 0; u < kStepKeys; ++u) {
          const int kk = kk0 + u, k = k0 + kk;
          if (src) {
            vis[u] = row_ok && k < n_cols && (k + 1) * a.block <= q - W + 1;
          } else {
            vis[u] = row_ok && k <= q && my_seg > 0 && s_seg[kk] == my_seg &&
                     (W == 0 || q - k < W || s_sink[kk]);
          }
          const float *kr = sk + kk * D + part * H2;
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int c = 0; c < H2; c += 2) {
            s0 = fmaf(qr[c], kr[c], s0);
            s1 = fmaf(qr[c + 1], kr[c + 1], s1);
          }
          sc[u] = s0 + s1;
        }
#pragma unroll
        for (int off = 1; off < kTpr; off <<= 1)
#pragma unroll
          for (int u = 0; u < kStepKeys; ++u) sc[u] += __shfl_xor_sync(0xffffffffu, sc[u], off);
        float mx = m;
#pragma unroll
        for (int u = 0; u < kStepKeys; ++u)
          if (vis[u]) mx = fmaxf(mx, sc[u]);
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
          if (!vis[u]) continue;
          const float pr = ex2(sc[u] - m);
          l += pr;
          const float *vr = sv + (kk0 + u) * D + part * H2;
#pragma unroll
          for (int c = 0; c < H2; ++c) o[c] = fmaf(pr, vr[c], o[c]);
        }
      }
      __syncthreads();  // the stage and the metadata are free again
    }
    cp_async_wait_group<0>();
  };

  if (a.block > 0) run(1, T / a.block);
  run(0, T);

  if (kSplit > 1) {
    // [B][Hq][T][kSplit] records of D values, then the max and the sum
    if (row_ok) {
      float *rec = partials + ((((size_t(b) * a.Hq + hq) * T + q) * kSplit) + split) * (D + 2);
#pragma unroll
      for (int c = 0; c < H2; ++c) rec[part * H2 + c] = o[c];
      if (part == 0) {
        rec[D] = m;
        rec[D + 1] = l;
      }
    }
    return;
  }
  if (row_ok) {
    float *O = static_cast<float *>(a.out);
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < H2; ++c) O[((size_t(b) * T + q) * a.Hq + hq) * D + part * H2 + c] = o[c] * inv;
    if (a.lse && part == 0)
      a.lse[(size_t(b) * a.Hq + hq) * T + q] =
          l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
  }
}

// Merge of the split partial states of one (row, channel): m = max m_s,
// l = sum l_s 2^(m_s - m), o = sum o_s 2^(m_s - m) / l (log2 domain).
template <int D, int kSplit>
__global__ void __launch_bounds__(256) simt_combine_kernel(const PrefillArgs a, const float *partials) {
  const size_t idx = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t rows = size_t(a.batch) * a.Hq * a.T;
  if (idx >= rows * D) return;
  const size_t row = idx / D;  // (b, hq, q)
  const int c = int(idx % D);
  const float *rec = partials + row * kSplit * (D + 2);
  float mx = -INFINITY;
#pragma unroll
  for (int s = 0; s < kSplit; ++s) mx = fmaxf(mx, rec[s * (D + 2) + D]);
  float l = 0.f, o = 0.f;
  if (mx != -INFINITY) {
#pragma unroll
    for (int s = 0; s < kSplit; ++s) {
      const float f = ex2(rec[s * (D + 2) + D] - mx);  // an empty split: 2^-inf = 0
      l += rec[s * (D + 2) + D + 1] * f;
      o += rec[s * (D + 2) + c] * f;
    }
  }
  const int q = int(row % a.T);
  const size_t bh = row / a.T;  // b * Hq + hq
  const int hq = int(bh % a.Hq), b = int(bh / a.Hq);
  static_cast<float *>(a.out)[((size_t(b) * a.T + q) * a.Hq + hq) * D + c] = l > 0.f ? o / l : 0.f;
  if (a.lse && c == 0) a.lse[bh * a.T + q] = l > 0.f ? (mx + __log2f(l)) * 0.6931471805599453f : -INFINITY;
}

constexpr int kSplitSmall = 4;  // key splits for problems of at most kSplitCtas row-tile CTAs
constexpr long kSplitCtas = 256;

int simt_splits(int batch, int T, int Hq) {
  const long ctas = long(batch) * Hq * ((T + kRows - 1) / kRows);
  return ctas <= kSplitCtas ? kSplitSmall : 1;
}

template <int D, int kSplit>
cudaError_t launch_simt(const PrefillArgs &a, float *partials, cudaStream_t stream) {
  const size_t smem = size_t(2) * 2 * kKeys * D * sizeof(float);  // two stages of K and V tiles
  auto kern = prefill_simt_kernel<D, kSplit>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((a.T + kRows - 1) / kRows, a.Hq, a.batch * kSplit);
  kern<<<grid, kThreads, smem, stream>>>(a, partials);
  e = cudaGetLastError();
  if (e != cudaSuccess || kSplit == 1) return e;
  const size_t n = size_t(a.batch) * a.Hq * a.T * D;
  simt_combine_kernel<D, kSplit><<<unsigned((n + 255) / 256), 256, 0, stream>>>(a, partials);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_f32_partial_bytes(int batch, int T, int Hq, int head_dim) {
  const int S = simt_splits(batch, T, Hq);
  if (S == 1) return 0;
  return (size_t(batch) * Hq * T * S * (head_dim + 2) * sizeof(float) + 255) / 256 * 256;
}

// fp32 inputs on CUDA cores (bf16 inputs always take the tensor-core kernel).
cudaError_t launch_prefill_f32(const PrefillArgs &a, void *partials, cudaStream_t stream) {
  if (size_t(a.batch) * a.T == 0) return cudaSuccess;
  if (a.dtype != ND_F32) return cudaErrorInvalidValue;
  float *pw = static_cast<float *>(partials);
  const bool split = simt_splits(a.batch, a.T, a.Hq) > 1;
  if (split && !pw) return cudaErrorInvalidValue;
  if (a.d == 64) return split ? launch_simt<64, kSplitSmall>(a, pw, stream) : launch_simt<64, 1>(a, pw, stream);
  if (a.d == 128) return split ? launch_simt<128, kSplitSmall>(a, pw, stream) : launch_simt<128, 1>(a, pw, stream);
  return cudaErrorInvalidValue;
}

}  // namespace nd
