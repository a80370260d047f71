// rope_pool.cu -- rotary embedding of q/k and block pooling with midpoint
// rotation, both HBM-bound elementwise kernels.
//
// "Compressed attention and the copy probe", section "Pool before rotating,
// not after": K and V are mean-pooled over blocks of `block` positions before
// any rotation, each pooled key is rotated once at its block midpoint
// j*block + block/2 (clamped to the table), and q / k are rotated at their own
// positions.  Rotation convention (the pages do not print apply_rope):
// rotate-half, channel pairs (i, i + d/2), angle = pos * theta^(-2i/d).
//
// Angles: theta^(-2i/d) is computed once on the host in double and passed in;
// pos * freq and the reduction mod 2*pi are done in double (two flops per
// (position, pair), amortised over every head), then sincosf on the reduced
// angle, so the rotation error is ~1e-7 rad even at position 4095.
#include "nd_common.cuh"
#include "nd_internal.h"

#include <math.h>

namespace nd {

namespace {

constexpr int kMaxHalf = 128;  // head_dim <= 256

struct Freqs {
  double f[kMaxHalf];
};

__device__ __forceinline__ float2 rot_cs(double pos, double freq) {
  const double two_pi = 6.283185307179586476925286766559;
  double a = pos * freq;
  a -= rint(a / two_pi) * two_pi;
  float s, c;
  sincosf(float(a), &s, &c);
  return make_float2(c, s);
}

template <typename E>
struct Elem;
template <>
struct Elem<uint16_t> {
  __device__ static float ld(const uint16_t *p, size_t i) { return __uint_as_float(uint32_t(p[i]) << 16); }
  __device__ static void st(uint16_t *p, size_t i, float x) {
    p[i] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
};
template <>
struct Elem<float> {
  __device__ static float ld(const float *p, size_t i) { return p[i]; }
  __device__ static void st(float *p, size_t i, float x) { p[i] = x; }
};

// One CTA per (b, t): the angle table for position t sits in shared memory and
// is applied to every head of up to two tensors (q with H1 heads, k with H2).
template <typename E>
__global__ void __launch_bounds__(128) rope_kernel(const E *x1, E *y1, int H1, const E *x2, E *y2,
                                                   int H2, int T, int D, Freqs fr) {
  __shared__ float2 cs[kMaxHalf];
  const int bt = blockIdx.x;
  const int t = bt % T;
  const int half = D / 2;
  for (int i = threadIdx.x; i < half; i += blockDim.x) cs[i] = rot_cs(double(t), fr.f[i]);
  __syncthreads();
  const int n1 = H1 * half, n = n1 + H2 * half;
  for (int idx = threadIdx.x; idx < n; idx += blockDim.x) {
    const bool second = idx >= n1;
    const int j = second ? idx - n1 : idx;
    const int h = j / half, i = j % half;
    const E *x = second ? x2 : x1;
    E *y = second ? y2 : y1;
    const int H = second ? H2 : H1;
    const size_t row = (size_t(bt) * H + h) * D;
    const float a = Elem<E>::ld(x, row + i), b = Elem<E>::ld(x, row + i + half);
    const float2 c = cs[i];
    Elem<E>::st(y, row + i, a * c.x - b * c.y);
    Elem<E>::st(y, row + i + half, b * c.x + a * c.y);
  }
}

// One CTA per (b, pooled block j): mean of `block` consecutive positions for
// every head and channel, K rotated at the block midpoint.
__global__ void __launch_bounds__(128) pool_kernel(const uint16_t *k, const uint16_t *v,
                                                   uint16_t *pk, uint16_t *pv, int T, int H, int D,
                                                   int block, int apply_rope, Freqs fr) {
  __shared__ float2 cs[kMaxHalf];
  const int nblk = T / block;
  const int b = blockIdx.x / nblk, j = blockIdx.x % nblk;
  const int half = D / 2;
  int mid = j * block + block / 2;
  if (mid > T - 1) mid = T - 1;
  if (apply_rope)
    for (int i = threadIdx.x; i < half; i += blockDim.x) cs[i] = rot_cs(double(mid), fr.f[i]);
  __syncthreads();
  for (int idx = threadIdx.x; idx < H * half; idx += blockDim.x) {
    const int h = idx / half, i = idx % half;
    float ka = 0.f, kb = 0.f, va = 0.f, vb = 0.f;
    for (int r = 0; r < block; ++r) {
      const size_t row = ((size_t(b) * T + size_t(j) * block + r) * H + h) * D;
      ka += __uint_as_float(uint32_t(k[row + i]) << 16);
      kb += __uint_as_float(uint32_t(k[row + i + half]) << 16);
      va += __uint_as_float(uint32_t(v[row + i]) << 16);
      vb += __uint_as_float(uint32_t(v[row + i + half]) << 16);
    }
    ka /= float(block);
    kb /= float(block);
    va /= float(block);
    vb /= float(block);
    float ko = ka, ko2 = kb;
    if (apply_rope) {
      const float2 c = cs[i];
      ko = ka * c.x - kb * c.y;
      ko2 = kb * c.x + ka * c.y;
    }
    const size_t orow = ((size_t(b) * nblk + j) * H + h) * D;
    pk[orow + i] = __bfloat16_as_ushort(__float2bfloat16_rn(ko));
    pk[orow + i + half] = __bfloat16_as_ushort(__float2bfloat16_rn(ko2));
    pv[orow + i] = __bfloat16_as_ushort(__float2bfloat16_rn(va));
    pv[orow + i + half] = __bfloat16_as_ushort(__float2bfloat16_rn(vb));
  }
}

Freqs make_freqs(int D, float theta) {
  Freqs fr;
  for (int i = 0; i < kMaxHalf; ++i)
    fr.f[i] = (i < D / 2) ? pow(double(theta), -2.0 * double(i) / double(D)) : 0.0;
  return fr;
}

}  // namespace

cudaError_t launch_rope(const void *x, void *y, int batch, int T, int n_heads, int head_dim,
                        float theta, cudaStream_t stream) {
  if (size_t(batch) * T == 0) return cudaSuccess;
  Freqs fr = make_freqs(head_dim, theta);
  rope_kernel<uint16_t><<<batch * T, 128, 0, stream>>>(
      static_cast<const uint16_t *>(x), static_cast<uint16_t *>(y), n_heads, nullptr, nullptr, 0, T,
      head_dim, fr);
  return cudaGetLastError();
}

// Rotate q and k of a prefill into separate output buffers in one launch.
cudaError_t launch_rope_qk(const void *q, void *q_out, int Hq, const void *k, void *k_out, int Hkv,
                           int batch, int T, int head_dim, float theta, bool f32,
                           cudaStream_t stream) {
  if (size_t(batch) * T == 0) return cudaSuccess;
  Freqs fr = make_freqs(head_dim, theta);
  if (f32)
    rope_kernel<float><<<batch * T, 128, 0, stream>>>(
        static_cast<const float *>(q), static_cast<float *>(q_out), Hq,
        static_cast<const float *>(k), static_cast<float *>(k_out), Hkv, T, head_dim, fr);
  else
    rope_kernel<uint16_t><<<batch * T, 128, 0, stream>>>(
        static_cast<const uint16_t *>(q), static_cast<uint16_t *>(q_out), Hq,
        static_cast<const uint16_t *>(k), static_cast<uint16_t *>(k_out), Hkv, T, head_dim, fr);
  return cudaGetLastError();
}

cudaError_t launch_compress_pool(const void *k, const void *v, int batch, int T, int n_heads,
                                 int head_dim, int block, float theta, void *pk, void *pv,
                                 cudaStream_t stream) {
  const int nblk = T / block;
  if (size_t(batch) * nblk == 0) return cudaSuccess;
  Freqs fr = make_freqs(head_dim, theta);
  pool_kernel<<<batch * nblk, 128, 0, stream>>>(
      static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(v),
      static_cast<uint16_t *>(pk), static_cast<uint16_t *>(pv), T, n_heads, head_dim, block,
      theta != 0.f ? 1 : 0, fr);
  return cudaGetLastError();
}

}  // namespace nd
