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
#include <algorithm>

#include "nd_common.cuh"
#include "nd_internal.h"

#include <math.h>

namespace nd {

namespace {

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
    float ya, yb;
    rope_pair(a, b, c.x, c.y, ya, yb);
    Elem<E>::st(y, row + i, ya);
    Elem<E>::st(y, row + i + half, yb);
  }
}

// Prefill path: the (cos, sin) table of every position and channel pair is
// built once per call (double-precision reduction as above), then one thread
// rotates 8 channel pairs of one (b, t, head) with 16-byte loads and stores.
// The bf16 prefill passes K alone through it; its attention kernel rotates q
// from the same table with the same rounding (rope_pair) as it stages q.
__global__ void rope_table_kernel(float2 *cs, int T, int half, Freqs fr, int wait_first) {
  // wait_first == 0: the kernel before this one writes nothing read or
  // written here; the wait before exit keeps the chain of completions intact
  if (wait_first) pdl_wait();
  pdl_trigger();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx < T * half) cs[idx] = rot_cs(double(idx / half), fr.f[idx % half]);
  if (!wait_first) pdl_wait();
}

// The block mean's divide, x / block, bit for bit: for a power-of-two block
// the product with the exact reciprocal 2^-k is the same correctly rounded
// value (one multiply instead of an IEEE divide per channel).
struct BlockMean {
  float f, r;
  bool pow2;
  __device__ explicit BlockMean(int block)
      : f(float(block)), r(1.f / float(block)), pow2((block & (block - 1)) == 0) {}
  __device__ float operator()(float x) const { return pow2 ? __fmul_rn(x, r) : __fdiv_rn(x, f); }
};

__device__ __forceinline__ void ld8(const uint16_t *p, float *x) {
  const uint4 w = *reinterpret_cast<const uint4 *>(p);
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16_lo(u[i]);
    x[2 * i + 1] = bf16_hi(u[i]);
  }
}
__device__ __forceinline__ void st8(uint16_t *p, const float *x) {
  uint4 w;
  w.x = pack_bf16x2(x[0], x[1]);
  w.y = pack_bf16x2(x[2], x[3]);
  w.z = pack_bf16x2(x[4], x[5]);
  w.w = pack_bf16x2(x[6], x[7]);
  *reinterpret_cast<uint4 *>(p) = w;
}
__device__ __forceinline__ void ld8(const float *p, float *x) {
  const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
  x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}
__device__ __forceinline__ void st8(float *p, const float *x) {
  reinterpret_cast<float4 *>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4 *>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

// item = ((b*T + t) * (H1 + H2) + head) * (D / 16) + group of 8 pairs; heads
// below H1 come from x1 / y1, the rest from x2 / y2.
template <typename E>
__global__ void __launch_bounds__(256) rope_vec_kernel(const E *x1, E *y1, int H1, const E *x2, E *y2,
                                                       int H2, int T, int D, const float2 *cs,
                                                       size_t n_items) {
  // The table is in.  No early trigger: this grid runs many waves, and an
  // attention grid scheduled early takes whole SMs from its later waves
  // (measured 14% slower on the packed step).
  pdl_wait();
  const size_t item = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (item >= n_items) return;
  const int half = D / 2, groups = half / 8;
  const int i0 = int(item % groups) * 8;
  const size_t rest = item / groups;
  const int hh = int(rest % (H1 + H2));
  const size_t bt = rest / (H1 + H2);
  const int t = int(bt % T);
  const bool second = hh >= H1;
  const E *x = second ? x2 : x1;
  E *y = second ? y2 : y1;
  const int H = second ? H2 : H1, h = second ? hh - H1 : hh;
  const size_t row = (bt * H + h) * D;
  float a[8], b[8], c[8], s_[8];
  ld8(x + row + i0, a);
  ld8(x + row + i0 + half, b);
  const float4 *t4 = reinterpret_cast<const float4 *>(cs + size_t(t) * half + i0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 w = t4[i];
    c[2 * i] = w.x, s_[2 * i] = w.y, c[2 * i + 1] = w.z, s_[2 * i + 1] = w.w;
  }
  float ya[8], yb[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) rope_pair(a[i], b[i], c[i], s_[i], ya[i], yb[i]);
  st8(y + row + i0, ya);
  st8(y + row + i0 + half, yb);
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
    const BlockMean mean(block);
    ka = mean(ka);
    kb = mean(kb);
    va = mean(va);
    vb = mean(vb);
    float ko = ka, ko2 = kb;
    if (apply_rope) {
      const float2 c = cs[i];
      rope_pair(ka, kb, c.x, c.y, ko, ko2);
    }
    const size_t orow = ((size_t(b) * nblk + j) * H + h) * D;
    pk[orow + i] = __bfloat16_as_ushort(__float2bfloat16_rn(ko));
    pk[orow + i + half] = __bfloat16_as_ushort(__float2bfloat16_rn(ko2));
    pv[orow + i] = __bfloat16_as_ushort(__float2bfloat16_rn(va));
    pv[orow + i + half] = __bfloat16_as_ushort(__float2bfloat16_rn(vb));
  }
}

// Vector form of the pooling (head_dim a multiple of 16, 16-byte aligned
// rows): a CTA of 128 threads takes kPoolJ pooled blocks and builds their
// midpoint angles in shared memory; each thread pools 8 channel pairs
// (i0..i0+7 and i0+half..) of one (block, head) of K or of V with 16-byte
// loads -- K and V on separate threads, so a thread holds 16 sums and an SM
// keeps more loads in flight.  One block per CTA makes many small CTAs that
// all fit at once and spread evenly over the SMs (at two blocks per 256-thread
// CTA, some SMs held four CTAs and others three, and the pass ran 13% longer).
// Each thread's first rows are prefetched to L2 before the angles are built.
// The sums, the mean and the rotation follow pool_kernel's order.
constexpr int kPoolJ = 1;
// A CTA takes the same kPoolJ blocks of up to kPoolB sequences: the midpoint
// angles depend on the block only, so they are built once for all of them
// (the double-precision reduction is the costly part of the pass).
constexpr int kPoolB = 4;
__global__ void __launch_bounds__(128, 8) pool_vec_kernel(const uint16_t *k, const uint16_t *v,
                                                       uint16_t *pk, uint16_t *pv, int B, int T, int H,
                                                       int D, int block, int apply_rope, Freqs fr) {
  __shared__ float2 cs[kPoolJ][kMaxHalf];
  const int nblk = T / block, n_grp = (nblk + kPoolJ - 1) / kPoolJ;
  const int b0 = (blockIdx.x / n_grp) * kPoolB, j0 = (blockIdx.x % n_grp) * kPoolJ;
  const int nj = min(kPoolJ, nblk - j0), nbt = min(kPoolB, B - b0);
  const int half = D / 2, groups = half / 8;
  const int per_kv = nj * H * groups;
  // the first item's rows go to L2 before the angles are built, so their
  // latency overlaps the double-precision work and the barrier
  if (int(threadIdx.x) < 2 * nbt * per_kv) {
    const int idx = threadIdx.x;
    const int bi = idx / (2 * per_kv), wi = idx % (2 * per_kv);
    const bool is_v = wi >= per_kv;
    const int w = is_v ? wi - per_kv : wi;
    const int g = w % groups, rest = w / groups;
    const uint16_t *src = (is_v ? v : k) +
                          ((size_t(b0 + bi) * T + size_t(j0 + rest / H) * block) * H + rest % H) * D + g * 8;
    for (int r = 0; r < min(block, 4); ++r) {
      asm volatile("prefetch.global.L2 [%0];" ::"l"(src + size_t(r) * H * D));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(src + size_t(r) * H * D + half));
    }
  }
  if (apply_rope)
    for (int idx = threadIdx.x; idx < nj * half; idx += blockDim.x) {
      const int jj = idx / half, i = idx % half;
      const int mid = min((j0 + jj) * block + block / 2, T - 1);
      cs[jj][i] = rot_cs(double(mid), fr.f[i]);
    }
  __syncthreads();
  const BlockMean mean(block);
  for (int idx = threadIdx.x; idx < 2 * nbt * per_kv; idx += blockDim.x) {
    const int bi = idx / (2 * per_kv), wi = idx % (2 * per_kv), b = b0 + bi;
    const bool is_v = wi >= per_kv;
    const int w = is_v ? wi - per_kv : wi;
    const int g = w % groups, rest = w / groups;
    const int h = rest % H, jj = rest / H;
    const int i0 = g * 8, j = j0 + jj;
    const uint16_t *x = is_v ? v : k;
    float sa[8], sb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) sa[e] = sb[e] = 0.f;
    const size_t row0 = ((size_t(b) * T + size_t(j) * block) * H + h) * D;
    const size_t rstride = size_t(H) * D;
#pragma unroll 4
    for (int r = 0; r < block; ++r) {
      const size_t row = row0 + r * rstride;
      float xa[8], xb[8];
      ld8(x + row + i0, xa);
      ld8(x + row + i0 + half, xb);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sa[e] += xa[e];
        sb[e] += xb[e];
      }
    }
    float ya[8], yb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sa[e] = mean(sa[e]);
      sb[e] = mean(sb[e]);
      ya[e] = sa[e];
      yb[e] = sb[e];
      if (apply_rope && !is_v) {
        const float2 c = cs[jj][i0 + e];
        rope_pair(sa[e], sb[e], c.x, c.y, ya[e], yb[e]);
      }
    }
    uint16_t *y = is_v ? pv : pk;
    const size_t orow = ((size_t(b) * nblk + j) * H + h) * D;
    st8(y + orow + i0, ya);
    st8(y + orow + i0 + half, yb);
  }
}

// The compressed prefill's pass over K and V, fused: K and V are read once;
// K is written rotated at every position (k_rot, from the angle table as
// rope_vec_kernel does) and the pooled blocks are written as pool_vec_kernel
// writes them (the same sums, mean and midpoint rotation, angles from the
// same table rows).  A CTA takes kPoolJ pooled blocks of one sequence (one
// thread per (block, head, 8 channel pairs) of K or of V); one more CTA per
// sequence rotates the positions past the last whole block.  cs == NULL: no
// rotation (pooling only, k_rot untouched).
// (The output pointers never alias the inputs: __restrict__ lets every row's
// loads go out before the first rotated row is stored.)
constexpr int kPoolRows = 4;  // rows of a block loaded before any is used
__global__ void __launch_bounds__(256) pool_rope_kernel(const uint16_t *__restrict__ k,
                                                        const uint16_t *__restrict__ v,
                                                        uint16_t *__restrict__ k_rot, uint16_t *__restrict__ pk,
                                                        uint16_t *__restrict__ pv, int T, int H, int D, int block,
                                                        int pos0, const float2 *__restrict__ cs) {
  pdl_wait();  // the angle table (or what the previous kernel wrote) is in
  // blocks tile positions pos0 .. pos0 + nblk*block - 1; the positions
  // before pos0 and past the last whole block are rotated by one more CTA
  const int nblk = (T - pos0) / block, n_grp = (nblk + kPoolJ - 1) / kPoolJ;
  const int tail = T - pos0 - nblk * block, n_rest = pos0 + tail;
  const int per_seq = n_grp + (n_rest > 0 ? 1 : 0);
  const int b = blockIdx.x / per_seq, grp = blockIdx.x % per_seq;
  const int half = D / 2, groups = half / 8;
  const size_t rstride = size_t(H) * D;
  auto rotate8 = [&](int t, int i0, const float *a, const float *bb, float *ya, float *yb) {
    const float4 *t4 = reinterpret_cast<const float4 *>(cs + size_t(t) * half + i0);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const float4 w = t4[q4];
      rope_pair(a[2 * q4], bb[2 * q4], w.x, w.y, ya[2 * q4], yb[2 * q4]);
      rope_pair(a[2 * q4 + 1], bb[2 * q4 + 1], w.z, w.w, ya[2 * q4 + 1], yb[2 * q4 + 1]);
    }
  };
  if (grp == n_grp) {  // positions outside the blocks: K's rotation only
    if (!cs) return;
    for (int idx = threadIdx.x; idx < n_rest * H * groups; idx += blockDim.x) {
      const int g = idx % groups, rest = idx / groups;
      const int h = rest % H, u = rest / H, i0 = g * 8;
      const int t = u < pos0 ? u : pos0 + nblk * block + (u - pos0);
      const size_t row = (size_t(b) * T + t) * rstride + size_t(h) * D;
      float xa[8], xb[8], ya[8], yb[8];
      ld8(k + row + i0, xa);
      ld8(k + row + i0 + half, xb);
      rotate8(t, i0, xa, xb, ya, yb);
      st8(k_rot + row + i0, ya);
      st8(k_rot + row + i0 + half, yb);
    }
    return;
  }
  const int j0 = grp * kPoolJ, nj = min(kPoolJ, nblk - j0);
  const BlockMean mean(block);
  const int per_kv = nj * H * groups;
  for (int idx = threadIdx.x; idx < 2 * per_kv; idx += blockDim.x) {
    const bool is_v = idx >= per_kv;
    const int w = is_v ? idx - per_kv : idx;
    const int g = w % groups, rest = w / groups;
    const int h = rest % H, j = j0 + rest / H;
    const int i0 = g * 8;
    const uint16_t *x = is_v ? v : k;
    float sa[8], sb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) sa[e] = sb[e] = 0.f;
    const size_t row0 = (size_t(b) * T + pos0 + size_t(j) * block) * rstride + size_t(h) * D;
    for (int r0 = 0; r0 < block; r0 += kPoolRows) {
      uint4 ra[kPoolRows], rb[kPoolRows];
#pragma unroll
      for (int r = 0; r < kPoolRows; ++r)
        if (r0 + r < block) {
          const size_t row = row0 + size_t(r0 + r) * rstride;
          ra[r] = *reinterpret_cast<const uint4 *>(x + row + i0);
          rb[r] = *reinterpret_cast<const uint4 *>(x + row + i0 + half);
        }
#pragma unroll
      for (int r = 0; r < kPoolRows; ++r) {
        if (r0 + r >= block) break;
        float xa[8], xb[8];
        const uint32_t ua[4] = {ra[r].x, ra[r].y, ra[r].z, ra[r].w}, ub[4] = {rb[r].x, rb[r].y, rb[r].z, rb[r].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          xa[2 * e] = bf16_lo(ua[e]), xa[2 * e + 1] = bf16_hi(ua[e]);
          xb[2 * e] = bf16_lo(ub[e]), xb[2 * e + 1] = bf16_hi(ub[e]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          sa[e] += xa[e];
          sb[e] += xb[e];
        }
        if (cs && !is_v) {
          const size_t row = row0 + size_t(r0 + r) * rstride;
          float ya[8], yb[8];
          rotate8(pos0 + j * block + r0 + r, i0, xa, xb, ya, yb);
          st8(k_rot + row + i0, ya);
          st8(k_rot + row + i0 + half, yb);
        }
      }
    }
    float ya[8], yb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sa[e] = mean(sa[e]);
      sb[e] = mean(sb[e]);
      ya[e] = sa[e];
      yb[e] = sb[e];
    }
    if (cs && !is_v) rotate8(min(pos0 + j * block + block / 2, T - 1), i0, sa, sb, ya, yb);
    uint16_t *y = is_v ? pv : pk;
    const size_t orow = ((size_t(b) * nblk + j) * H + h) * D;
    st8(y + orow + i0, ya);
    st8(y + orow + i0 + half, yb);
  }
}

// The fused pass fed by bulk copies.  The rows of nj_max consecutive pooled
// blocks of one sequence are one contiguous stretch of K, of V and of the
// angle table, so one thread moves each stretch into shared memory with a
// single cp.async.bulk; a ring of kBulkStages chunks keeps the next ones in
// flight while all threads work from shared memory: K rows rotated and
// stored, K and V pooled, pooled K rotated at the block midpoint (one thread
// per (block, head, 8 channel pairs) of K or of V, so a CTA has as many
// threads as a chunk has such lanes, up to 256).  The CTAs are persistent
// and walk the chunks with a stride of the grid, then rotate the positions
// outside whole blocks.  A chunk is one pooled block: small chunks and small
// CTAs put four CTAs on an SM, which measured faster than chunks of four
// blocks at two CTAs per SM; two stages measured faster than three.  Sums,
// means, angles and roundings are those of pool_rope_kernel, so the results
// are the same bits.
constexpr int kBulkStages = 2;
constexpr int kBulkBytes = 16384;  // K (and V) bytes per chunk, at most
constexpr int kBulkMaxJ = 1;       // pooled blocks per chunk, at most
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void lds4(uint32_t addr, uint32_t *w) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
}
__global__ void __launch_bounds__(256) pool_rope_bulk_kernel(const uint16_t *__restrict__ k,
                                                             const uint16_t *__restrict__ v,
                                                             uint16_t *__restrict__ k_rot, uint16_t *__restrict__ pk,
                                                             uint16_t *__restrict__ pv, int B, int T, int H, int D,
                                                             int block, int pos0, int nj_max,
                                                             const float2 *__restrict__ cs, int *err) {
  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ __align__(8) uint64_t full[kBulkStages];
  pdl_wait();  // the angle table (or what the previous kernel wrote) is in
  const int nblk = (T - pos0) / block, per_seq = (nblk + nj_max - 1) / nj_max, n_chunks = B * per_seq;
  const int half = D / 2, groups = half / 8;
  const uint32_t row_bytes = uint32_t(H) * D * 2, tensor_bytes = uint32_t(nj_max) * block * row_bytes;
  const uint32_t cs_row = uint32_t(half) * 8, cs_bytes = cs ? uint32_t(nj_max) * block * cs_row : 0u;
  const uint32_t stage_bytes = 2 * tensor_bytes + cs_bytes;
  const uint32_t base = smem_u32(stage_mem);
  const size_t rstride = size_t(H) * D;
  auto chunk = [&](int c, int &b, int &j0, int &nj) {
    b = c / per_seq;
    j0 = (c % per_seq) * nj_max;
    nj = min(nj_max, nblk - j0);
  };
  auto issue = [&](int c, int st) {  // one thread
    int b, j0, nj;
    chunk(c, b, j0, nj);
    const int t0 = pos0 + j0 * block;
    const uint32_t bytes = uint32_t(nj) * block * row_bytes, cb = cs ? uint32_t(nj) * block * cs_row : 0u;
    const size_t off = (size_t(b) * T + t0) * rstride;
    const uint32_t dst = base + st * stage_bytes;
    mbar_arrive_expect_tx(&full[st], 2 * bytes + cb);
    bulk_g2s(dst, k + off, bytes, &full[st]);
    bulk_g2s(dst + tensor_bytes, v + off, bytes, &full[st]);
    if (cs) bulk_g2s(dst + 2 * tensor_bytes, cs + size_t(t0) * half, cb, &full[st]);
  };
  if (threadIdx.x == 0) {
    for (int st = 0; st < kBulkStages; ++st) mbar_init(&full[st], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    for (int i = 0; i < kBulkStages; ++i)
      if (blockIdx.x + i * gridDim.x < n_chunks) issue(blockIdx.x + i * gridDim.x, i);
  // (the plain divide for the mean, not BlockMean: the multiply frees
  // registers, the occupancy query then gives six CTAs per SM instead of
  // four, and that grid measured slower; the results are the same bits)
  const float fblock = float(block);
  bool ok = true;
  for (int i = 0, c = blockIdx.x; c < n_chunks && ok; ++i, c += gridDim.x) {
    const int st = i % kBulkStages;
    int b, j0, nj;
    chunk(c, b, j0, nj);
    const uint32_t par = (i / kBulkStages) & 1;
    ok = mbar_test_wait(&full[st], par) || mbar_wait(&full[st], par, err);
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }
    const uint32_t sk = base + st * stage_bytes, scs = sk + 2 * tensor_bytes;
    const int per_kv = nj * H * groups;
    for (int idx = threadIdx.x; idx < 2 * per_kv; idx += blockDim.x) {
      const bool is_v = idx >= per_kv;
      const int w = is_v ? idx - per_kv : idx;
      const int g = w % groups, rest = w / groups;
      const int h = rest % H, jj = rest / H;
      const int i0 = g * 8;
      const bool rot = cs && !is_v;
      float sa[8], sb[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) sa[e] = sb[e] = 0.f;
      const uint32_t src = sk + (is_v ? tensor_bytes : 0u) + uint32_t(jj * block) * row_bytes + uint32_t(h * D + i0) * 2;
      // rotated rotation angles of this row's pairs: 8 float2 at (row, i0)
      auto angles = [&](int r, float *cc, float *ss) {
        uint32_t wv[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          lds4(scs + uint32_t(jj * block + r) * cs_row + uint32_t(i0 + 2 * q4) * 8, wv);
          cc[2 * q4] = __uint_as_float(wv[0]), ss[2 * q4] = __uint_as_float(wv[1]);
          cc[2 * q4 + 1] = __uint_as_float(wv[2]), ss[2 * q4 + 1] = __uint_as_float(wv[3]);
        }
      };
      const size_t grow0 = (size_t(b) * T + pos0 + size_t(j0 + jj) * block) * rstride + size_t(h) * D;
      for (int r = 0; r < block; ++r) {
        uint32_t a[4], bb[4];
        lds4(src + r * row_bytes, a);
        lds4(src + r * row_bytes + half * 2, bb);
        float xa[8], xb[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          xa[2 * e] = bf16_lo(a[e]), xa[2 * e + 1] = bf16_hi(a[e]);
          xb[2 * e] = bf16_lo(bb[e]), xb[2 * e + 1] = bf16_hi(bb[e]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          sa[e] += xa[e];
          sb[e] += xb[e];
        }
        if (rot) {
          float cc[8], ss[8], ya[8], yb[8];
          angles(r, cc, ss);
#pragma unroll
          for (int e = 0; e < 8; ++e) rope_pair(xa[e], xb[e], cc[e], ss[e], ya[e], yb[e]);
          st8(k_rot + grow0 + size_t(r) * rstride + i0, ya);
          st8(k_rot + grow0 + size_t(r) * rstride + i0 + half, yb);
        }
      }
      float ya[8], yb[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sa[e] /= fblock;
        sb[e] /= fblock;
        ya[e] = sa[e];
        yb[e] = sb[e];
      }
      if (rot) {  // the midpoint row j*block + block/2 lies inside the block
        float cc[8], ss[8];
        angles(block / 2, cc, ss);
#pragma unroll
        for (int e = 0; e < 8; ++e) rope_pair(sa[e], sb[e], cc[e], ss[e], ya[e], yb[e]);
      }
      uint16_t *y = is_v ? pv : pk;
      const size_t orow = ((size_t(b) * nblk + j0 + jj) * H + h) * D;
      st8(y + orow + i0, ya);
      st8(y + orow + i0 + half, yb);
    }
    __syncthreads();  // the stage is free again
    if (threadIdx.x == 0 && c + kBulkStages * int(gridDim.x) < n_chunks) {
      // the async-proxy refill follows the threads' generic-proxy reads
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(c + kBulkStages * gridDim.x, st);
    }
  }
  if (!ok) {  // a copy that never landed: give any still in flight time to land before the CTA exits
    for (int i = 0; i < 2000; ++i) __nanosleep(1000);
    return;
  }
  // positions before pos0 and past the last whole block: K's rotation only
  if (!cs) return;
  const int tail = T - pos0 - nblk * block, n_rest = pos0 + tail;
  const size_t n_items = size_t(B) * n_rest * H * groups;
  for (size_t idx = size_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < n_items; idx += size_t(gridDim.x) * blockDim.x) {
    const int g = int(idx % groups);
    size_t rest = idx / groups;
    const int h = int(rest % H);
    rest /= H;
    const int u = int(rest % n_rest), b = int(rest / n_rest), i0 = g * 8;
    const int t = u < pos0 ? u : pos0 + nblk * block + (u - pos0);
    const size_t row = (size_t(b) * T + t) * rstride + size_t(h) * D;
    float xa[8], xb[8], ya[8], yb[8];
    ld8(k + row + i0, xa);
    ld8(k + row + i0 + half, xb);
    const float4 *t4 = reinterpret_cast<const float4 *>(cs + size_t(t) * half + i0);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const float4 wv = t4[q4];
      rope_pair(xa[2 * q4], xb[2 * q4], wv.x, wv.y, ya[2 * q4], yb[2 * q4]);
      rope_pair(xa[2 * q4 + 1], xb[2 * q4 + 1], wv.z, wv.w, ya[2 * q4 + 1], yb[2 * q4 + 1]);
    }
    st8(k_rot + row + i0, ya);
    st8(k_rot + row + i0 + half, yb);
  }
}

}  // namespace

// The angle table (when theta != 0), then the fused pass; the table kernel
// is chained as in launch_rope_qk.  head_dim a multiple of 16, 16-byte
// aligned tensors.
cudaError_t launch_pool_rope(const void *k, const void *v, void *k_rot, void *pk, void *pv, int batch, int T,
                             int n_heads, int head_dim, int block, int pos0, float theta, void *table, bool chained,
                             cudaStream_t stream) {
  if (size_t(batch) * T == 0) return cudaSuccess;
  float2 *cs = nullptr;
  if (theta != 0.f) {
    Freqs fr = make_freqs(head_dim, theta);
    cs = static_cast<float2 *>(table);
    const int half = head_dim / 2;
    cudaError_t e = launch_pdl(rope_table_kernel, dim3((T * half + 255) / 256), dim3(256), 0, stream, cs, T,
                               half, fr, chained ? 0 : 1);
    if (e != cudaSuccess) return e;
  }
  const int nblk = (T - pos0) / block, n_grp = (nblk + kPoolJ - 1) / kPoolJ;
  const size_t block_bytes = size_t(block) * n_heads * head_dim * 2;
  if (nblk > 0 && block_bytes <= size_t(kBulkBytes)) {
    const int nj_max = int(std::min<size_t>(kBulkMaxJ, kBulkBytes / block_bytes));
    const int n_chunks = batch * ((nblk + nj_max - 1) / nj_max);
    const size_t stage = 2 * nj_max * block_bytes + (cs ? size_t(nj_max) * block * (head_dim / 2) * 8 : 0);
    const int smem = int(kBulkStages * stage);
    cudaError_t e = cudaFuncSetAttribute(pool_rope_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    int sms = 0, dev = 0, per_sm = 0;
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int lanes = nj_max * n_heads * head_dim / 8, threads = std::min(256, (lanes + 31) / 32 * 32);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pool_rope_bulk_kernel, threads, smem);
    if (e != cudaSuccess) return e;
    const int grid = std::min(n_chunks, std::max(1, per_sm) * sms);
    return launch_pdl(pool_rope_bulk_kernel, dim3(unsigned(grid)), dim3(unsigned(threads)), size_t(smem), stream,
                      static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(v),
                      static_cast<uint16_t *>(k_rot), static_cast<uint16_t *>(pk), static_cast<uint16_t *>(pv), batch,
                      T, n_heads, head_dim, block, pos0, nj_max, static_cast<const float2 *>(cs),
                      device_error_word());
  }
  const int per_seq = n_grp + (T - nblk * block > 0 ? 1 : 0);
  if (per_seq == 0) return cudaSuccess;
  return launch_pdl(pool_rope_kernel, dim3(unsigned(size_t(batch) * per_seq)), dim3(256), 0, stream,
                    static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(v), static_cast<uint16_t *>(k_rot),
                    static_cast<uint16_t *>(pk), static_cast<uint16_t *>(pv), T, n_heads, head_dim, block, pos0,
                    static_cast<const float2 *>(cs));
}

Freqs make_freqs(int D, float theta) {
  Freqs fr;
  for (int i = 0; i < kMaxHalf; ++i)
    fr.f[i] = (i < D / 2) ? pow(double(theta), -2.0 * double(i) / double(D)) : 0.0;
  return fr;
}

cudaError_t launch_rope(const void *x, void *y, int batch, int T, int n_heads, int head_dim,
                        float theta, cudaStream_t stream) {
  if (size_t(batch) * T == 0) return cudaSuccess;
  Freqs fr = make_freqs(head_dim, theta);
  rope_kernel<uint16_t><<<batch * T, 128, 0, stream>>>(
      static_cast<const uint16_t *>(x), static_cast<uint16_t *>(y), n_heads, nullptr, nullptr, 0, T,
      head_dim, fr);
  return cudaGetLastError();
}

size_t rope_table_bytes(int T, int head_dim) { return size_t(T) * (head_dim / 2) * sizeof(float2); }

// Rotate q (when Hq > 0) and k of a prefill into separate output buffers: the
// angle table into `table` (rope_table_bytes), then one vectorised pass;
// both are dependent launches.  head_dim must be a multiple of 16.
cudaError_t launch_rope_qk(const void *q, void *q_out, int Hq, const void *k, void *k_out, int Hkv,
                           int batch, int T, int head_dim, float theta, bool f32, void *table,
                           bool chained, cudaStream_t stream) {
  if (size_t(batch) * T == 0) return cudaSuccess;
  Freqs fr = make_freqs(head_dim, theta);
  float2 *cs = static_cast<float2 *>(table);
  const int half = head_dim / 2;
  cudaError_t e = launch_pdl(rope_table_kernel, dim3((T * half + 255) / 256), dim3(256), 0, stream, cs, T,
                             half, fr, chained ? 0 : 1);
  if (e != cudaSuccess) return e;
  const size_t n = size_t(batch) * T * (Hq + Hkv) * (half / 8);
  const dim3 grid(unsigned((n + 255) / 256));
  if (f32)
    return launch_pdl(rope_vec_kernel<float>, grid, dim3(256), 0, stream, static_cast<const float *>(q),
                      static_cast<float *>(q_out), Hq, static_cast<const float *>(k),
                      static_cast<float *>(k_out), Hkv, T, head_dim, static_cast<const float2 *>(cs), n);
  return launch_pdl(rope_vec_kernel<uint16_t>, grid, dim3(256), 0, stream, static_cast<const uint16_t *>(q),
                    static_cast<uint16_t *>(q_out), Hq, static_cast<const uint16_t *>(k),
                    static_cast<uint16_t *>(k_out), Hkv, T, head_dim, static_cast<const float2 *>(cs), n);
}

cudaError_t launch_compress_pool(const void *k, const void *v, int batch, int T, int n_heads,
                                 int head_dim, int block, float theta, void *pk, void *pv,
                                 cudaStream_t stream) {
  const int nblk = T / block;
  if (size_t(batch) * nblk == 0) return cudaSuccess;
  Freqs fr = make_freqs(head_dim, theta);
  const bool vec = head_dim % 16 == 0 && ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
                                           reinterpret_cast<uintptr_t>(pk) | reinterpret_cast<uintptr_t>(pv)) &
                                          15) == 0;
  if (vec) {
    const int n_grp = (nblk + kPoolJ - 1) / kPoolJ;
    pool_vec_kernel<<<((batch + kPoolB - 1) / kPoolB) * n_grp, 128, 0, stream>>>(
        static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(v), static_cast<uint16_t *>(pk),
        static_cast<uint16_t *>(pv), batch, T, n_heads, head_dim, block, theta != 0.f ? 1 : 0, fr);
    return cudaGetLastError();
  }
  pool_kernel<<<batch * nblk, 128, 0, stream>>>(
      static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(v),
      static_cast<uint16_t *>(pk), static_cast<uint16_t *>(pv), T, n_heads, head_dim, block,
      theta != 0.f ? 1 : 0, fr);
  return cudaGetLastError();
}

}  // namespace nd
