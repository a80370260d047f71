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
  const float scale = __fdiv_rn(amax, 127.0f);
  int c[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    float r = 0.f;
    if (amax != 0.f) r = fminf(fmaxf(rintf(__fdiv_rn(x[i], scale)), -127.f), 127.f);
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

}  // namespace

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
