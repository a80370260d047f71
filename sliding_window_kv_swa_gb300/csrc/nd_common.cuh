// nd_common.cuh -- device helpers shared by the libnd kernels (sm_103a only).
//
// Bounded waits: every mbarrier wait in this library polls at most
// ND_WAIT_LIMIT times and then records flag ND_DEVERR_TIMEOUT in the
// device error word instead of spinning forever.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define ND_DEVERR_TIMEOUT 1
#define ND_DEVERR_METADATA 2

namespace nd {

// Kernels OR flags into the device error word whose address the host passes
// in (see nd_device_errors()).
__device__ __forceinline__ void raise_device_error(int *err, int flag) {
  if (err) atomicOr(err, flag);
}

constexpr uint32_t kWaitLimit = 1u << 22;  // polls of try_wait (each may sleep)

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe: has the phase with parity `parity` completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of `bar`.  Returns false (and raises the
// timeout flag) if the phase did not complete within kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *err) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  raise_device_error(err, ND_DEVERR_TIMEOUT);
  return false;
}

// ---------------------------------------------------------------- dependent launch
// Kernels launched with programmatic stream serialization may start while the
// previous kernel on the stream runs.  pdl_wait() returns once that kernel has
// completed and its writes are visible (a no-op for an ordinary launch);
// pdl_trigger() lets the next such kernel be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- conversions
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// One rotate-half pair (x_i, x_{i+d/2}) turned by the angle with cosine c and
// sine s.  The rounding order is fixed here (products rounded, then one
// fused add) so every kernel that rotates q or k produces the same bits.
__device__ __forceinline__ void rope_pair(float a, float b, float c, float s, float &ya, float &yb) {
  ya = __fmaf_rn(a, c, -__fmul_rn(b, s));
  yb = __fmaf_rn(b, c, __fmul_rn(a, s));
}

// (cos, sin) of the rotation angle pos * freq: the product and its reduction
// modulo 2 pi in double, then sincosf of the reduced angle, so the angle
// error stays ~1e-7 rad at any position.  Every kernel that rotates takes its
// angles from here (and rounds with rope_pair), so all give the same bits.
__device__ __forceinline__ float2 rot_cs(double pos, double freq) {
  const double two_pi = 6.283185307179586476925286766559, inv_two_pi = 0.15915494309189533576888376337251;
  double a = pos * freq;
  // the quotient only picks the multiple of 2 pi to subtract: multiplying by
  // 1 / (2 pi) instead of dividing can move it by one at a half-turn, which
  // still leaves |a| <= pi (+ one ulp)
  a = fma(-rint(a * inv_two_pi), two_pi, a);
  float s, c;
  sincosf(float(a), &s, &c);
  return make_float2(c, s);
}

// rint(x / scale) with the IEEE fp32 divide, bit for bit, without paying
// for the divide on almost every element: p = x * fl(1/scale) differs from
// the rounded quotient fl(x/scale) by at most |x/scale| * 1.5 * 2^-23
// <= 2.3e-5 (|x/scale| <= 127.5 for codec inputs), so rint(p) equals
// rint(fl(x/scale)) unless p lies within that distance of a half-integer;
// within 1e-4 of one (or for scales so small that 1/scale could overflow) the
// quotient is taken with the IEEE divide.  inv = __frcp_rn(scale).  The
// distance of p from the nearest half-integer is | |p - rint(p)| - 1/2 |;
// p - rint(p) and the subtraction of 1/2 are exact in fp32 wherever that
// distance is below 1/4, so rint(p) serves both the test and the result.
__device__ __forceinline__ float codec_rint(float x, float scale, float inv) {
  const float p = x * inv;
  const float r = rintf(p);
  if (fabsf(fabsf(p - r) - 0.5f) > 1e-4f && scale >= 1e-30f) return r;
  return rintf(__fdiv_rn(x, scale));
}

// The cache codec on one row of 32*CPL channels held by a full warp (lane l
// has channels [l*CPL, l*CPL + CPL)): per 32-channel group amax = max |x|
// (a shuffle over the group's 32/CPL lanes), scale = amax / 127 and
// code = clamp(rint(x / scale), +-127), both divides IEEE fp32; amax == 0
// gives scale 0 and zero codes.  Returns the scale of this lane's group.
template <int CPL>
__device__ __forceinline__ float quant_lanes(const float *x, int *code) {
  constexpr int kLanesPerGroup = 32 / CPL;
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < CPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int off = kLanesPerGroup / 2; off >= 1; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = __fdiv_rn(amax, 127.0f), inv = __frcp_rn(scale);
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    float r = 0.f;
    if (amax != 0.f) r = fminf(fmaxf(codec_rint(x[i], scale, inv), -127.f), 127.f);
    code[i] = int(r);
  }
  return scale;
}

__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Two int8 codes -> half2, exactly.  `w` holds four codes already biased to
// unsigned (code + 128, i.e. xor 0x80 per byte).  Each selected byte u becomes
// the low mantissa byte of an fp16 with exponent 2^10 (value 1024 + u); one
// packed subtract of 1152 leaves the signed code (|code| <= 127 is exact).
// sel_lo selects bytes (0,1), sel_hi bytes (2,3).
__device__ __forceinline__ uint32_t codes_to_half2(uint32_t w_biased, uint32_t sel) {
  uint32_t h = prmt(w_biased, 0x64646464u, sel);
  uint32_t r;
  const uint32_t bias = 0x64806480u;  // half2(1152, 1152)
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(bias));
  return r;
}
constexpr uint32_t kSelBytes01 = 0x5140u;  // [b0, 0x64, b1, 0x64]
constexpr uint32_t kSelBytes23 = 0x5342u;  // [b2, 0x64, b3, 0x64]

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- mma.sync
// D = A * B + C, m16n8k16, fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float &d0, float &d1, float &d2, float &d3,
                                              uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace nd
