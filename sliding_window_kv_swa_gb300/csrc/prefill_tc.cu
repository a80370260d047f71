// prefill_tc.cu -- bf16 prefill attention on the 5th-generation tensor cores
// (tcgen05 MMAs with TMEM accumulators, TMA-staged tiles), for the mask of
// "How the 256-Token Sliding Window Works with Tools as KV Sinks in Needle",
// section "KV Sinks for Tools" (same segment, causal, window or sink), and for
// the compressed columns of "Compressed attention and the copy probe", section
// "Two kinds of columns" (pooled block j visible iff (j+1)*block <= q-W+1,
// then the exact sliding window).
//
// Work split.  A small plan pass lists, for every (sequence, 128-row query
// tile), the 64-key tiles that can hold a visible key (segment-id ranges,
// causal bound, window bound, sink presence; pooled tiles below the threshold),
// so the cost follows window + sink rather than T^2.  One CTA (4 warps) then
// runs one (sequence, query tile, query head):
//   TMA   : Q tile [128 x d] once; K and V tiles [64 x d] double-buffered,
//           128-byte swizzled, issued by one thread on mbarriers.
//   MMA   : S = Q K^T (M=128, N=64) into TMEM; O_tile = P V (M=128, N=d) into
//           TMEM, P read from shared memory (K-major), V as an MN-major
//           operand straight from its TMA tile.  One thread issues, commits
//           to an mbarrier.
//   softmax: thread i owns query row i = TMEM lane i: loads its S row,
//           applies the exact mask, online softmax in the log2 domain,
//           writes bf16 P, and accumulates O = O*alpha + O_tile in registers.
// Every mbarrier wait is bounded; on timeout the CTA raises the device error
// flag, stops issuing work and frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>

#include "nd_common.cuh"
#include "nd_internal.h"

namespace nd {

namespace {

constexpr int BM = 128;  // query rows per CTA = TMEM lanes
constexpr int BN = 64;   // keys per tile
constexpr int kThreads = 128;

struct TileSummary {
  int seg_lo, seg_hi, any_sink;
};

struct TcParams {
  int B, T, Hq, Hkv, G, W, block, nb, n_qt, n_kt, n_pt, plan_stride;
  const int32_t *seg;
  const uint8_t *sink;
  const int32_t *plan;
  uint16_t *out;
  float *lse;
  int *err;
};

// ------------------------------------------------------------------ plan

__global__ void tile_summary_kernel(const int32_t *seg, const uint8_t *sink, int T, int n_kt,
                                    TileSummary *sum, int B) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B * n_kt) return;
  const int b = i / n_kt, j = i % n_kt;
  int lo = INT_MAX, hi = INT_MIN, any = 0;
  for (int k = j * BN; k < min(T, (j + 1) * BN); ++k) {
    const int s = seg ? seg[size_t(b) * T + k] : 1;
    if (s > 0) {
      lo = min(lo, s);
      hi = max(hi, s);
    }
    if (sink) any |= sink[size_t(b) * T + k] != 0;
  }
  sum[i] = {lo, hi, any};
}

__global__ void tile_plan_kernel(const int32_t *seg, const TileSummary *sum, TcParams p,
                                 int32_t *plan) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= p.B * p.n_qt) return;
  const int b = i / p.n_qt, qt = i % p.n_qt;
  const int q0 = qt * BM, q1 = min(p.T, q0 + BM) - 1;
  int32_t *out = plan + size_t(i) * p.plan_stride;
  int n = 0;
  if (p.block > 0) {
    // pooled columns j < nb visible from some row iff (j+1)*block <= q1 - W + 1
    const int lim = q1 - p.W + 1;
    const int ncol = lim >= p.block ? min(lim / p.block, p.nb) : 0;
    for (int j = 0; j * BN < ncol; ++j) out[1 + n++] = (1 << 20) | j;
  }
  int qlo = INT_MAX, qhi = INT_MIN;
  for (int q = q0; q <= q1; ++q) {
    const int s = seg ? seg[size_t(b) * p.T + q] : 1;
    if (s > 0) {
      qlo = min(qlo, s);
      qhi = max(qhi, s);
    }
  }
  if (qlo <= qhi) {
    for (int j = 0; j * BN <= q1; ++j) {
      const TileSummary t = sum[size_t(b) * p.n_kt + j];
      if (t.seg_lo > t.seg_hi || t.seg_lo > qhi || t.seg_hi < qlo) continue;
      const bool in_window = p.W == 0 || (j + 1) * BN - 1 >= q0 - p.W + 1;
      if (!in_window && !t.any_sink) continue;
      out[1 + n++] = j;
    }
  }
  out[0] = n;
}

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;  // descriptor version for sm_100 family
  d |= uint64_t(2) << 61;  // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: bf16 A and B, fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(b_mn_major) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ kernel

template <int D>
struct Smem {
  static constexpr int kBoxes = D / 64;                // 64-column swizzle atoms per row
  static constexpr int kQ = kBoxes * BM * 128;         // Q tile bytes
  static constexpr int kKV = kBoxes * BN * 128;        // one K (or V) tile
  static constexpr int kP = BM * BN * 2;               // P tile (one atom column)
  static constexpr bool kAliasP = (kKV == kP);         // P reuses the consumed K stage
  static constexpr int kBytes = kQ + 4 * kKV + (kAliasP ? 0 : kP) + 1024;  // + alignment slack
  static constexpr int kTmemCols = (BN + D) <= 128 ? 128 : 256;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_pk,
                      const __grid_constant__ CUtensorMap tm_pv, const TcParams p) {
  using L = Smem<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q, bar_kv[2], bar_s, bar_o;
  __shared__ uint32_t s_tmem;
  bool fail = false, aborted = false;  // this thread saw a wait time out; the CTA did
  __shared__ int s_seg[2][BN];
  __shared__ unsigned char s_sink[2][BN];

  const int qt = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int hk = hq / p.G;
  const int q0 = qt * BM;
  const int q = q0 + tid;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;
  const uint32_t sK[2] = {base + L::kQ, base + L::kQ + L::kKV};
  const uint32_t sV[2] = {base + L::kQ + 2 * L::kKV, base + L::kQ + 3 * L::kKV};
  const uint32_t sPsep = base + L::kQ + 4 * L::kKV;

  const int32_t *plan = p.plan + (size_t(b) * p.n_qt + qt) * p.plan_stride;
  const int n_tiles = plan[0];

  if (tid == 0) {
    mbar_init(&bar_q, 1);
    mbar_init(&bar_kv[0], 1);
    mbar_init(&bar_kv[1], 1);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_o, 1);

    fence_barrier_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s_tmem)),
                 "r"(L::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t tS = tmem, tO = tmem + BN;
  const uint32_t lane_base = uint32_t(warp * 32) << 16;

  auto issue_kv = [&](int it) {
    const int e = plan[1 + it];
    const bool pooled = (e >> 20) & 1;
    const int j = e & 0xFFFFF;
    const int st = it & 1;
    mbar_arrive_expect_tx(&bar_kv[st], 2 * L::kKV);
    const CUtensorMap *mk = pooled ? &tm_pk : &tm_k;
    const CUtensorMap *mv = pooled ? &tm_pv : &tm_v;
#pragma unroll
    for (int x = 0; x < L::kBoxes; ++x) {
      tma_load_4d(sK[st] + x * BN * 128, mk, 64 * x, hk, j * BN, b, &bar_kv[st]);
      tma_load_4d(sV[st] + x * BN * 128, mv, 64 * x, hk, j * BN, b, &bar_kv[st]);
    }
  };
  auto load_meta = [&](int it) {  // key metadata of tile `it` into buffer it & 1
    if (it >= n_tiles || tid >= BN) return;
    const int e = plan[1 + it];
    const int k = (e & 0xFFFFF) * BN + tid;
    if ((e >> 20) & 1) {
      s_seg[it & 1][tid] = k;  // pooled: column index
      s_sink[it & 1][tid] = 0;
    } else {
      s_seg[it & 1][tid] = k < p.T ? (p.seg ? p.seg[size_t(b) * p.T + k] : 1) : 0;
      s_sink[it & 1][tid] = (k < p.T && p.sink) ? p.sink[size_t(b) * p.T + k] : 0;
    }
  };

  if (tid == 0 && n_tiles > 0) {
    mbar_arrive_expect_tx(&bar_q, L::kQ);
#pragma unroll
    for (int x = 0; x < L::kBoxes; ++x) tma_load_4d(sQ + x * BM * 128, &tm_q, 64 * x, hq, q0, b, &bar_q);
    issue_kv(0);
  }
  load_meta(0);

  const int myseg = q < p.T ? (p.seg ? p.seg[size_t(b) * p.T + q] : 1) : 0;
  const int W = p.W == 0 ? INT_MAX : p.W;
  const float c = 1.4426950408889634f * rsqrtf(float(D));  // log2(e) / sqrt(d), applied to scores
  float o[D];
#pragma unroll
  for (int i = 0; i < D; ++i) o[i] = 0.f;
  float m = -INFINITY, l = 0.f;
  __syncthreads();

  constexpr uint32_t kIdS = idesc_bf16(BM, BN, 0);
  constexpr uint32_t kIdPV = idesc_bf16(BM, D, 1);

  for (int it = 0; it < n_tiles; ++it) {
    const int st = it & 1;
    const int e = plan[1 + it];
    const bool pooled = (e >> 20) & 1;
    const int j = e & 0xFFFFF;
    // ---- issue S = Q K^T
    if (tid == 0 && !fail) {
      if (it + 1 < n_tiles) issue_kv(it + 1);  // stage st^1 is free: tile it-1 finished
      bool ok = true;
      if (it == 0) ok = mbar_wait(&bar_q, 0, p.err);
      ok = ok && mbar_wait(&bar_kv[st], (it >> 1) & 1, p.err);
      if (!ok) {
        fail = true;
      } else {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;  // 16 columns = 32 bytes inside the atom
          const uint64_t a = sdesc_sw128(sQ + (kk >> 2) * BM * 128 + off, 16, 1024);
          const uint64_t bd = sdesc_sw128(sK[st] + (kk >> 2) * BN * 128 + off, 16, 1024);
          mma_bf16(tS, a, bd, kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar_s);
      }
    }
    // ---- softmax on row `tid`
    if (!mbar_wait(&bar_s, it & 1, p.err)) fail = true;
    __syncwarp();
    tc_fence_after();
    float s[BN];
    tmem_ld32(tS + lane_base, s);
    tmem_ld32(tS + lane_base + 32, s + 32);
    const int *ks = s_seg[st];
    const unsigned char *kn = s_sink[st];
    float mx = -INFINITY;
#pragma unroll
    for (int x = 0; x < BN; ++x) {
      bool vis;
      if (pooled) {
        const int jp = ks[x];
        vis = myseg > 0 && jp < p.nb && (jp + 1) * p.block <= q - p.W + 1;
      } else {
        const int k = j * BN + x;
        vis = myseg > 0 && k <= q && ks[x] == myseg && (q - k < W || kn[x]);
      }
      s[x] = vis ? s[x] : -INFINITY;
      mx = fmaxf(mx, s[x]);
    }
    const float m_new = fmaxf(m, mx);
    const float alpha = (m_new == -INFINITY) ? 1.f : ex2((m - m_new) * c);
    const float mc = (m_new == -INFINITY) ? 0.f : m_new * c;
    float rs = 0.f;
    // P row -> shared memory, K-major 128B-swizzled (16-byte chunk ch of row r
    // lands at chunk ch ^ (r & 7)), 8 probabilities per chunk
    const uint32_t sP = L::kAliasP ? sK[st] : sPsep;
#pragma unroll
    for (int ch = 0; ch < BN / 8; ++ch) {
      uint32_t w[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float p0 = ex2(fmaf(s[8 * ch + 2 * x], c, -mc));
        const float p1 = ex2(fmaf(s[8 * ch + 2 * x + 1], c, -mc));
        rs += p0 + p1;
        w[x] = pack_bf16x2(p0, p1);
      }
      st_shared_v4(sP + tid * 128 + ((ch ^ (tid & 7)) << 4), w[0], w[1], w[2], w[3]);
    }
    l = l * alpha + rs;
    m = m_new;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- issue O_tile = P V
    if (tid == 0 && !fail) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        const uint64_t a = sdesc_sw128(sP + kk * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(sV[st] + kk * 16 * 128, BN * 128, 1024);
        mma_bf16(tO, a, bd, kIdPV, kk > 0 ? 1u : 0u);
      }
      mma_commit(&bar_o);
    }
    load_meta(it + 1);
    if (!mbar_wait(&bar_o, it & 1, p.err)) fail = true;
    __syncwarp();
    tc_fence_after();
#pragma unroll
    for (int x = 0; x < D; x += 32) {
      float ot[32];
      tmem_ld32(tO + lane_base + x, ot);
#pragma unroll
      for (int i = 0; i < 32; ++i) o[x + i] = fmaf(o[x + i], alpha, ot[i]);
    }
    tc_fence_before();
    if (__syncthreads_or(fail)) {
      aborted = true;
      break;
    }
  }

  // ---- error path: give copies and MMAs that may still be in flight a
  //      bounded time (about 2 ms) to land before the CTA releases its shared
  //      memory and TMEM
  if (aborted)
    for (int i = 0; i < 2000; ++i) __nanosleep(1000);
  // ---- epilogue
  if (q < p.T && !aborted) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint16_t *dst = p.out + ((size_t(b) * p.T + q) * p.Hq + hq) * D;
#pragma unroll
    for (int x = 0; x < D; x += 8) {
      uint4 v;
      v.x = pack_bf16x2(o[x] * inv, o[x + 1] * inv);
      v.y = pack_bf16x2(o[x + 2] * inv, o[x + 3] * inv);
      v.z = pack_bf16x2(o[x + 4] * inv, o[x + 5] * inv);
      v.w = pack_bf16x2(o[x + 6] * inv, o[x + 7] * inv);
      *reinterpret_cast<uint4 *>(dst + x) = v;
    }
    if (p.lse)
      p.lse[(size_t(b) * p.Hq + hq) * p.T + q] =
          l > 0.f ? (m * c + __log2f(l)) * 0.6931471805599453f : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(L::kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// [B][rows][H][D] bf16 tensor as a 4-D map (D, H, rows, B); box (64, 1, box_rows, 1).
bool make_map(CUtensorMap *map, const void *ptr, int B, int rows, int H, int D, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {cuuint64_t(D), cuuint64_t(H), cuuint64_t(rows), cuuint64_t(B)};
  cuuint64_t strides[3] = {cuuint64_t(D) * 2, cuuint64_t(H) * D * 2, cuuint64_t(rows) * H * D * 2};
  cuuint32_t box[4] = {64, 1, cuuint32_t(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct PlanDims {
  int n_qt, n_kt, n_pt, stride;
  size_t sum_bytes, plan_bytes;
};

PlanDims plan_dims(int B, int T, int block) {
  PlanDims d;
  d.n_qt = (T + BM - 1) / BM;
  d.n_kt = (T + BN - 1) / BN;
  const int nb = block > 0 ? T / block : 0;
  d.n_pt = (nb + BN - 1) / BN;
  d.stride = 1 + d.n_kt + d.n_pt;
  d.sum_bytes = (size_t(B) * d.n_kt * sizeof(TileSummary) + 255) / 256 * 256;
  d.plan_bytes = size_t(B) * d.n_qt * d.stride * sizeof(int32_t);
  return d;
}

template <int D>
cudaError_t launch_tc(const PrefillArgs &a, void *ws, int *err, cudaStream_t stream) {
  PlanDims pd = plan_dims(a.batch, a.T, a.block);
  TileSummary *sum = static_cast<TileSummary *>(ws);
  int32_t *plan = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + pd.sum_bytes);
  TcParams p;
  p.B = a.batch;
  p.T = a.T;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.W = a.window;
  p.block = a.block;
  p.nb = a.block > 0 ? a.T / a.block : 0;
  p.n_qt = pd.n_qt;
  p.n_kt = pd.n_kt;
  p.n_pt = pd.n_pt;
  p.plan_stride = pd.stride;
  p.seg = a.seg_ids;
  p.sink = a.sink;
  p.plan = plan;
  p.out = static_cast<uint16_t *>(a.out);
  p.lse = a.lse;
  p.err = err;

  CUtensorMap tq, tk, tv, tpk, tpv;
  if (!make_map(&tq, a.q, a.batch, a.T, a.Hq, D, BM) || !make_map(&tk, a.k, a.batch, a.T, a.Hkv, D, BN) ||
      !make_map(&tv, a.v, a.batch, a.T, a.Hkv, D, BN))
    return cudaErrorInvalidValue;
  if (a.block > 0 && p.nb > 0) {
    if (!make_map(&tpk, a.pooled_k, a.batch, p.nb, a.Hkv, D, BN) ||
        !make_map(&tpv, a.pooled_v, a.batch, p.nb, a.Hkv, D, BN))
      return cudaErrorInvalidValue;
  } else {
    tpk = tk;
    tpv = tv;
  }
  const int ns = a.batch * pd.n_kt;
  tile_summary_kernel<<<(ns + 127) / 128, 128, 0, stream>>>(a.seg_ids, a.sink, a.T, pd.n_kt, sum, a.batch);
  const int nq = a.batch * pd.n_qt;
  tile_plan_kernel<<<(nq + 127) / 128, 128, 0, stream>>>(a.seg_ids, sum, p, plan);
  auto kern = prefill_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<D>::kBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(pd.n_qt, a.Hq, a.batch);
  kern<<<grid, kThreads, Smem<D>::kBytes, stream>>>(tq, tk, tv, tpk, tpv, p);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_plan_bytes(int batch, int T, int block) {
  PlanDims pd = plan_dims(batch, T, block);
  return pd.sum_bytes + pd.plan_bytes;
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, void *plan_ws, int *err, cudaStream_t stream) {
  if (size_t(a.batch) * a.T == 0) return cudaSuccess;
  if (a.d == 128) return launch_tc<128>(a, plan_ws, err, stream);
  if (a.d == 64) return launch_tc<64>(a, plan_ws, err, stream);
  return cudaErrorInvalidValue;
}

}  // namespace nd
