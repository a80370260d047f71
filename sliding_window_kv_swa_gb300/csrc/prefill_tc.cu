// prefill_tc.cu -- bf16 prefill attention on the 5th-generation tensor cores
// (tcgen05 MMAs with TMEM accumulators, TMA-staged tiles), for the mask of
// "How the 256-Token Sliding Window Works with Tools as KV Sinks in Needle",
// section "KV Sinks for Tools" (same segment, causal, window or sink), and for
// the compressed columns of "Compressed attention and the copy probe", section
// "Two kinds of columns" (pooled block j visible iff (j+1)*block <= q-W+1,
// then the exact sliding window).
//
// Work split.  A plan pass lists, for every (sequence, row span), the 64-key
// tiles that can hold a visible key (segment-id ranges, causal bound, window
// bound, sink presence; pooled tiles below the threshold), so the cost follows
// window + sink rather than T^2.
//
// One CTA runs two 128-row blocks that share their K/V tiles: two query heads
// of one GQA group (same rows), or, when the group size is odd, two
// consecutive row blocks of one head.  The kernel is persistent: one CTA per
// SM walks work items (sequence, row span, block pair) with a stride of the
// grid, and every role keeps running tile counts, so the next item's Q and
// first tiles load while the current one finishes.  Its sixteen warps
// specialise:
//   warps 0-3, 4-7 : one softmax warpgroup per row block; thread i owns row i
//                    (= TMEM lane i): exact mask, online softmax in the log2
//                    domain; bf16 P(g) goes back into TMEM over the front of
//                    S(g)'s buffer (already read out).
//   warp 8         : TMA loader: Q (two buffers), K tiles (freed as soon as
//                    both blocks' S MMAs have read them) and, for the packing
//                    mask, the tiles' segment / sink records (cp.async, freed
//                    once the softmax warps have built their masks); at
//                    d = 64 also V.
//   warps 9, 10    : one MMA issuer per row block: S(g) = Q K(g)^T (M128
//                    N64) into S buffer g % NS, then O += P(g-1) V(g-1)
//                    (M128, N=d, P read from TMEM, V an MN-major shared
//                    operand), so neither block waits behind the other's.
//                    The MMAs one thread issues run in issue order, so S(g)
//                    needs no wait for PV(g - NS), the last reader of the P
//                    its buffer held.
//   warp 11        : V loader at d = 128 (V tiles, freed after both blocks'
//                    PV); idle at d = 64.
//   warps 12-15    : epilogue: rotate the next item's Q in shared memory
//                    (when the call applies RoPE), read O out of TMEM and
//                    write O / l.
// TMEM per CTA: S 2 x NS x 64 (NS = 2 at d = 128, 3 at d = 64) and O 2 x d
// fp32 columns: 512 either way.
// O accumulates in TMEM; a row's O is rescaled (TMEM load / multiply / store)
// only when its running max grows by more than 2^8, so most tiles touch O
// only through the MMA.  Tiles every row of a warp fully sees skip the
// per-element mask; tiles no row of a warp sees skip the scores and the
// softmax and store a zero P.  Waits first probe the barrier without
// blocking (a completed phase costs tens of cycles that way, against
// hundreds for the blocking try_wait).  Every mbarrier wait is bounded; a wait that gives up
// raises the device error flag and a shared abort flag, and all roles then run
// to the common exit, which frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>

#include <vector>

#include "nd_common.cuh"
#include "nd_internal.h"

namespace nd {

namespace {

constexpr int BM = 128;  // rows per block = TMEM lanes
constexpr int BN = 64;   // keys per tile
// warps 0-7 softmax (block 0: 0-3, block 1: 4-7), 8 Q/K loader, 9-10 MMA
// issuers (block 0, block 1), 11 V loader, 12-15 epilogue
constexpr int kWarpLoad = 8, kWarpMma0 = 9, kWarpLoadV = 11, kWarpEpi0 = 12;
constexpr int kThreads = 16 * 32;
// Register split (setmaxnreg, per warpgroup): the softmax warpgroups hold a
// 64-score row per thread; the loader / issuer and epilogue warpgroups need
// few.  Launched at 128 a thread: 2 x 128 x 168 + 2 x 128 x 88 = 512 x 128.
constexpr int kRegsSoftmax = 168, kRegsOther = 88;
static_assert(2 * 128 * kRegsSoftmax + 2 * 128 * kRegsOther == kThreads * 128, "register split");
constexpr float kRescaleLog2 = 8.f;  // rescale O only when the max grows by more than 2^8

// Per (sequence, 64-key tile) metadata record, written once per call by
// tile_prep_kernel and copied asynchronously into shared memory by the loader
// next to the tile's K/V: segment ids, sink flags and summary flags.
struct alignas(128) TileMeta {
  int seg[BN];                     // 0 for keys past T
  unsigned long long sink_bits;    // bit x = key x is a sink
  unsigned long long id_mask[4];   // bit x = key x carries ids[i]
  int ids[4];                      // the distinct positive segment ids, in key order
  int n_ids;                       // how many (0..4); -1: more than four
  int seg_lo, seg_hi;              // over keys with a positive id (lo > hi: none)
  int all_sink, any_sink;
  int uniform_seg;                 // the one id every key < T carries (> 0), else 0
  int pad[12];
};
static_assert(sizeof(TileMeta) == 384, "16-byte chunks for cp.async");

struct TcParams {
  int B, T, Hq, Hkv, G, W, block, nb, n_span, span, n_kt, plan_stride, pair_heads, n_pairs;
  // queries are key rows q_off .. T-1 (Tq = T - q_off of them); q, out and lse
  // hold only those rows
  int q_off, Tq;
  // compressed variant: keys 0 .. n_pinned-1 are pinned (visible at any
  // distance) and the pooled blocks tile the positions after them
  int n_pinned;
  const int32_t *seg;
  const uint8_t *sink;
  const int32_t *plan;
  const TileMeta *meta;  // [B][n_kt]
  uint16_t *out;
  float *lse;
  int *err;
  const float2 *rope_cs;  // (cos, sin) [T][D/2]: rotate Q while staging it; NULL: Q as given
};

// ------------------------------------------------------------------ plan

// One warp builds the record of key tile j of sequence b; lane l handles keys
// l and l + 32.  Returns (to every lane) the tile's positive segment-id range
// and whether it holds a sink, for the plan.
__device__ void build_tile_meta(const int32_t *seg, const uint8_t *sink, int T, int b, int j, int lane,
                                TileMeta &m, int &seg_lo, int &seg_hi, int &any_sink) {
  int lo = INT_MAX, hi = INT_MIN, all = 1, any = 0, padding = 0;
  uint32_t sink_word[2];
  int sv[2];
  for (int kk = lane, half = 0; kk < BN; kk += 32, ++half) {
    const int k = j * BN + kk;
    const int s = k < T ? (seg ? seg[size_t(b) * T + k] : 1) : 0;
    const int sk = (k < T && sink) ? (sink[size_t(b) * T + k] != 0) : 0;
    m.seg[kk] = s;
    sv[half] = s;
    if (s > 0) {
      lo = min(lo, s);
      hi = max(hi, s);
    }
    padding |= (k < T) & (s <= 0);
    all &= sk;
    any |= sk;
    sink_word[half] = __ballot_sync(0xffffffffu, sk != 0);
  }
  // the distinct positive ids and, for each, the keys carrying it: at most
  // four, taken in key order (a tile with more keeps n_ids = -1)
  bool done0 = sv[0] <= 0, done1 = sv[1] <= 0;
  int n_ids = 0;
  for (int i = 0; i <= 4; ++i) {
    const unsigned b0 = __ballot_sync(0xffffffffu, !done0), b1 = __ballot_sync(0xffffffffu, !done1);
    if (!b0 && !b1) break;
    if (i == 4) {
      n_ids = -1;
      break;
    }
    const int cand = b0 ? __shfl_sync(0xffffffffu, sv[0], __ffs(b0) - 1)
                        : __shfl_sync(0xffffffffu, sv[1], __ffs(b1) - 1);
    const unsigned m0 = __ballot_sync(0xffffffffu, sv[0] == cand), m1 = __ballot_sync(0xffffffffu, sv[1] == cand);
    if (lane == 0) {
      m.ids[i] = cand;
      m.id_mask[i] = (unsigned long long)m0 | ((unsigned long long)m1 << 32);
    }
    done0 |= sv[0] == cand;
    done1 |= sv[1] == cand;
    n_ids = i + 1;
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, off));
    all &= __shfl_xor_sync(0xffffffffu, all, off);
    any |= __shfl_xor_sync(0xffffffffu, any, off);
    padding |= __shfl_xor_sync(0xffffffffu, padding, off);
  }
  if (lane == 0) {
    m.seg_lo = lo;
    m.seg_hi = hi;
    m.all_sink = all;
    m.any_sink = any;
    m.sink_bits = (unsigned long long)sink_word[0] | ((unsigned long long)sink_word[1] << 32);
    m.uniform_seg = (lo == hi && !padding) ? lo : 0;
    m.n_ids = n_ids;
  }
  seg_lo = lo;
  seg_hi = hi;
  any_sink = any;
}

// One block per sequence: first the records of all its key tiles (kept in
// global memory for the attention kernel and, as segment-id range and sink
// flag, in shared memory), then one warp per row span lists the key tiles any
// row of the span may see -- pooled tiles first (entry bit 20 set), then
// exact tiles, ascending.  Dynamic shared memory: 3 ints per key tile.
__global__ void __launch_bounds__(1024) tile_prep_kernel(TcParams p, TileMeta *meta, int32_t *plan) {
  extern __shared__ int s_tile[];  // [3][n_kt]: seg_lo, seg_hi, any_sink
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  int *t_lo = s_tile, *t_hi = s_tile + p.n_kt, *t_any = s_tile + 2 * p.n_kt;
  pdl_trigger();  // the next kernel reads nothing written here before it waits
  for (int j = warp; j < p.n_kt; j += nw) {
    int lo, hi, any;
    build_tile_meta(p.seg, p.sink, p.T, b, j, lane, meta[size_t(b) * p.n_kt + j], lo, hi, any);
    if (lane == 0) {
      t_lo[j] = lo;
      t_hi[j] = hi;
      t_any[j] = any;
    }
  }
  __syncthreads();
  for (int sp = warp; sp < p.n_span; sp += nw) {
    const int q0 = p.q_off + sp * p.span, q1 = min(p.T, q0 + p.span) - 1;
    int32_t *out = plan + (size_t(b) * p.n_span + sp) * p.plan_stride;
    int n = 0;
    if (p.block > 0) {
      // pooled column j visible iff (j+1)*block <= q - W + 1 - n_pinned
      const int lim = q1 - p.W + 1 - p.n_pinned;
      const int ncol = lim >= p.block ? min(lim / p.block, p.nb) : 0;
      n = (ncol + BN - 1) / BN;
      for (int j = lane; j < n; j += 32) out[1 + j] = (1 << 20) | j;
    }
    int qlo = INT_MAX, qhi = INT_MIN;
    for (int q = q0 + lane; q <= q1; q += 32) {
      const int s = p.seg ? p.seg[size_t(b) * p.T + q] : 1;
      if (s > 0) {
        qlo = min(qlo, s);
        qhi = max(qhi, s);
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      qlo = min(qlo, __shfl_xor_sync(0xffffffffu, qlo, off));
      qhi = max(qhi, __shfl_xor_sync(0xffffffffu, qhi, off));
    }
    if (qlo <= qhi) {
      const int jmax = q1 / BN;
      for (int j0 = 0; j0 <= jmax; j0 += 32) {
        const int j = j0 + lane;
        bool keep = false;
        if (j <= jmax) {
          const bool in_window = p.W == 0 || (j + 1) * BN - 1 >= q0 - p.W + 1;
          const bool pinned = j * BN < p.n_pinned;  // holds a pinned key (compressed variant)
          keep = t_lo[j] <= t_hi[j] && t_lo[j] <= qhi && t_hi[j] >= qlo && (in_window || t_any[j] || pinned);
        }
        const unsigned m = __ballot_sync(0xffffffffu, keep);
        if (keep) out[1 + n + __popc(m & ((1u << lane) - 1u))] = j;
        n += __popc(m);
      }
    }
    if (lane == 0) out[0] = n;
  }
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

// One lane of a converged warp, chosen by elect.sync (1 there, 0 elsewhere).
// The MMA, commit and TMA helpers below take it as a predicate: the whole warp
// executes them converged and only the elected lane issues.  Issuing tcgen05
// instructions this way is several times cheaper than from a lane-divergent
// branch.
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred e;\n .reg .b32 x;\n elect.sync x|e, 0xffffffff;\n selp.u32 %0, 1, 0, e;\n}\n"
      : "=r"(r));
  return r;
}

// tcgen05 MMA, kind::f16 (bf16 operands, fp32 accumulation), A and B from
// shared memory.
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate, uint32_t leader) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 e, %5, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(leader));
}

// Same with the A operand (M x K, K-major) read from TMEM.
__device__ __forceinline__ void mma_bf16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate, uint32_t leader) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 e, %5, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(idesc), "r"(accumulate), "r"(leader));
}

__device__ __forceinline__ void mma_commit(uint64_t *bar, uint32_t leader) {
  asm volatile(
      "{\n .reg .pred e;\n setp.ne.b32 e, %1, 0;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(
          smem_u32(bar)),
      "r"(leader)
      : "memory");
}

// Packed fp32 pairs (sm_100 family): (o0, o1) = (a0, a1) * b + c with b, c packed.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void fma_f32x2(float &o0, float &o1, float a0, float a1, uint64_t b, uint64_t c) {
  asm("{\n .reg .b64 a, r;\n mov.b64 a, {%2, %3};\n fma.rn.f32x2 r, a, %4, %5;\n mov.b64 {%0, %1}, r;\n}\n"
      : "=f"(o0), "=f"(o1)
      : "f"(a0), "f"(a1), "l"(b), "l"(c));
}
// (s0, s1) += (a0, a1)
__device__ __forceinline__ void add_f32x2(float &s0, float &s1, float a0, float a1) {
  asm("{\n .reg .b64 s, a;\n mov.b64 s, {%0, %1};\n mov.b64 a, {%2, %3};\n add.rn.f32x2 s, s, a;\n"
      " mov.b64 {%0, %1}, s;\n}\n"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint64_t *bar, uint32_t leader) {
  asm volatile(
      "{\n .reg .pred e;\n setp.ne.b32 e, %7, 0;\n"
      " @e cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5}], [%6];\n}\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)),
      "r"(leader)
      : "memory");
}

__device__ __forceinline__ void expect_tx(uint64_t *bar, uint32_t bytes, uint32_t leader) {
  asm volatile(
      "{\n .reg .pred e;\n setp.ne.b32 e, %2, 0;\n"
      " @e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n}\n" ::"r"(smem_u32(bar)),
      "r"(bytes), "r"(leader)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Bounded wait that also gives up at once when another role already did.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, int *err,
                                              volatile int *abort_flag) {
  // A phase that has already completed is seen by the non-blocking probe in
  // tens of cycles; try_wait costs hundreds even then, so it is only the
  // fallback for a phase still in progress.
  if (mbar_test_wait(bar, parity)) return true;
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_flag) return false;
  }
  raise_device_error(err, ND_DEVERR_TIMEOUT);
  *abort_flag = 1;
  return false;
}

// The same for a whole warp: every lane polls (the warp never diverges, so
// it is woken as one), and leaves converged with the common outcome.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int *err, volatile int *abort_flag) {
  const bool ok = wait_or_abort(bar, parity, err, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// Failure-path test mode (nd.h: nd_set_prefill_epilogue_wait_limit): with
// a limit set, the epilogue's wait for a block's last PV -- a wait that
// guards no copy in flight -- is replaced by `limit` non-blocking polls of a
// barrier nothing arrives on, so it runs out on every CTA and the kernel
// takes its abort path.  0 (the default): the ordinary bounded wait.
__device__ unsigned g_epi_wait_limit = 0;

__device__ __forceinline__ bool warp_wait_never(uint64_t *never, int *err, volatile int *abort_flag,
                                                uint32_t limit) {
  bool ok = false;
  for (uint32_t i = 0; i < limit && !ok; ++i) ok = mbar_test_wait(never, 0);
  if (!ok && !*abort_flag) {
    raise_device_error(err, ND_DEVERR_TIMEOUT);
    *abort_flag = 1;
  }
  return __all_sync(0xffffffffu, ok);
}

// The same for the loader's waits at d = 64: try_wait with a suspend-time
// hint, so the waiting loader sleeps instead of re-polling and leaves issue
// slots to the softmax warps on its SM sub-partition (measured: 2% off the
// compressed kernel, 1% onto the packed d = 128 one, which keeps warp_wait).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(2000)
      : "memory");
  return ok != 0;
}
// Bounded like wait_or_abort: at most kWaitLimit / 64 polls of at most 2 us.
__device__ __forceinline__ bool warp_wait_sleep(uint64_t *bar, uint32_t parity, int *err,
                                                volatile int *abort_flag) {
  bool ok = mbar_test_wait(bar, parity);
  for (uint32_t i = 0; i < kWaitLimit / 64 && !ok; ++i) {
    if (mbar_try_wait_sleep(bar, parity)) {
      ok = true;
      break;
    }
    if (*abort_flag) break;
  }
  if (!ok && !*abort_flag) {
    raise_device_error(err, ND_DEVERR_TIMEOUT);
    *abort_flag = 1;
  }
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ kernel

template <int D>
struct Lay {
  static constexpr int NK = D == 64 ? 6 : 3;       // K stages
  static constexpr int NV = D == 64 ? 5 : 2;       // V stages
  static constexpr int NM = D == 64 ? 8 : 4;       // tile-record stages (>= NK: a record rides with its K tile)
  static constexpr int kBoxes = D / 64;            // 64-column swizzle atoms per row
  static constexpr int kQ = kBoxes * BM * 128;     // one block's Q tile
  static constexpr int kKV = kBoxes * BN * 128;    // one K (or V) tile
  static constexpr int oQ = 0;                     // Q[2 buffers][2 blocks]
  static constexpr int oK = 4 * kQ;                // K[NK stages]
  static constexpr int oV = oK + NK * kKV;         // V[NV stages]
  static constexpr int oM = oV + NV * kKV;         // TileMeta[NM stages]
  static constexpr int kBytes = oM + NM * int(sizeof(TileMeta)) + 1024;  // + alignment slack
  static_assert(NM >= NK, "tile records ride with K tiles");
  // S buffers per block: P(g) is written over the front of S(g)'s buffer,
  // which S(g + NS) reuses once PV(g) (issued before it) has read P(g); at
  // d = 64 three fit beside O
  static constexpr int NS = D == 64 ? 3 : 2;
  // TMEM columns: S[block][NS buffers] (BN fp32 each; P(g), BN/2 columns of
  // bf16 pairs, overwrites the front of S(g)'s buffer), O[block] (D fp32 each)
  static constexpr int cS = 0, cO = 2 * NS * BN;
  static constexpr int kCols = cO + 2 * D;
  static_assert(kCols <= 512, "TMEM budget");
  static constexpr int kTmemCols = kCols <= 256 ? 256 : 512;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once this thread's earlier cp.async copies have landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c,
                                             uint32_t &d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void st_global_v4(void *ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// kPooled: the compressed variant (pooled column tiles, no segment ids or
// sinks); otherwise exact tiles under the packing mask only.  The two are
// separate instantiations so each carries only its own masking code.
template <int D, bool kPooled>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_pk,
                      const __grid_constant__ CUtensorMap tm_pv, const TcParams p) {
  using L = Lay<D>;
  constexpr int NK = L::NK, NV = L::NV, NM = L::NM, NS = L::NS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t q_full[2], q_empty[2], k_full[NK], k_empty[NK], v_full[NV], v_empty[NV],
      m_full[NM], m_empty[NM], s_full[2][NS], p_full[2][NS], pv_done[2][NS], o_free[2], epi_full[2],
      epi_empty[2], q_rot[2];
  __shared__ float s_inv[2][BM];  // 1 / row sum, from the softmax warps to the epilogue warps
  __shared__ __align__(128) uint8_t s_stage[4][32 * 64];  // epilogue staging, one block per warp
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ __align__(8) uint64_t s_never;  // failure-path test mode only: nothing arrives on it

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int *abort_flag = &s_abort;
  // Work items (sequence, 128-row span, head pair), pairs fastest so CTAs
  // running side by side share K/V tiles in L2; CTA c takes items c,
  // c + gridDim.x, ...  Every role walks the same items and keeps running
  // tile counts, so the barrier phases carry over from item to item.
  const int n_items = p.B * p.n_span * p.n_pairs;
  struct Item {
    int b, head0, head1, row00, row01, hk, n;
    const int32_t *tiles;  // the plan's tile entries (global memory)
  };
  auto item_at = [&](int w) {
    Item it;
    const int pr = w % p.n_pairs, rest = w / p.n_pairs, sp = rest % p.n_span;
    it.b = rest / p.n_span;
    it.head0 = p.pair_heads ? 2 * pr : pr;
    it.head1 = p.pair_heads ? it.head0 + 1 : it.head0;
    it.row00 = p.q_off + (p.pair_heads ? sp * BM : sp * 2 * BM);
    it.row01 = p.pair_heads ? it.row00 : it.row00 + BM;
    it.hk = it.head0 / p.G;
    const int32_t *plan = p.plan + (size_t(it.b) * p.n_span + sp) * p.plan_stride;
    it.n = plan[0];
    it.tiles = plan + 1;
    return it;
  };

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  auto sQ = [&](int qb, int rb) { return base + L::oQ + (2 * qb + rb) * L::kQ; };
  auto sK = [&](int st) { return base + L::oK + st * L::kKV; };
  auto sV = [&](int st) { return base + L::oV + st * L::kKV; };
  auto sM = [&](int st) { return base + L::oM + st * uint32_t(sizeof(TileMeta)); };
  auto meta_at = [&](int st) {  // generic pointer to a stage's tile record
    return reinterpret_cast<const TileMeta *>(smem_raw + (sM(st) - smem_u32(smem_raw)));
  };

  if (tid == 0) {
    for (int u = 0; u < 2; ++u) {
      mbar_init(&q_full[u], 1);
      mbar_init(&q_empty[u], 2);  // committed by both issuers after an item's last S MMA
      mbar_init(&q_rot[u], BM);   // the epilogue threads have rotated the buffer's rows
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 2);  // one commit from each block's issuer
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 2);
    }
    for (int s = 0; s < NM; ++s) {
      mbar_init(&m_full[s], 32);   // one cp.async arrival per loader lane
      mbar_init(&m_empty[s], 8);   // one arrival per softmax warp
    }
    for (int r = 0; r < 2; ++r) {
      // one barrier triple per S/P buffer: a buffer's next use (two tiles
      // on) cannot start before the current one has been consumed, so no
      // wait ever sees a phase run two ahead
      for (int u = 0; u < NS; ++u) {
        mbar_init(&s_full[r][u], 1);
        mbar_init(&p_full[r][u], BM);
        mbar_init(&pv_done[r][u], 1);
      }
      mbar_init(&o_free[r], BM);     // the epilogue warps have read the block's O out of TMEM
      mbar_init(&epi_full[r], BM);   // the softmax threads have posted 1 / l for the item
      mbar_init(&epi_empty[r], BM);  // the epilogue threads have taken it
    }
    s_abort = 0;
    mbar_init(&s_never, 1);
    fence_barrier_init();
  }
  if (warp == kWarpMma0) {
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
  // dependent launch: the setup above overlapped the kernel before this one;
  // every global read below (plan, tile records, Q, K, V, table) follows it
  pdl_wait();
  auto tS = [&](int rb, int buf) { return tmem + L::cS + (NS * rb + buf) * BN; };
  auto tO = [&](int rb) { return tmem + L::cO + rb * D; };
  bool fail = false;

  if (warp >= 8) {
  // loader / issuer / epilogue warpgroups: registers to the softmax warpgroups
  regs_dec<kRegsOther>();
  // at d = 64 (shallower tiles, deeper rings) one warp loads both and measured
  // slightly faster; warp 11 then idles
  constexpr bool kSplitLoad = D == 128;
  if (warp == kWarpLoad || (kSplitLoad && warp == kWarpLoadV)) {
    // ------------------------------------------------ TMA loaders
    //   Warp 8: Q (two buffers, so item i+1's Q lands while item i runs), K
    //   tiles (NK stages, freed once both blocks' S MMAs read them) and tile
    //   records (NM stages, freed once all eight softmax warps built their
    //   masks).  Warp 11: V tiles (NV stages, freed after both blocks' PV).
    //   Two warps, so the K ring never waits behind the V ring (at an item
    //   boundary the next item's first K tiles go out as soon as K slots
    //   free).  Each warp stays converged; the elected lane issues.
    const bool vwarp = warp == kWarpLoadV;
    const uint32_t leader = elect_one();
    auto lwait = [&](uint64_t *bar, uint32_t parity) {
      return D == 64 ? warp_wait_sleep(bar, parity, p.err, abort_flag) : warp_wait(bar, parity, p.err, abort_flag);
    };
    int gt = 0;  // tiles loaded before the current item
    auto load_q = [&](int w, int it) {
      const Item I = item_at(w);
      const int qb = it & 1;
      // the buffer's previous user, item it-2, has run all its S MMAs
      if (it >= 2 && !lwait(&q_empty[qb], ((it >> 1) - 1) & 1)) return false;
      expect_tx(&q_full[qb], 2 * L::kQ, leader);
      for (int x = 0; x < L::kBoxes; ++x) {
        tma_load_4d(sQ(qb, 0) + x * BM * 128, &tm_q, 64 * x, I.head0, I.row00 - p.q_off, I.b, &q_full[qb], leader);
        tma_load_4d(sQ(qb, 1) + x * BM * 128, &tm_q, 64 * x, I.head1, I.row01 - p.q_off, I.b, &q_full[qb], leader);
      }
      return true;
    };
    if (!vwarp && blockIdx.x < n_items) fail = !load_q(blockIdx.x, 0);
    for (int w = blockIdx.x, it = 0; w < n_items && !fail; w += gridDim.x, ++it) {
      const Item I = item_at(w);
      // Ring positions and phases follow the running tile count g.
      auto load_k = [&](int j) {
        const int e = I.tiles[j];
        const bool pooled = kPooled && ((e >> 20) & 1);
        const int jt = e & 0xFFFFF;
        const int g = gt + j, st = g % NK, sm = g % NM;
        if (!((g < NK || lwait(&k_empty[st], ((g / NK) - 1) & 1)) &&
              (kPooled || g < NM || lwait(&m_empty[sm], ((g / NM) - 1) & 1))))
          return false;
        expect_tx(&k_full[st], L::kKV, leader);
        for (int x = 0; x < L::kBoxes; ++x)
          tma_load_4d(sK(st) + x * BN * 128, pooled ? &tm_pk : &tm_k, 64 * x, I.hk, jt * BN, I.b, &k_full[st], leader);
        // the tile's record (384 bytes) rides along asynchronously; the
        // compressed variant's masks need none
        if constexpr (!kPooled) {
          constexpr int kChunks = int(sizeof(TileMeta)) / 16;
          if (lane < kChunks)
            cp_async16(sM(sm) + lane * 16, reinterpret_cast<const char *>(p.meta + size_t(I.b) * p.n_kt + jt) + lane * 16);
          cp_async_arrive(&m_full[sm]);
        }
        __syncwarp();
        return true;
      };
      auto load_v = [&](int j) {
        const int e = I.tiles[j];
        const bool pooled = kPooled && ((e >> 20) & 1);
        const int jt = e & 0xFFFFF;
        const int g = gt + j, st = g % NV;
        if (!(g < NV || lwait(&v_empty[st], ((g / NV) - 1) & 1))) return false;
        expect_tx(&v_full[st], L::kKV, leader);
        for (int x = 0; x < L::kBoxes; ++x)
          tma_load_4d(sV(st) + x * BN * 128, pooled ? &tm_pv : &tm_v, 64 * x, I.hk, jt * BN, I.b, &v_full[st], leader);
        return true;
      };
      // the next item's Q goes out once K(NK-1) of this one has (its ring
      // slot freed means the previous item's S MMAs, the last readers of
      // that Q buffer, are done or nearly so)
      const int jq = I.n < NK - 1 ? I.n : NK - 1;
      const bool more = w + int(gridDim.x) < n_items;
      if (vwarp) {
        for (int j = 0; j < I.n && !fail; ++j)
          if (!load_v(j)) fail = true;
      } else {
        // (one warp: K runs one tile ahead of V: K(0), K(1), V(0), K(2), ...)
        for (int j = 0; j <= I.n && !fail; ++j) {
          if (j < I.n && !load_k(j)) fail = true;
          if (!kSplitLoad && !fail && j >= 1 && !load_v(j - 1)) fail = true;
          if (!fail && j == jq && more && !load_q(w + gridDim.x, it + 1)) fail = true;
        }
      }
      gt += I.n;
    }
  } else if (warp == kWarpMma0 || warp == kWarpMma0 + 1) {
    // ------------------------------------------------ MMA issuers, one per block
    //   Per tile g of the block (g: running tile count over its items):
    //   S(g) = Q K(g)^T into S buffer g % NS once K(g) has landed; then
    //   O += P(g-1) V(g-1) once P(g-1) is in TMEM and V(g-1) has landed.
    const int rb = warp - kWarpMma0;
    const uint32_t leader = elect_one();
    constexpr uint32_t kIdS = idesc_bf16(BM, BN, 0);
    constexpr uint32_t kIdPV = idesc_bf16(BM, D, 1);
    bool ok = true;
    int gt = 0, used = 0;  // used: items so far whose O went through TMEM
    // PV(g) is issued after S(g + 1), also across items (the next item's
    // first S goes out before this item's last PV).  PV(g - NS), the last
    // reader of the buffer S(g) overwrites, was issued NS - 1 iterations
    // earlier by this thread.
    constexpr int kLag = 1;
    int pv_g[2] = {-1, -1}, pv_first[2] = {0, 0}, pv_ofree[2] = {-1, -1};  // pending PVs, oldest first
    int npend = 0;
    auto issue_pv = [&]() {
      const int g = pv_g[0], first = pv_first[0], ofree = pv_ofree[0], sv = g % NV, u = g % NS;
      pv_g[0] = pv_g[1];
      pv_first[0] = pv_first[1];
      pv_ofree[0] = pv_ofree[1];
      --npend;
      // an item's first PV overwrites O: the epilogue warps must have read
      // out the O of the previous item that used it
      // the three conditions are probed together first (non-blocking, their
      // latencies overlap); only one still in progress takes the blocking path
      const bool ready = D == 64 && __all_sync(0xffffffffu, (ofree < 0 || mbar_test_wait(&o_free[rb], ofree)) &
                                                                mbar_test_wait(&p_full[rb][u], (g / NS) & 1) &
                                                                mbar_test_wait(&v_full[sv], (g / NV) & 1));
      ok = ready || ((ofree < 0 || warp_wait(&o_free[rb], ofree, p.err, abort_flag)) &&
                     warp_wait(&p_full[rb][u], (g / NS) & 1, p.err, abort_flag) &&
                     warp_wait(&v_full[sv], (g / NV) & 1, p.err, abort_flag));
      if (!ok) return;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {  // 16 keys = 8 TMEM columns of bf16 pairs
        const uint64_t bd = sdesc_sw128(sV(sv) + kk * 16 * 128, BN * 128, 1024);
        mma_bf16_ts(tO(rb), tS(rb, u) + kk * 8, bd, kIdPV, (!first || kk > 0) ? 1u : 0u, leader);
      }
      mma_commit(&pv_done[rb][u], leader);
      mma_commit(&v_empty[sv], leader);
    };
    Item In = item_at(blockIdx.x);  // the next item's plan row, read one item ahead
    for (int w = blockIdx.x, it = 0; w < n_items && ok; w += gridDim.x, ++it) {
      const Item I = In;
      if (w + int(gridDim.x) < n_items) In = item_at(w + gridDim.x);
      const int qb = it & 1;
      ok = warp_wait(p.rope_cs ? &q_rot[qb] : &q_full[qb], (it >> 1) & 1, p.err, abort_flag);
      for (int j = 0; j < I.n && ok; ++j) {
        const int g = gt + j, st = g % NK;
        // The buffer holds P(g - NS) until PV(g - NS) has read it.  This
        // thread issued that PV before this S, and the MMAs a thread issues
        // run in issue order, so S(g) cannot overwrite P(g - NS) early.
        ok = warp_wait(&k_full[st], (g / NK) & 1, p.err, abort_flag);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;  // 16 columns = 32 bytes inside the atom
          const uint64_t a = sdesc_sw128(sQ(qb, rb) + (kk >> 2) * BM * 128 + off, 16, 1024);
          const uint64_t bd = sdesc_sw128(sK(st) + (kk >> 2) * BN * 128 + off, 16, 1024);
          mma_bf16(tS(rb, g % NS), a, bd, kIdS, kk > 0 ? 1u : 0u, leader);
        }
        mma_commit(&s_full[rb][g % NS], leader);
        mma_commit(&k_empty[st], leader);
        if (j + 1 == I.n) mma_commit(&q_empty[qb], leader);  // Q may be replaced once these have run
        if (npend == kLag) issue_pv();
        const int of = (j == 0 && used > 0) ? ((used - 1) & 1) : -1;
        if (npend == 0) {  // (fixed slots keep the queue in registers)
          pv_g[0] = g;
          pv_first[0] = j == 0;
          pv_ofree[0] = of;
        } else {
          pv_g[1] = g;
          pv_first[1] = j == 0;
          pv_ofree[1] = of;
        }
        ++npend;
      }
      if (I.n == 0) mma_commit(&q_empty[qb], leader);
      if (I.n > 0) ++used;
      gt += I.n;
    }
    while (ok && npend > 0) issue_pv();
    fail = !ok;
  } else if (warp >= kWarpEpi0) {
    // ------------------------------------------------ epilogue warps
    //   Warp 12 + x reads TMEM lanes 32x..32x+31 of each block's O once the
    //   item's last PV has landed, frees O for the next item, and writes
    //   O / l as bf16 rows straight to global memory (one row per thread,
    //   sixteen-byte stores).
    const int qd = warp & 3;
    const int r = qd * 32 + lane;
    const uint32_t lane_base = uint32_t(qd * 32) << 16;
    const uint32_t o_test_limit = g_epi_wait_limit;
    const uint32_t stage = smem_u32(&s_stage[qd][0]);
    bool ok = true;
    int gt = 0;
    // Rotary embedding of an item's Q, in place in shared memory, once its
    // TMA load has landed: rotate-half pairs (i, i + D/2) at the row's own
    // position t, from the (cos, sin) table.  In the 128-byte swizzle a row's
    // 16-byte chunk c sits at chunk c ^ (row & 7); at D = 128 the partner of
    // column i is column i of the second 64-column box (the same offset), at
    // D = 64 it is chunk c + 4 of the same row.  Lane -> (row, chunk) so a
    // warp reads whole table rows.  Rows at or past T (zero-filled) stay zero.
    auto rotate_q = [&](int w, int it) {
      const Item I = item_at(w);
      const int qb = it & 1;
      if (!warp_wait(&q_full[qb], (it >> 1) & 1, p.err, abort_flag)) return false;
      constexpr int kPairChunks = D / 16, kRowsPerPass = 32 / kPairChunks;
      const int c = lane % kPairChunks;
#pragma unroll 1
      for (int pass = 0; pass < 32 / kRowsPerPass; ++pass) {
        const int rr = qd * 32 + pass * kRowsPerPass + lane / kPairChunks;
#pragma unroll
        for (int rb = 0; rb < 2; ++rb) {
          const int t = (rb ? I.row01 : I.row00) + rr;
          if (t >= p.T) continue;
          const float4 *cs4 = reinterpret_cast<const float4 *>(p.rope_cs + size_t(t) * (D / 2) + 8 * c);
          float cc[8], ss[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 v = __ldg(cs4 + i);
            cc[2 * i] = v.x, ss[2 * i] = v.y, cc[2 * i + 1] = v.z, ss[2 * i + 1] = v.w;
          }
          const uint32_t row = sQ(qb, rb) + rr * 128;
          const uint32_t lo = row + ((c ^ (rr & 7)) << 4);
          const uint32_t hi = D == 128 ? lo + BM * 128 : row + (((c + 4) ^ (rr & 7)) << 4);
          uint32_t a[4], b[4], ya[4], yb[4];
          ld_shared_v4(lo, a[0], a[1], a[2], a[3]);
          ld_shared_v4(hi, b[0], b[1], b[2], b[3]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float x0, x1, y0, y1;
            rope_pair(bf16_lo(a[i]), bf16_lo(b[i]), cc[2 * i], ss[2 * i], x0, y0);
            rope_pair(bf16_hi(a[i]), bf16_hi(b[i]), cc[2 * i + 1], ss[2 * i + 1], x1, y1);
            ya[i] = pack_bf16x2(x0, x1);
            yb[i] = pack_bf16x2(y0, y1);
          }
          st_shared_v4(lo, ya[0], ya[1], ya[2], ya[3]);
          st_shared_v4(hi, yb[0], yb[1], yb[2], yb[3]);
        }
      }
      // the MMA reads Q through the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(&q_rot[qb]);
      return true;
    };
    // Q(it + 1) is rotated before item it's epilogue: it lands early in item
    // it, and the issuer wants it as soon as item it's last S has gone out.
    if (p.rope_cs && blockIdx.x < n_items) ok = rotate_q(blockIdx.x, 0);
    for (int w = blockIdx.x, it = 0; w < n_items && ok; w += gridDim.x, ++it) {
      const Item I = item_at(w);
      const int n = I.n;
      if (p.rope_cs && w + int(gridDim.x) < n_items && !rotate_q(w + gridDim.x, it + 1)) {
        ok = false;
        break;
      }
      for (int rb = 0; rb < 2 && ok; ++rb) {
        ok = warp_wait(&epi_full[rb], it & 1, p.err, abort_flag);
        if (!ok) break;
        const float inv = s_inv[rb][r];
        mbar_arrive(&epi_empty[rb]);
        const int head = rb ? I.head1 : I.head0;
        if (n > 0) {
          // PV(gl) landing implies every earlier MMA of the block has
          const int gl = gt + n - 1;
          ok = o_test_limit ? warp_wait_never(&s_never, p.err, abort_flag, o_test_limit)
                            : warp_wait(&pv_done[rb][gl % NS], (gl / NS) & 1, p.err, abort_flag);
          if (!ok) break;
          tc_fence_after();
        }
        // 32 columns at a time: TMEM -> registers (scaled, bf16) -> this
        // warp's 2 KB staging block (row = lane, 64 bytes, 16-byte chunks
        // swizzled) -> 8 rows x 64 contiguous bytes per warp store
        const int row0 = (rb ? I.row01 : I.row00) + qd * 32;
#pragma unroll 1
        for (int x = 0; x < D; x += 32) {
          uint32_t ov[32];
          if (n > 0) {
            tmem_ld32(tO(rb) + lane_base + x, ov);
            tmem_ld_wait();
            if (x + 32 == D) {
              tc_fence_before();
              mbar_arrive(&o_free[rb]);  // the next item's PV may overwrite O
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = 0u;  // no visible key
          }
#pragma unroll
          for (int y = 0; y < 4; ++y)
            st_shared_v4(stage + lane * 64 + ((y ^ ((lane >> 1) & 3)) << 4),
                         pack_bf16x2(__uint_as_float(ov[8 * y]) * inv, __uint_as_float(ov[8 * y + 1]) * inv),
                         pack_bf16x2(__uint_as_float(ov[8 * y + 2]) * inv, __uint_as_float(ov[8 * y + 3]) * inv),
                         pack_bf16x2(__uint_as_float(ov[8 * y + 4]) * inv, __uint_as_float(ov[8 * y + 5]) * inv),
                         pack_bf16x2(__uint_as_float(ov[8 * y + 6]) * inv, __uint_as_float(ov[8 * y + 7]) * inv));
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int rr = 8 * k + (lane >> 2), ch = lane & 3;
            uint32_t a0, a1, a2, a3;
            ld_shared_v4(stage + rr * 64 + ((ch ^ ((rr >> 1) & 3)) << 4), a0, a1, a2, a3);
            const int qq = row0 + rr;
            if (qq < p.T)
              st_global_v4(p.out + ((size_t(I.b) * p.Tq + (qq - p.q_off)) * p.Hq + head) * D + x + 8 * ch, a0, a1,
                           a2, a3);
          }
          __syncwarp();  // the staging block is free again
        }
      }
      gt += n;
    }
    fail = !ok;
  }
  } else {
    // ------------------------------------------------ softmax warpgroups
    regs_inc<kRegsSoftmax>();
    const int rb = warp >> 2;
    const int r = tid & (BM - 1);
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const int W = p.W == 0 ? INT_MAX : p.W;
    const float c = 1.4426950408889634f * rsqrtf(float(D));  // log2(e) / sqrt(d)
    int gt = 0;
    // An item's plan count, first tile entry and this row's segment id are
    // fetched one item ahead: at an item boundary these global loads would
    // otherwise queue behind the epilogue warps' stores.  (A plan row always
    // has room for one entry, so tiles[0] is read even when n is 0.)
    auto row_seg = [&](const Item &J) {
      const int qq = (rb ? J.row01 : J.row00) + r;
      return qq < p.T ? (p.seg ? p.seg[size_t(J.b) * p.T + qq] : 1) : 0;
    };
    Item In = item_at(blockIdx.x);
    int seg_n = row_seg(In), e_n = In.tiles[0];
    for (int w = blockIdx.x, it = 0; w < n_items; w += gridDim.x, ++it) {
    const Item I = In;
    const int n = I.n, b = I.b;
    const int q = (rb ? I.row01 : I.row00) + r;
    const int head = rb ? I.head1 : I.head0;
    const int myseg = seg_n;
    float m_used = -INFINITY, l = 0.f;
    int e_next = e_n;  // the next tile's entry, read a tile ahead
    if (w + int(gridDim.x) < n_items) {
      In = item_at(w + gridDim.x);
      seg_n = row_seg(In);
      e_n = In.tiles[0];
    }
    for (int j = 0; j < n; ++j) {
      const int g = gt + j, sm = g % NM;
      const int e = e_next;
      if (j + 1 < n) e_next = I.tiles[j + 1];
      const bool pooled = kPooled && ((e >> 20) & 1);
      const int k0 = (e & 0xFFFFF) * BN;
      // The row's visibility over the tile comes first (it needs only the
      // tile record), so it overlaps the S MMA; a tile no row of the warp
      // sees skips the score load and the softmax and stores a zero P.
      // (the compressed variant reads no tile records: no handshake)
      if (!kPooled && !fail && !wait_or_abort(&m_full[sm], (g / NM) & 1, p.err, abort_flag)) fail = true;
      __syncwarp();
      constexpr uint32_t kNegInf = 0xff800000u;
      // This row's 64-bit visibility word over the tile (bit x = key k0 + x),
      // built from shifts: a prefix for pooled columns (j visible iff
      // (j+1)*block <= q-W+1), (causal bound) and (window or sink) and (the
      // row's segment) for exact keys.
      const unsigned long long all1 = ~0ull;
      auto prefix = [&](int last) {  // bits 0..last
        return last < 0 ? 0ull : (last >= 63 ? all1 : (all1 >> (63 - last)));
      };
      unsigned long long vis;
      if (pooled) {
        const int lim = q - p.W + 1 - p.n_pinned;
        const int ncol = lim >= p.block ? min(lim / p.block, p.nb) : 0;
        vis = myseg > 0 ? prefix(ncol - 1 - k0) : 0ull;
      } else {
        const int lo = W == INT_MAX ? 0 : q - W + 1 - k0;  // first key inside the window
        const unsigned long long window = lo <= 0 ? all1 : (lo > 63 ? 0ull : (all1 << lo));
        const unsigned long long causal = prefix(q - k0);
        if (kPooled) {
          // no segment ids in the compressed variant; keys below n_pinned
          // are pinned (visible at any distance)
          vis = myseg > 0 ? (causal & (window | prefix(p.n_pinned - 1 - k0))) : 0ull;
        } else {
          const TileMeta *f = meta_at(sm);
          const unsigned long long cw = causal & (window | f->sink_bits);
          const int nid = f->n_ids;
          vis = 0ull;
          if (nid >= 0) {
            // the keys of this row's segment: one of the tile's few ids
#pragma unroll
            for (int i = 0; i < 4; ++i) vis = (i < nid && f->ids[i] == myseg) ? f->id_mask[i] : vis;
          } else {
            // more than four ids in the tile: compare every key's id, four
            // at a time; the loop stays rolled so the loads do not pile up
            const uint32_t mseg = sM(sm);
#pragma unroll 1
            for (int x = 0; x < BN; x += 4) {
              int sg[4];
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(sg[0]), "=r"(sg[1]), "=r"(sg[2]), "=r"(sg[3])
                           : "r"(mseg + x * 4));
              unsigned long long bits = 0ull;
#pragma unroll
              for (int i = 0; i < 4; ++i) bits |= (unsigned long long)(sg[i] == myseg) << i;
              vis |= bits << x;
            }
          }
          vis = myseg > 0 ? (vis & cw) : 0ull;
        }
      }
      __syncwarp();
      if (!kPooled && lane == 0) mbar_arrive(&m_empty[sm]);  // this warp is done with the tile record
      const bool none = __all_sync(0xffffffffu, vis == 0ull);
      if (!fail && !wait_or_abort(&s_full[rb][g % NS], (g / NS) & 1, p.err, abort_flag)) fail = true;
      __syncwarp();
      tc_fence_after();
      if (none) {
        // P(g) = 0 for this warp's rows (the MMA reads all 128 lanes)
        uint32_t z[BN / 2];
#pragma unroll
        for (int i = 0; i < BN / 2; ++i) z[i] = 0u;
        if constexpr (D == 64) {
          tmem_st16(tS(rb, g % NS) + lane_base, z);
          tmem_st16(tS(rb, g % NS) + lane_base + 16, z + 16);
        } else {
          tmem_st32(tS(rb, g % NS) + lane_base, z);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[rb][g % NS]);
        continue;
      }
      // one 64-register row buffer: raw scores, then masked scores, then p
      uint32_t v[BN];
      tmem_ld32(tS(rb, g % NS) + lane_base, v);
      tmem_ld32(tS(rb, g % NS) + lane_base + 32, v + 32);
      tmem_ld_wait();
      // whole-warp all-visible tiles skip the per-key select
      if (!__all_sync(0xffffffffu, vis == all1)) {
        const uint32_t v0 = uint32_t(vis), v1 = uint32_t(vis >> 32);
#pragma unroll
        for (int x = 0; x < BN; ++x) {
          const uint32_t bit = x < 32 ? (v0 >> x) & 1u : (v1 >> (x - 32)) & 1u;
          v[x] = bit ? v[x] : kNegInf;
        }
      }
      // row max: three-input max over 8 independent chains (keys i, i+8, ...,
      // i+56 on chain i)
      static_assert(BN == 64, "max chains cover 64 keys");
      float mxp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        mxp[i] = max3(__uint_as_float(v[i]), __uint_as_float(v[8 + i]), __uint_as_float(v[16 + i]));
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        mxp[i] = max3(mxp[i], __uint_as_float(v[24 + i]), __uint_as_float(v[32 + i]));
        mxp[i] = max3(mxp[i], __uint_as_float(v[40 + i]), __uint_as_float(v[48 + i]));
        mxp[i] = fmaxf(mxp[i], __uint_as_float(v[56 + i]));
      }
      const float mx = max3(max3(mxp[0], mxp[1], mxp[2]), max3(mxp[3], mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7]));
      if (m_used == -INFINITY) m_used = mx;  // nothing accumulated yet: no rescale
      const bool need = mx > m_used && (mx - m_used) * c > kRescaleLog2;
      const float alpha = need ? ex2((m_used - mx) * c) : 1.f;
      if (need) {
        l *= alpha;
        m_used = mx;
      }
      const float mc = m_used == -INFINITY ? 0.f : m_used * c;
      // p = 2^(s c - m c), two scores per packed fp32 FMA / add; P(g) as bf16
      // pairs over the front of S(g)'s buffer (already read out), the A
      // operand of the block's PV.  At d = 64 (softmax-bound) P is stored in
      // two halves so the first store runs while the second half is
      // computed; at d = 128 one store measured faster.
      const uint64_t c2 = pack_f32x2(c, c), nmc2 = pack_f32x2(-mc, -mc);
      float rsp[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (D == 64) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
          for (int x = 32 * hh; x < 32 * hh + 32; x += 2) {
            float a, bb;
            fma_f32x2(a, bb, __uint_as_float(v[x]), __uint_as_float(v[x + 1]), c2, nmc2);
            a = ex2(a);
            bb = ex2(bb);
            add_f32x2(rsp[(x >> 1) & 1 ? 2 : 0], rsp[(x >> 1) & 1 ? 3 : 1], a, bb);
            v[x] = __float_as_uint(a);
            v[x + 1] = __float_as_uint(bb);
          }
          // keys 32hh..32hh+31 -> v[32hh .. 32hh+15] (reads never behind writes)
#pragma unroll
          for (int i = 0; i < 16; ++i)
            v[32 * hh + i] = pack_bf16x2(__uint_as_float(v[32 * hh + 2 * i]), __uint_as_float(v[32 * hh + 2 * i + 1]));
          tmem_st16(tS(rb, g % NS) + lane_base + 16 * hh, v + 32 * hh);
        }
      } else {
#pragma unroll
        for (int x = 0; x < BN; x += 2) {
          float a, bb;
          fma_f32x2(a, bb, __uint_as_float(v[x]), __uint_as_float(v[x + 1]), c2, nmc2);
          a = ex2(a);
          bb = ex2(bb);
          add_f32x2(rsp[(x >> 1) & 1 ? 2 : 0], rsp[(x >> 1) & 1 ? 3 : 1], a, bb);
          v[x] = __float_as_uint(a);
          v[x + 1] = __float_as_uint(bb);
        }
      }
      l += (rsp[0] + rsp[1]) + (rsp[2] + rsp[3]);
      // O is rescaled only when the max grew by more than 2^8 (rare), after
      // PV(g-1) has landed
      if (__any_sync(0xffffffffu, need) && j >= 1) {
        if (!fail && !wait_or_abort(&pv_done[rb][(g - 1) % NS], ((g - 1) / NS) & 1, p.err, abort_flag))
          fail = true;
        __syncwarp();
        tc_fence_after();
#pragma unroll 1
        for (int x = 0; x < D; x += 32) {
          uint32_t ov[32];
          tmem_ld32(tO(rb) + lane_base + x, ov);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tmem_st32(tO(rb) + lane_base + x, ov);
        }
      }
      if constexpr (D != 64) {
#pragma unroll
        for (int i = 0; i < BN / 2; ++i)
          v[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        tmem_st32(tS(rb, g % NS) + lane_base, v);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[rb][g % NS]);
    }
    // post 1 / l for the epilogue warps (once they have taken the previous
    // item's) and write the row's log-sum-exp
    if (it >= 1 && !fail && !wait_or_abort(&epi_empty[rb], (it - 1) & 1, p.err, abort_flag)) fail = true;
    s_inv[rb][r] = l > 0.f ? 1.f / l : 0.f;
    mbar_arrive(&epi_full[rb]);
    if (q < p.T && p.lse && !fail)
      p.lse[(size_t(b) * p.Hq + head) * p.Tq + (q - p.q_off)] =
          l > 0.f ? (m_used * c + __log2f(l)) * 0.6931471805599453f : -INFINITY;
    gt += n;
    }
  }

  // ---- common exit: on the error path give copies and MMAs still in flight a
  //      bounded time (about 2 ms) to land before shared memory and TMEM go
  tc_fence_before();
  if (__syncthreads_or(fail || *abort_flag))
    for (int i = 0; i < 2000; ++i) __nanosleep(1000);
  __syncthreads();
  if (warp == kWarpMma0) {
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
  int span, n_span, n_kt, n_pt, stride;
  size_t sum_bytes, plan_bytes;
};

// span = rows one CTA covers: 128 (two heads of a GQA pair) or 256 (two
// consecutive row blocks of one head).  The workspace is sized for the larger
// of the two so the query does not depend on the head layout.
PlanDims plan_dims(int B, int T, int block, int span, int Tq) {
  PlanDims d;
  d.span = span;
  d.n_span = (Tq + span - 1) / span;
  d.n_kt = (T + BN - 1) / BN;
  const int nb = block > 0 ? T / block : 0;
  d.n_pt = (nb + BN - 1) / BN;
  d.stride = 1 + d.n_kt + d.n_pt;
  d.sum_bytes = (size_t(B) * d.n_kt * sizeof(TileMeta) + 255) / 256 * 256;
  d.plan_bytes = size_t(B) * ((Tq + BM - 1) / BM) * d.stride * sizeof(int32_t);
  return d;
}

struct TcSetup {
  PlanDims pd;
  TcParams p;
  TileMeta *meta;
  int32_t *plan;
};

TcSetup tc_setup(const PrefillArgs &a, void *ws, int *err) {
  TcSetup S;
  const int G = a.Hq / a.Hkv;
  const bool pair_heads = G % 2 == 0;
  S.pd = plan_dims(a.batch, a.T, a.block, pair_heads ? BM : 2 * BM, a.T - a.q_off);
  S.meta = static_cast<TileMeta *>(ws);
  S.plan = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + S.pd.sum_bytes);
  TcParams &p = S.p;
  p.B = a.batch;
  p.T = a.T;
  p.q_off = a.q_off;
  p.Tq = a.T - a.q_off;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = G;
  p.W = a.window;
  p.block = a.block;
  p.n_pinned = a.block > 0 ? a.n_pinned : 0;
  p.nb = a.block > 0 ? (a.T - p.n_pinned) / a.block : 0;
  p.n_span = S.pd.n_span;
  p.span = S.pd.span;
  p.n_kt = S.pd.n_kt;
  p.plan_stride = S.pd.stride;
  p.pair_heads = pair_heads ? 1 : 0;
  p.n_pairs = pair_heads ? a.Hq / 2 : a.Hq;
  p.seg = a.seg_ids;
  p.sink = a.sink;
  p.plan = S.plan;
  p.meta = S.meta;
  p.out = static_cast<uint16_t *>(a.out);
  p.lse = a.lse;
  p.err = err;
  p.rope_cs = static_cast<const float2 *>(a.rope_cs);
  return S;
}

template <int D>
cudaError_t launch_tc(const PrefillArgs &a, void *ws, int *err, cudaStream_t stream) {
  const TcSetup S = tc_setup(a, ws, err);
  const TcParams &p = S.p;
  CUtensorMap tq, tk, tv, tpk, tpv;
  if (!make_map(&tq, a.q, a.batch, a.T - a.q_off, a.Hq, D, BM) || !make_map(&tk, a.k, a.batch, a.T, a.Hkv, D, BN) ||
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
  auto kern = a.block > 0 ? prefill_tc_kernel<D, true> : prefill_tc_kernel<D, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay<D>::kBytes);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (or per item, when there are fewer items)
  int sms = 0, dev = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long n_items = long(a.batch) * S.pd.n_span * p.n_pairs;
  const dim3 grid(unsigned(n_items < sms ? n_items : sms));
  return launch_pdl(kern, grid, dim3(kThreads), size_t(Lay<D>::kBytes), stream, tq, tk, tv, tpk, tpv, p);
}

}  // namespace

size_t prefill_plan_bytes(int batch, int T, int block) {
  PlanDims pd = plan_dims(batch, T, block, BM, T);  // the 128-row span has the most plan rows
  return pd.sum_bytes + pd.plan_bytes;
}

cudaError_t launch_prefill_tc_prep(const PrefillArgs &a, void *plan_ws, cudaStream_t stream) {
  if (size_t(a.batch) * a.T == 0) return cudaSuccess;
  const TcSetup S = tc_setup(a, plan_ws, nullptr);
  // tile records and plan: one block per sequence
  const size_t prep_smem = size_t(3) * S.pd.n_kt * sizeof(int);
  if (prep_smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(tile_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(prep_smem));
    if (e != cudaSuccess) return e;
  }
  tile_prep_kernel<<<a.batch, 1024, prep_smem, stream>>>(S.p, S.meta, S.plan);
  return cudaGetLastError();
}

// Every work item (sequence, span, head pair) multiplies each tile of its
// span's plan entry with both of its 128-row blocks (two heads of a GQA pair,
// or two row blocks of one head): per (sequence, span) the plan's count times
// Hq (pairs) or 2 Hq (row-block pairs) products of a 128 x 64 tile.
cudaError_t prefill_tile_count(const PrefillArgs &a, const void *plan_ws, long long *tiles) {
  *tiles = 0;
  if (size_t(a.batch) * a.T == 0) return cudaSuccess;
  const TcSetup S = tc_setup(a, const_cast<void *>(plan_ws), nullptr);
  const size_t rows = size_t(a.batch) * S.pd.n_span;
  std::vector<int32_t> n(rows);
  cudaError_t e = cudaMemcpy2D(n.data(), sizeof(int32_t), S.plan, size_t(S.pd.stride) * sizeof(int32_t),
                               sizeof(int32_t), rows, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return e;
  long long total = 0;
  for (size_t i = 0; i < rows; ++i) total += n[i];
  *tiles = total * (S.p.pair_heads ? a.Hq : 2LL * a.Hq);
  return cudaSuccess;
}

cudaError_t set_epilogue_wait_limit(unsigned polls) {
  return cudaMemcpyToSymbol(g_epi_wait_limit, &polls, sizeof(polls));
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, void *plan_ws, int *err, cudaStream_t stream) {
  if (size_t(a.batch) * a.T == 0) return cudaSuccess;
  if (a.d == 128) return launch_tc<128>(a, plan_ws, err, stream);
  if (a.d == 64) return launch_tc<64>(a, plan_ws, err, stream);
  return cudaErrorInvalidValue;
}

}  // namespace nd
