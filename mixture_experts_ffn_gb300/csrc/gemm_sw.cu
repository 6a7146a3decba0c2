// Grouped GEMM with the weights as the MMA's M operand and the tokens as its
// N operand, on SM pairs (tcgen05.mma.cta_group::2), for the expert-segmented
// row layout of TileOPs "MoE Operators", MoEGroupedGemmFwdOp:
//   out[rows of e] = act(a[rows of e] @ w[e]^T (+ bias[e]))
// with the gated activation (silu_and_mul / gelu_and_mul / clamped SwiGLU over
// stacked or interleaved gate/up rows) fused into the epilogue.
//
// Why this orientation: an expert's segment holds a few hundred rows whose
// count is arbitrary.  As the MMA's M dimension (128 rows per tile) a
// segment pads to a multiple of 128 (28% more MMA work on the DeepSeek-V3-
// style routing, 100% on gpt-oss-style); as its N dimension it pads to a
// multiple of 16 (5% and 12%), and tcgen05.mma time scales with N (N/2
// cycles per K16 step from N = 128 up, measured).  The weights fill M with
// no padding: 256 weight rows per CTA pair.
//
// Two forms, chosen per call (MH = M halves per CTA):
//
// Wide form (MH = 2; the default for long-K products whose segments
// average >= 128 rows):
//   pair tile = 512 weight rows (256 per CTA, two M halves) x one token chunk
//   of an expert (N <= 256 tokens, a multiple of 16; an expert of n rows is
//   cut into ceil(n / 256) chunks of equal size rounded up to 16).  Each K16
//   step issues two M256 x N MMAs, one per half, both reading the same token
//   slice, into two 256-column accumulators that fill TMEM.  A ring stage is
//   one 64-wide K atom: per CTA 2 x 16 KB of weights and its half of the
//   chunk's token rows (<= 16 KB); 4 stages.  Two thirds of every stage are
//   weights, against half in the narrow form, so more DRAM bytes are in
//   flight per SM.  Gated modes put a CTA's gate rows in one half and the
//   matching up rows in the other (a 4-D map [E][2][F][K]), so TMEM lane l of
//   both accumulators belongs to one activation column and each lane pairs
//   its own values.  With one accumulator pair the next tile's MMAs wait for
//   the drain: with tiled token rows three epilogue warpgroups share it.
// Narrow form (MH = 1):
//   pair tile = 256 weight rows (128 per CTA) x one token chunk; a stage
//   holds two K atoms (weights 2 x 16 KB, tokens up to 32 KB); 3 stages; two
//   256-column accumulators, so the epilogue of one tile overlaps the next
//   tile's MMAs.  Gated modes: a 5-D tensor map loads each group of 8 gate
//   rows next to its 8 up rows (TMEM lanes l and l ^ 8 of one warp), and the
//   epilogue pairs them with one shfl_xor per value.
// Both forms: contiguous token rows come by a tiled TMA box of 32, 64 or
// 128 rows per atom; rows gathered through the permutation (the forward's
// gate_up) come by cp.async from four loader warps, and the peer's loaders'
// arrivals reach the leader through a forwarding thread.  Both CTAs' copies
// complete on the leader's barriers; the leader issues eight MMAs per stage
// and multicasts the commit that frees it in both CTAs.  The ring is 192 KB.
// Tile schedule: pairs take tiles round-robin except for the last two
// rounds, whose tiles go to whichever pair asks first (a counter in the
// workspace's status area that the launch's last pair resets), so that
// pairs with light tiles do not idle while others finish heavy ones.  The
// leader's producer picks each tile and publishes it to every role of both
// CTAs through a small ring of shared-memory entries.
// Roles (192 threads per CTA; 320 with cp.async token rows; 448 in the wide
// form with tiled token rows)
//   warp 0 lane 0 : producer -- the weight boxes, the tiled token boxes, and
//                   in the leader the stage's expected bytes
//   warp 1        : TMEM allocation (pair); lane 0 of the leader issues MMAs,
//                   lane 0 of the peer forwards its cp.async arrivals
//   warps 2..5    : epilogue of the CTA's 128 TMEM lanes (bias, activation,
//                   rounding, transposed staging and TMA stores)
//   warps 6..9    : cp.async token loaders (gathered rows), or with 448
//                   threads, like warps 10..13, more epilogue warpgroups
//                   (the 32-token chunks of a tile taken in turn; loader
//                   warps that also drained between their copies were
//                   measured slower, 2.87 vs 2.81 ms)
// Every wait is bounded (2 s); on a timeout the block latches the timeout
// bit, drains what it issued and frees TMEM.
//
// Measured (DeepSeek-V3-style workload, CUDA events): gathered gate_up 2.87
// ms wide vs 3.25 ms narrow vs 3.32 ms for the one-SM row-tile kernel
// (gemm_tc.cu); down 1.53 vs 1.61 vs 1.75 ms.  With short K (Qwen3-style
// down) or 64-row segments (gpt-oss-style) the one-SM kernel is faster.
#include <cuda.h>

#include <algorithm>
#include <cstdlib>
#include <type_traits>

#include "common.cuh"
#include "gemm_epilogue.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moe {
namespace {

using namespace tc;

constexpr int BK = 64;                           // one 128-byte swizzle atom of K
constexpr int ROWS = 128;                        // weight rows per CTA and M half
constexpr int NMAX = 256;                        // tokens per chunk (MMA N)
constexpr int ATOM_BYTES = ROWS * BK * 2;        // 16 KB: 128 rows of one atom
constexpr int TMEM_COLS = 512;
constexpr int NUM_THREADS = 192;
constexpr int kMaxStages = 4;
constexpr int kOutBufs = 12;  // 2 KB output staging buffers: 4 warps x 2, or 12 warps x 1
// Dynamic tile schedule: the leader's producer takes the next tile of the
// list from a global counter when it is ready to load it and publishes it to
// both CTAs' rings of kSched entries.  No role of a pair trails the
// producer by more than STAGES + 3 tiles (its ring stages wait for the MMAs,
// which wait for the drain of the tile before last), so entries are never
// overwritten unread.
constexpr int kSched = 16;
constexpr int kNoTile = 0x7fffffff;

// Ring geometry by M halves per CTA (MH): MH = 1, 128 weight rows per CTA,
// stages of two K atoms (weights 32 KB + tokens up to 32 KB) x 3, and two
// accumulators so the epilogue of a tile overlaps the next tile's MMAs;
// MH = 2, 256 weight rows per CTA (two M256 MMAs per K16 step share each
// token slice), stages of one K atom (weights 32 KB + tokens up to 16 KB)
// x 4, and one accumulator pair filling TMEM.  Both rings are 192 KB.
template <int MH>
struct SwGeom {
  static constexpr int KA = MH == 2 ? 1 : 2;                    // K atoms per stage
  static constexpr int BKS = BK * KA;                           // K per stage
  static constexpr int STAGES = MH == 2 ? 4 : 3;
  static constexpr int A_BYTES = MH * KA * ATOM_BYTES;          // weights per stage
  static constexpr int B_BYTES = KA * (NMAX / 2) * BK * 2;      // tokens (half the chunk)
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int NACC = MH == 2 ? 1 : 2;                  // accumulator buffers
  static_assert(STAGES <= kMaxStages && STAGES * STAGE_BYTES == 192 * 1024, "ring");
};
constexpr int kRingBytes = 192 * 1024;

// Accumulator layouts: plain (lane = weight row = output column), or gated
// groups of 8 gate rows then their 8 up rows.
enum SwMode { kSwPlain = 0, kSwGated = 1 };

struct SwShared {
  uint64_t full[kMaxStages];   // leader: both CTAs' copies of a stage complete here
  uint64_t afull[kMaxStages];  // peer, cp.async rows: this CTA's rows of a stage landed
  uint64_t empty[kMaxStages];  // both: the leader's MMA commit frees the stage
  uint64_t tfull[2];       // both: accumulator ready
  uint64_t tempty[2];      // leader: both CTAs' epilogues drained the accumulator
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int prefix[kMaxExperts + 1];
  int scan_tmp[33];
  int sched[kSched];        // tile of schedule entry j at j % kSched (kNoTile: none left)
  uint64_t sfull[kSched];   // entry j written (phase (j / kSched) & 1)
};
constexpr size_t kSmemBytes =
    (size_t)kRingBytes + kOutBufs * OUT_BUF_BYTES + sizeof(SwShared) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
  return d;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait, acquiring at cluster scope (the entry may have been written
// by the peer CTA); false on abort or timeout.
__device__ __noinline__ bool wait_cluster(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
  const uint32_t addr = su32(b);
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait_cluster(addr, parity)) {
    if (*abort_flag) return false;
    if (global_ns() - t0 > kTimeoutNs) {
      *abort_flag = 1;
      latch_error(status, kDevTimeout);
      return false;
    }
  }
  return true;
}
// v to the peer's shared memory at addr_cluster, completing on the peer's
// barrier bar_cluster (4 bytes of transaction, and the one arrival the phase
// expects): no fence, the barrier's transaction count orders the data.
__device__ __forceinline__ void publish_remote_u32(uint32_t addr_cluster, uint32_t bar_cluster,
                                                   int v) {
  asm volatile(
      "mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], 4;\n\t"
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%1], %2, [%0];" ::"r"(
          bar_cluster),
      "r"(addr_cluster), "r"(v)
      : "memory");
}

// TMA loads into this CTA's shared memory that complete on the leader's
// barrier (shared::cluster address); coordinates innermost first.
__device__ __forceinline__ void tma2_2d(void* dst, const CUtensorMap* m, uint32_t bar, int c0,
                                        int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma2_3d(void* dst, const CUtensorMap* m, uint32_t bar, int c0,
                                        int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma2_4d(void* dst, const CUtensorMap* m, uint32_t bar, int c0,
                                        int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void tma2_5d(void* dst, const CUtensorMap* m, uint32_t bar, int c0,
                                        int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
// The eight K16 MMAs of a stage (two K atoms; atom a of A at ad + a * 16 KB,
// of B at bd + a * b_atom, descriptor units of 16 bytes) and the commit that
// frees the stage in both CTAs.
__device__ __forceinline__ void umma2_stage(uint32_t d_tmem, uint64_t ad, uint64_t bd,
                                            uint32_t b_atom16, uint32_t idesc,
                                            uint32_t accumulate, uint32_t bar) {
  const uint64_t ad1 = ad + (ATOM_BYTES >> 4), bd1 = bd + b_atom16;
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %6, %7, %3, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %8, %9, %3, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %10, %11, %3, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %12, %13, %3, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %14, %15, %3, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %16, %17, %3, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %18, %19, %3, t;\n\t"
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%5], %20;\n\t}" ::"r"(d_tmem),
      "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate), "r"(bar), "l"(ad + 2), "l"(bd + 2),
      "l"(ad + 4), "l"(bd + 4), "l"(ad + 6), "l"(bd + 6), "l"(ad1), "l"(bd1), "l"(ad1 + 2),
      "l"(bd1 + 2), "l"(ad1 + 4), "l"(bd1 + 4), "l"(ad1 + 6), "l"(bd1 + 6), "h"((uint16_t)3)
      : "memory");
}
// The eight K16 MMAs of a one-atom stage with two M halves per CTA: half h's
// weight atom at ad + h * 16 KB accumulates into d0 + h * NMAX, both halves
// reading the same token slice (bd); then the commit that frees the stage.
__device__ __forceinline__ void umma2_stage_wide(uint32_t d0, uint64_t ad, uint64_t bd,
                                                 uint32_t idesc, uint32_t accumulate,
                                                 uint32_t bar) {
  const uint64_t a1 = ad + (ATOM_BYTES >> 4);
  const uint32_t d1 = d0 + NMAX;
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "setp.eq.b32 t, %5, %5;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %2, %3, %4, p;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%1], %7, %3, %4, p;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %8, %9, %4, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%1], %10, %9, %4, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %11, %12, %4, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%1], %13, %12, %4, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %14, %15, %4, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%1], %16, %15, %4, t;\n\t"
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%6], %17;\n\t}" ::"r"(d0),
      "r"(d1), "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate), "r"(bar), "l"(a1), "l"(ad + 2),
      "l"(bd + 2), "l"(a1 + 2), "l"(ad + 4), "l"(bd + 4), "l"(a1 + 4), "l"(ad + 6), "l"(bd + 6),
      "l"(a1 + 6), "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void umma2_commit_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(su32(bar)),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void umma2_commit_self(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          su32(bar))
      : "memory");
}
// Instruction descriptor, kind::f16 with f32 accumulation, both operands
// K-major: bf16 (or float16 when f16) A and B, M x N.
__device__ __forceinline__ uint32_t idesc_sw(int M, int N, int f16) {
  const uint32_t fmt = f16 ? 0u : ((1u << 7) | (1u << 10));
  return (1u << 4) | fmt | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// One pair tile: expert e, weight-row tile nt (256 rows: 128 per CTA), and a
// chunk of the expert's rows [m0, m0 + nv) as the N dimension (N columns,
// nv <= N <= 256, N a multiple of 16 and at least 32).  nv == 0: an empty
// tile (every role skips it alike).
struct SwTile {
  int e, nt, ci, m0, nv, N;
};

// Tile t of the list built by build_tile_prefix(.., NMAX, n_ftiles, ..):
// expert e owns n_ftiles * ce tiles, ce = ceil(n / 256) chunks; inside an
// expert the chunk index runs fastest, so the pairs that share a weight tile
// run together and the L2 serves its re-reads.
__device__ __forceinline__ SwTile sw_decode(int t, const int* prefix, const int32_t* seg_end,
                                            int E, int M, int n_ftiles, int stride) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {  // last e with prefix[e] <= t (skips empty experts)
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  int s, u;
  seg_bounds(seg_end, lo, M, stride, s, u);
  const int n = u - s;
  const int ce = (n + NMAX - 1) / NMAX;
  const int local = t - prefix[lo];
  SwTile r;
  r.e = lo;
  r.nt = local / ce;
  const int ci = local % ce;
  r.ci = ci;
  const int per = (((n + ce - 1) / ce) + 15) & ~15;
  const int start = min(ci * per, n);
  r.m0 = s + start;
  r.nv = min(per, n - start);
  r.N = max(32, (r.nv + 15) & ~15);
  return r;
}

template <bool F16>
__device__ __forceinline__ void st16(__nv_bfloat16* p, float v) {
  if constexpr (F16)
    *reinterpret_cast<__half*>(p) = __float2half_rn(v);
  else
    *p = __float2bfloat16_rn(v);
}
template <bool F16>
__device__ __forceinline__ uint16_t bits16(float v) {
  if constexpr (F16)
    return __half_as_ushort(__float2half_rn(v));
  else
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

template <int ACT>
__device__ __forceinline__ float act1(float x) {
  if constexpr (ACT == MOE_ACT_RELU) return fmaxf(x, 0.0f);
  else if constexpr (ACT == MOE_ACT_GELU) return gelu_f(x);
  else if constexpr (ACT == MOE_ACT_SILU) return x * fast_sigmoid(x);
  else return x;
}

// One 32-token x 32-column box of the calling warp: lane l holds output
// column f0 + l (fok: inside the output), v[i] the value of token m0 + i.  A
// whole box goes through swizzled staging and one TMA store; a ragged tail
// (nval < 32 tokens) is stored row by row (64 contiguous bytes per token).
template <bool F16, int NBUF>
__device__ __forceinline__ void sw_emit32(const float (&v)[32], int nval, int m0, int f0, int f,
                                          int Nout, const CUtensorMap* tm_out, int tma_out,
                                          __nv_bfloat16* __restrict__ out, uint8_t* obufs,
                                          int& obuf, int lane) {
  if (tma_out && nval == 32 && f0 < Nout) {
    uint8_t* buf = obufs + obuf * OUT_BUF_BYTES;
    if (lane == 0) bulk_wait_read<NBUF - 1>();  // the store that last read this buffer
    __syncwarp();
    // token i, column lane: row i of the box, 64-byte swizzle
    const uint32_t base = su32(buf) + (uint32_t)((lane & 7) * 2);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      sts16(base + i * 64 + ((((lane >> 3) ^ ((i >> 1) & 3))) << 4), bits16<F16>(v[i]));
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tm_out, buf, f0, m0);
      bulk_commit();
    }
    obuf = NBUF == 1 ? 0 : obuf ^ 1;
  } else if (f < Nout) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < nval) st16<F16>(out + (size_t)(m0 + i) * Nout + f, v[i]);
  }
}

// Plain epilogue of the calling warp: TMEM lane l holds output column
// f0 + l for the tile's tokens (TMEM column j = token m0 + j), 32 tokens at a
// time, the 32-token chunks c0 = cs, cs + step, ...  Columns at or past Nout
// are not written.
template <int ACT, bool F16, int NBUF>
__device__ __forceinline__ void sw_drain_plain(uint32_t tbase, int nv, int cs, int step, int m0,
                                               int f0, int Nout,
                                               const __nv_bfloat16* __restrict__ bias_e,
                                               const CUtensorMap* tm_out, int tma_out,
                                               __nv_bfloat16* __restrict__ out, uint8_t* obufs,
                                               int& obuf, int lane) {
  const int f = f0 + lane;
  const float b = bias_e && f < Nout ? ld16<F16>(bias_e + f) : 0.0f;
#pragma unroll 1
  for (int c0 = cs; c0 < nv; c0 += step) {
    uint32_t r[32];
    tmem_ld32(tbase + (uint32_t)c0, r);
    tmem_wait_ld();
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = act1<ACT>(__uint_as_float(r[i]) + b);
    sw_emit32<F16, NBUF>(v, min(32, nv - c0), m0 + c0, f0, f, Nout, tm_out, tma_out, out, obufs,
                         obuf, lane);
  }
}

// Gated epilogue with the gate rows in one M half and the up rows in the
// other (two M halves per CTA): TMEM lane l of both accumulators belongs to
// activation column f0 + l, so each lane pairs its own gate and up values.
// Bias: b[gate row] and b[up row] of the column (stacked: f and F + f;
// interleaved: 2f and 2f + 1).  Chunks c0 = cs, cs + step, ...
template <int ACT, bool F16, int NBUF>
__device__ __forceinline__ void sw_drain_gated_split(
    uint32_t tgate, uint32_t tup, int nv, int cs, int step, int m0, int f0, int Nout, int F, int interleaved,
    const __nv_bfloat16* __restrict__ bias_e, float limit, float alpha, float beta,
    const CUtensorMap* tm_out, int tma_out, __nv_bfloat16* __restrict__ out, uint8_t* obufs,
    int& obuf, int lane) {
  const int f = f0 + lane;
  float bg = 0.0f, bu = 0.0f;
  if (bias_e && f < Nout) {
    bg = ld16<F16>(bias_e + (interleaved ? 2 * f : f));
    bu = ld16<F16>(bias_e + (interleaved ? 2 * f + 1 : F + f));
  }
#pragma unroll 1
  for (int c0 = cs; c0 < nv; c0 += step) {
    uint32_t rg[32], ru[32];
    tmem_ld32(tgate + (uint32_t)c0, rg);
    tmem_ld32(tup + (uint32_t)c0, ru);
    tmem_wait_ld();
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i)
      v[i] = gated<ACT>(__uint_as_float(rg[i]) + bg, __uint_as_float(ru[i]) + bu, limit, alpha,
                        beta);
    sw_emit32<F16, NBUF>(v, min(32, nv - c0), m0 + c0, f0, f, Nout, tm_out, tma_out, out, obufs,
                         obuf, lane);
  }
}

// Gated epilogue of the calling warp: lanes 0..7 and 16..23 hold gate rows,
// lanes l ^ 8 the matching up rows, of the 16 activation columns f0 ..
// f0 + 15 (lane l: column f0 + 8 (l >> 4) + (l & 7)).  Per 32 tokens the two
// partners swap half of their values (shfl_xor 8): the gate lane then holds
// (gate, up) of tokens 0..15, the up lane those of tokens 16..31, and each
// computes its 16 activations.  Whole 32-token boxes go through staging
// (16 columns x 32 tokens) and one TMA store; a ragged tail is stored
// directly.  Bias: b[gate row] / b[up row] of the lane's own weight row.
template <int ACT, bool F16>
__device__ __forceinline__ void sw_drain_gated(uint32_t tbase, int nv, int m0, int f0, int Nout,
                                               int F, int interleaved,
                                               const __nv_bfloat16* __restrict__ bias_e,
                                               float limit, float alpha, float beta,
                                               const CUtensorMap* tm_out, int tma_out,
                                               __nv_bfloat16* __restrict__ out, uint8_t* obufs,
                                               int& obuf, int lane) {
  const bool is_gate = (lane & 8) == 0;
  const int fl = 8 * (lane >> 4) + (lane & 7);  // column within the warp's 16
  const int f = f0 + fl;
  const bool fok = f < Nout;
  float b = 0.0f;
  if (bias_e && fok) {
    const int row = interleaved ? 2 * f + (is_gate ? 0 : 1) : (is_gate ? f : F + f);
    b = ld16<F16>(bias_e + row);
  }
#pragma unroll 1
  for (int c0 = 0; c0 < nv; c0 += 32) {
    uint32_t r[32];
    tmem_ld32(tbase + (uint32_t)c0, r);
    tmem_wait_ld();
    float a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float lo = __uint_as_float(r[i]) + b, hi = __uint_as_float(r[16 + i]) + b;
      const float recv = __shfl_xor_sync(0xffffffffu, is_gate ? hi : lo, 8);
      // one activation per value on selected operands (no per-lane branch)
      const float g = is_gate ? lo : recv, u = is_gate ? recv : hi;
      a[i] = gated<ACT>(g, u, limit, alpha, beta);
    }
    const int tok0 = is_gate ? 0 : 16;  // this lane's tokens: c0 + tok0 + i
    const int nval = min(32, nv - c0);
    if (tma_out && nval == 32 && f0 < Nout) {
      uint8_t* buf = obufs + obuf * OUT_BUF_BYTES;
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
      const uint32_t base = su32(buf) + (uint32_t)(tok0 * 32 + fl * 2);
#pragma unroll
      for (int i = 0; i < 16; ++i) sts16(base + i * 32, bits16<F16>(a[i]));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tm_out, buf, f0, m0 + c0);
        bulk_commit();
      }
      obuf ^= 1;
    } else if (fok) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (tok0 + i < nval) st16<F16>(out + (size_t)(m0 + c0 + tok0 + i) * Nout + f, a[i]);
    }
  }
}

// How the token rows reach shared memory.
enum SwTok {
  kTokTiled = 0,    // contiguous rows: one tiled TMA box per stage
  kTokCpAsync = 1,  // rows through the row map: cp.async by four loader warps
};
constexpr int kLoaderWarp0 = NUM_THREADS / 32;
constexpr int NUM_THREADS_LOAD = NUM_THREADS + 128;
// Epilogue warpgroups: three (warps 2..5, 6..9 and 10..13, taking the
// 32-token chunks in turn) when the next tile's MMAs wait for the drain (two
// M halves, one accumulator pair) and no loader warps are needed (tiled
// token rows); else one (warps 2..5).
template <int TOK, int MH>
struct SwRoles {
  static constexpr int EPI_GROUPS = TOK == kTokTiled && MH == 2 ? 3 : 1;
  static constexpr int THREADS = EPI_GROUPS == 3 ? NUM_THREADS + 256
                                 : TOK == kTokCpAsync ? NUM_THREADS_LOAD
                                                      : NUM_THREADS;
  static constexpr int NBUF = EPI_GROUPS > 1 ? 1 : 2;  // staging buffers per epilogue warp
};

__device__ __forceinline__ void mbar_arrive_remote_cta(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

// Token-row boxes of 32, 64 and 128 rows x one K atom: 2-D maps [rows][K] of
// the rows' source.
struct TokMaps {
  CUtensorMap m[3];
};

// The token rows of a stage sit as KA atoms of h rows each (h = 32, 64 or
// 128, the smallest that holds the CTA's half of the chunk).
__device__ __forceinline__ int tok_box_sel(int half) { return half <= 32 ? 0 : half <= 64 ? 1 : 2; }

// tm_w: weights, 3-D [E][N1][K] box {64, 128, 1} (plain), or the 5-D gated
// view [E][F/8][2][8][K] box {64, 8, 2, 8, 1} (a group is 8 activation
// columns: their 8 gate rows, then their 8 up rows); one box per K atom, so
// columns past K and rows past the expert's read as zeros.  Row r of the
// segmented row space is source row grows[r] / gdiv (the hidden states read
// through the permutation; rows with an out-of-range entry read zeros) or,
// without grows, row r of the source itself.
template <int MODE, int ACT, bool F16, int TOK, int MH>
__global__ void __launch_bounds__(SwRoles<TOK, MH>::THREADS, 1)
    gemm_sw_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ TokMaps tm_a,
                   const __grid_constant__ CUtensorMap tm_out, int tma_out,
                   const __nv_bfloat16* __restrict__ bias, const int32_t* __restrict__ seg_end,
                   int M, int Nout, int N1, int K, int E, int interleaved, float limit,
                   float alpha, float beta, __nv_bfloat16* __restrict__ out, int* status,
                   const __nv_bfloat16* __restrict__ asrc, const int32_t* __restrict__ grows,
                   int gdiv, int src_rows, int seg_stride) {
  using G = SwGeom<MH>;
  constexpr int STAGES = G::STAGES, STAGE_BYTES = G::STAGE_BYTES, A_BYTES = G::A_BYTES;
  constexpr int KA = G::KA, BKS = G::BKS, NACC = G::NACC;
  using R = SwRoles<TOK, MH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* out_stage = smem + (size_t)kRingBytes;  // 1024-byte aligned
  SwShared* sh = reinterpret_cast<SwShared*>(out_stage + kOutBufs * OUT_BUF_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  volatile int* abort_flag = &sh->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // the leader's expect-tx arrival (+ both CTAs' TMA bytes); with cp.async
      // rows also one arrival per leader loader thread and the peer's
      // forwarded arrival
      mbar_init(&sh->full[s], TOK == kTokCpAsync ? 1 + 128 + 1 : 1);
      mbar_init(&sh->afull[s], 128);
      mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->tfull[a], 1);
      mbar_init(&sh->tempty[a], 2 * 128 * R::EPI_GROUPS);
    }
    mbar_init(&sh->drain, 1);
    for (int i = 0; i < kSched; ++i) mbar_init(&sh->sfull[i], 1);
    sh->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
    if constexpr (TOK == kTokTiled)
      for (int i = 0; i < 3; ++i)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_a.m[i]))
                     : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(&sh->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  // a pair tile covers 2 * ROWS * MH weight rows: as many output columns
  // (plain), or half as many activation columns (gated)
  const int n_ftiles = MODE == kSwPlain ? (Nout + 2 * ROWS * MH - 1) / (2 * ROWS * MH)
                                        : (Nout + ROWS * MH - 1) / (ROWS * MH);
  // everything above overlaps the previous launch; seg_end and the operands
  // are read only after this
  pdl_wait();
  const int total =
      build_tile_prefix(seg_end, E, M, NMAX, n_ftiles, sh->prefix, sh->scan_tmp, seg_stride);
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  const int nks = (K + BKS - 1) / BKS;  // ring stages per tile
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  auto decode = [&](int t) { return sw_decode(t, sh->prefix, seg_end, E, M, n_ftiles, seg_stride); };
  // schedule: gctr[0] is the next tile of the list, gctr[1] the pairs done
  // taking tiles; the last of them zeroes both for the next launch (a launch
  // that failed leaves them for the status clear the error requires)
  int* gctr = status + 8;
  // entry j of the schedule (kNoTile: no tiles left, or the wait failed)
  auto next_tile = [&](int j) -> int {
    if (!wait_cluster(&sh->sfull[j % kSched], (uint32_t)(j / kSched) & 1u, abort_flag, status))
      return kNoTile;
    return *reinterpret_cast<volatile int*>(&sh->sched[j % kSched]);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------- producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = 0;
      bool ok = true, done = false;
      // The leader's tiles: round-robin for all but the last two rounds (the
      // pairs that share a weight tile stay in step), then the next tile of
      // the rest from the counter (the pairs finish together).  It takes a
      // tile one ahead (the counter's latency hides behind the current
      // tile's copies), skips empty ones, and publishes it.
      const int r_static = max(0, total / npairs - 2);
      int k_static = 0;
      auto grab = [&]() {
        return k_static < r_static ? pair + npairs * k_static++
                                   : npairs * r_static + atomicAdd(gctr, 1);
      };
      int ahead = leader ? grab() : 0;
      for (int j = 0; ok; ++j) {
        int tile;
        if (leader) {
          tile = ahead;
          while (tile < total && decode(tile).nv == 0) tile = grab();
          if (tile >= total) tile = kNoTile;
          else ahead = grab();
          const int slot = j % kSched;
          *reinterpret_cast<volatile int*>(&sh->sched[slot]) = tile;
          mbar_arrive(&sh->sfull[slot]);
          publish_remote_u32(map_to_rank(su32(&sh->sched[slot]), 1),
                             map_to_rank(su32(&sh->sfull[slot]), 1), tile);
        } else {
          tile = next_tile(j);
        }
        if (tile >= total) { done = tile == kNoTile; break; }
        const SwTile st = decode(tile);
        const int half = st.N >> 1;  // token rows of this CTA
        const int bsel = tok_box_sel(half);
        const uint32_t tx =
            (uint32_t)A_BYTES + (TOK == kTokTiled ? (uint32_t)KA * (32u << bsel) * BK * 2 : 0u);
        for (int ks = 0; ks < nks; ++ks) {
          if (!wait_fast(&sh->empty[stage], phase ^ 1u, abort_flag, status)) { ok = false; break; }
          uint8_t* a_dst = smem + (size_t)stage * STAGE_BYTES;
          uint8_t* b_dst = a_dst + A_BYTES;
          const uint32_t bar = map_to_rank(su32(&sh->full[stage]), 0);
          if (leader) mbar_expect_tx(&sh->full[stage], 2 * tx);
#pragma unroll
          for (int a = 0; a < KA; ++a) {  // one box per K atom, M half and operand
            const int k0 = ks * BKS + a * BK;
#pragma unroll
            for (int h = 0; h < MH; ++h) {
              uint8_t* dst = a_dst + (a * MH + h) * ATOM_BYTES;
              if constexpr (MODE == kSwPlain)
                tma2_3d(dst, &tm_w, bar, k0,
                        (st.nt * MH + h) * 2 * ROWS + ROWS * (int)rank, st.e);
              else if constexpr (MH == 2)  // half 0 the gate rows, half 1 the up rows
                tma2_4d(dst, &tm_w, bar, k0, st.nt * 2 * ROWS + ROWS * (int)rank, h, st.e);
              else
                tma2_5d(dst, &tm_w, bar, k0, 0, 0, st.nt * 16 + 8 * (int)rank, st.e);
            }
            if constexpr (TOK == kTokTiled)
              tma2_2d(b_dst + a * ((32 << bsel) * BK * 2), &tm_a.m[bsel], bar, k0,
                      st.m0 + (int)rank * half);
          }
          ++issued[stage];
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (leader && done && !*abort_flag) {
        __threadfence();  // this pair's last grab before its done count
        if (atomicAdd(gctr + 1, 1) == npairs - 1) {
          __threadfence();  // every pair's grabs before the reset
          atomicExch(gctr, 0);
          atomicExch(gctr + 1, 0);
        }
      }
      if (!ok && leader) {  // both CTAs' copies complete on the leader's barriers
        for (int s = 0; s < STAGES; ++s)
          if (issued[s]) drain_wait(&sh->full[s], (issued[s] - 1u) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------- MMA issuer (leader)
      int stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      bool ok = true, any = false;
      const uint64_t adesc0 = sw128_desc(su32(smem));
      const uint64_t bdesc0 = sw128_desc(su32(smem + A_BYTES));
      uint32_t empty_addr[STAGES];
      for (int s = 0; s < STAGES; ++s) empty_addr[s] = su32(&sh->empty[s]);
      for (int j = 0; ok; ++j) {
        const int tile = next_tile(j);
        if (tile >= total) break;
        const SwTile st = decode(tile);
        const uint32_t idesc = idesc_sw(2 * ROWS, st.N, F16 ? 1 : 0);  // M256 per MMA
        // token atoms h rows apart (16-byte descriptor units)
        const uint32_t b_atom16 = (uint32_t)((32 << tok_box_sel(st.N >> 1)) * BK * 2) >> 4;
        if (!wait_fast(&sh->tempty[acc], aphase ^ 1u, abort_flag, status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * NMAX);
        for (int ks = 0; ks < nks; ++ks) {
          if (!wait_fast(&sh->full[stage], phase, abort_flag, status)) { ok = false; break; }
          // cp.async rows of this CTA were written through the generic proxy;
          // the MMA reads them through the async proxy (the peer's forwarder
          // fences the peer's rows)
          if constexpr (TOK == kTokCpAsync) fence_proxy_async_smem();
          tc_fence_after();
          const uint64_t off = (uint64_t)((stage * STAGE_BYTES) >> 4);
          if constexpr (MH == 2)
            umma2_stage_wide(d_tmem, adesc0 + off, bdesc0 + off, idesc, ks != 0 ? 1u : 0u,
                             empty_addr[stage]);
          else
            umma2_stage(d_tmem, adesc0 + off, bdesc0 + off, b_atom16, idesc, ks != 0 ? 1u : 0u,
                        empty_addr[stage]);
          any = true;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma2_commit_both(&sh->tfull[acc]);
        if (++acc == NACC) { acc = 0; aphase ^= 1u; }
      }
      if (!ok && any) {
        umma2_commit_self(&sh->drain);
        drain_wait(&sh->drain, 0);
      }
    }
    if constexpr (TOK == kTokCpAsync) {
      if (lane == 0 && !leader) {
        // -------------------------------------------- forwarder (peer)
        // the peer's rows of a stage have landed: order them for the async
        // proxy and pass one arrival to the leader's full barrier (released
        // at CTA scope: a cluster-scope release would wait for every copy
        // this SM has in flight)
        int stage = 0;
        uint32_t phase = 0;
        const uint32_t full_remote0 = map_to_rank(su32(&sh->full[0]), 0);
        bool ok = true;
        for (int j = 0; ok; ++j) {
          if (next_tile(j) >= total) break;
          for (int ks = 0; ks < nks; ++ks) {
            if (!wait_fast(&sh->afull[stage], phase, abort_flag, status)) { ok = false; break; }
            fence_proxy_async_smem();
            mbar_arrive_remote_cta(full_remote0 + (uint32_t)(stage * sizeof(uint64_t)));
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
      }
    }
  } else if (TOK == kTokCpAsync && warp >= kLoaderWarp0) {
    // ------------------------------------------------ token loaders (cp.async)
    // thread lt copies 16-byte chunk lt % 8 of rows lt / 8 + 16 i of this
    // CTA's half, for both K atoms of a stage, into the 128-byte swizzle
    // (chunk ch of row r at ch ^ (r % 8)); padding rows and columns past K
    // are zero-filled
    const int lt = threadIdx.x - kLoaderWarp0 * 32;
    const int ch = lt & 7, r0 = lt >> 3;
    const uint32_t dst0 = (uint32_t)(r0 * 128 + ((ch ^ (r0 & 7)) << 4));
    uint64_t keep_policy;  // the hidden rows stay in L2 ahead of the weight stream
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep_policy));
    uint64_t* arrive_bar = leader ? sh->full : sh->afull;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int j = 0; ok; ++j) {
      const int tile = next_tile(j);
      if (tile >= total) break;
      const SwTile st = decode(tile);
      const int half = st.N >> 1;
      const uint32_t atom_bytes = (uint32_t)(32 << tok_box_sel(half)) * BK * 2;
      const __nv_bfloat16* src[8];
      uint32_t valid = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = r0 + 16 * i;
        const int j = (int)rank * half + r;
        int t = 0;
        if (r < half && j < st.nv) {
          const int row = st.m0 + j;
          if (grows) {
            const int rt = grows[row];
            if (rt >= 0 && rt / gdiv < src_rows) { t = rt / gdiv; valid |= 1u << i; }
          } else {
            t = row;
            valid |= 1u << i;
          }
        }
        src[i] = asrc + (size_t)t * K + ch * 8;
      }
      for (int ks = 0; ks < nks; ++ks) {
        if (!wait_fast(&sh->empty[stage], phase ^ 1u, abort_flag, status)) { ok = false; break; }
        const uint32_t b_dst = su32(smem + (size_t)stage * STAGE_BYTES + A_BYTES) + dst0;
#pragma unroll
        for (int a = 0; a < KA; ++a) {
          const int k0 = ks * BKS + a * BK;
          const bool kin = k0 + ch * 8 < K;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (r0 + 16 * i >= half) break;
            const bool v = kin && ((valid >> i) & 1u);
            asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(
                             b_dst + a * atom_bytes + i * 16 * 128),
                         "l"(v ? src[i] + k0 : asrc), "r"(v ? 16 : 0), "l"(keep_policy)
                         : "memory");
          }
        }
        // arrives on the stage's barrier of this CTA once this thread's copies land
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                         su32(&arrive_bar[stage]))
                     : "memory");
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // nothing in flight at exit
  } else {
    // ------------------------------------------------ epilogue (both CTAs)
    const int quad = warp & 3;
    const int grp = (warp - 2) >> 2;  // epilogue warpgroup
    const int cs = 32 * grp, step = 32 * R::EPI_GROUPS;
    int acc = 0;
    uint32_t aphase = 0;
    const uint32_t tempty_remote[2] = {map_to_rank(su32(&sh->tempty[0]), 0),
                                       map_to_rank(su32(&sh->tempty[1]), 0)};
    // staging buffers of 2 KB: two per warp of one group, or one per warp
    uint8_t* obufs = out_stage + (grp * 4 + quad) * R::NBUF * OUT_BUF_BYTES;
    int obuf = 0;
    for (int j = 0;; ++j) {
      const int tile = next_tile(j);
      if (tile >= total) break;
      const SwTile st = decode(tile);
      if (!wait_fast(&sh->tfull[acc], aphase, abort_flag, status)) break;
      tc_fence_after();
      const __nv_bfloat16* be = bias ? bias + (size_t)st.e * N1 : nullptr;
      const uint32_t tq = tmem_base + ((uint32_t)(quad * 32) << 16);
      if constexpr (MODE == kSwGated && MH == 2) {
        sw_drain_gated_split<ACT, F16, R::NBUF>(tq, tq + NMAX, st.nv, cs, step, st.m0,
                                       st.nt * 2 * ROWS + ROWS * (int)rank + 32 * quad, Nout, Nout,
                                       interleaved, be, limit, alpha, beta, &tm_out, tma_out, out,
                                       obufs, obuf, lane);
      } else {
#pragma unroll 1
        for (int h = 0; h < MH; ++h) {
          // MH = 2: half h in columns h * NMAX of the one accumulator pair
          const uint32_t tb = tq + (uint32_t)((MH == 2 ? h : acc) * NMAX);
          const int g = st.nt * MH + h;  // 256-weight-row group of the expert
          if constexpr (MODE == kSwPlain)
            sw_drain_plain<ACT, F16, R::NBUF>(tb, st.nv, cs, step, st.m0,
                                     g * 2 * ROWS + ROWS * (int)rank + 32 * quad, Nout, be,
                                     &tm_out, tma_out, out, obufs, obuf, lane);
          else
            sw_drain_gated<ACT, F16>(tb, st.nv, st.m0,
                                     g * ROWS + (ROWS / 2) * (int)rank + 16 * quad, Nout, Nout,
                                     interleaved, be, limit, alpha, beta, &tm_out, tma_out, out,
                                     obufs, obuf, lane);
        }
      }
      // the drain's TMEM loads have completed (tcgen05.wait::ld): a CTA-scope
      // release orders them before the leader's next MMAs (a cluster-scope
      // one would also wait for every copy this SM has in flight)
      tc_fence_before();
      mbar_arrive_remote_cta(tempty_remote[acc]);
      if (++acc == NACC) { acc = 0; aphase ^= 1u; }
    }
    if (lane == 0) bulk_wait_all();  // every staged box written before the pair exits
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA frees TMEM or exits while its peer still works
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

}  // namespace

// ------------------------------------------------------------ host side
namespace {

template <int MODE, int ACT, bool F16, int TOK, int MH>
const void* sw_kernel_ptr() {
  return (const void*)gemm_sw_kernel<MODE, ACT, F16, TOK, MH>;
}

template <bool F16, int TOK, int MH>
const void* pick_sw(int mode, int kind) {
  if (mode == kSwPlain) {
    switch (kind) {
      case MOE_ACT_RELU: return sw_kernel_ptr<kSwPlain, MOE_ACT_RELU, F16, TOK, MH>();
      case MOE_ACT_GELU: return sw_kernel_ptr<kSwPlain, MOE_ACT_GELU, F16, TOK, MH>();
      case MOE_ACT_SILU: return sw_kernel_ptr<kSwPlain, MOE_ACT_SILU, F16, TOK, MH>();
      default: return sw_kernel_ptr<kSwPlain, MOE_ACT_IDENTITY, F16, TOK, MH>();
    }
  }
  switch (kind) {
    case MOE_ACT_SWIGLU: return sw_kernel_ptr<kSwGated, MOE_ACT_SWIGLU, F16, TOK, MH>();
    case MOE_ACT_GELU_AND_MUL:
      return sw_kernel_ptr<kSwGated, MOE_ACT_GELU_AND_MUL, F16, TOK, MH>();
    default: return sw_kernel_ptr<kSwGated, MOE_ACT_SILU_AND_MUL, F16, TOK, MH>();
  }
}

template <int MH>
const void* pick_sw_mh(bool f16, int tok, int mode, int kind) {
  return tok == kTokTiled ? (f16 ? pick_sw<true, kTokTiled, MH>(mode, kind)
                                 : pick_sw<false, kTokTiled, MH>(mode, kind))
                          : (f16 ? pick_sw<true, kTokCpAsync, MH>(mode, kind)
                                 : pick_sw<false, kTokCpAsync, MH>(mode, kind));
}

}  // namespace

cudaError_t launch_gemm_sw(const void* a, const void* w, const void* bias, const int32_t* seg_end,
                           int M, int N, int K, int E, const moe_act_params* act, void* out,
                           int* status, cudaStream_t s, const int32_t* gather_rows,
                           int gather_div, int gather_src_rows, int seg_stride, bool f16,
                           bool wide) {
  if (M == 0 || N == 0) return cudaSuccess;
  int mode = kSwPlain, kind = MOE_ACT_IDENTITY, N1 = N, inter = 0;
  float limit = 0.f, alpha = 1.f, beta = 0.f;
  if (act) kind = act->kind;
  if (act && act_is_gated(act->kind)) {
    mode = kSwGated;
    inter = (kind == MOE_ACT_SWIGLU && act->swiglu_fusion == 1) ? 1 : 0;
    N1 = 2 * N;
    limit = act->limit;
    alpha = act->alpha;
    beta = act->beta;
  }
  if (N % 8 != 0 || K % 8 != 0) return cudaErrorInvalidValue;
  CUtensorMap mw, mo;
  const uint64_t K2 = (uint64_t)K * 2;
  if (mode == kSwPlain) {
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)N1, (cuuint64_t)E};
    cuuint64_t str[2] = {K2, (cuuint64_t)N1 * K2};
    cuuint32_t box[3] = {BK, ROWS, 1};
    if (!tmap::encode_bf16(&mw, w, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B, f16))
      return cudaErrorInvalidValue;
  } else if (wide) {
    // [E][2][F][K]: the gate rows (index 0) and the up rows (index 1) of the
    // activation columns (stacked: up rows F below the gate rows;
    // interleaved: rows 2j, 2j + 1), one 128-row box per M half
    cuuint64_t dims[4] = {(cuuint64_t)K, (cuuint64_t)N, 2, (cuuint64_t)E};
    cuuint64_t st_stacked[3] = {K2, (cuuint64_t)N * K2, (cuuint64_t)N1 * K2};
    cuuint64_t st_inter[3] = {2 * K2, K2, (cuuint64_t)N1 * K2};
    cuuint32_t box[4] = {BK, ROWS, 1, 1};
    if (!tmap::encode_bf16(&mw, w, 4, dims, inter ? st_inter : st_stacked, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, f16))
      return cudaErrorInvalidValue;
  } else {
    // groups of 8 activation columns: their 8 gate rows, then their 8 up rows
    // (stacked: up rows F below the gate rows; interleaved: rows 2j, 2j + 1)
    cuuint64_t dims[5] = {(cuuint64_t)K, 8, 2, (cuuint64_t)N / 8, (cuuint64_t)E};
    cuuint64_t st_stacked[4] = {K2, (cuuint64_t)N * K2, 8 * K2, (cuuint64_t)N1 * K2};
    cuuint64_t st_inter[4] = {2 * K2, K2, 16 * K2, (cuuint64_t)N1 * K2};
    cuuint32_t box[5] = {BK, 8, 2, 8, 1};
    if (!tmap::encode_bf16(&mw, w, 5, dims, inter ? st_inter : st_stacked, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, f16))
      return cudaErrorInvalidValue;
  }
  // token rows: boxes of 32 / 64 / 128 rows of one K atom (contiguous rows);
  // cp.async reads gathered rows without a map
  const int tok = gather_rows ? kTokCpAsync : kTokTiled;
  TokMaps ma;
  if (tok == kTokTiled) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)std::max(M, 1)};
    cuuint64_t str[1] = {K2};
    for (int i = 0; i < 3; ++i) {
      cuuint32_t box[2] = {BK, 32u << i};
      if (!tmap::encode_bf16(&ma.m[i], a, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B, f16))
        return cudaErrorInvalidValue;
    }
  } else {
    ma.m[0] = ma.m[1] = ma.m[2] = mw;  // unused
  }
  // staged output boxes: 32 columns x 32 rows (64-byte swizzle), or 16 x 32
  // for the gated mode with gate and up rows in one M half; rows stored
  // directly when the output's base or pitch is not 16-byte aligned
  int tma_out = 0;
  if ((reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    const bool box32 = mode == kSwPlain || wide;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t str[1] = {(cuuint64_t)N * 2};
    cuuint32_t box[2] = {box32 ? 32u : 16u, 32u};
    tma_out = tmap::encode_bf16(&mo, out, 2, dims, str, box,
                                box32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                f16)
                  ? 1
                  : 0;
  }
  if (!tma_out) mo = mw;  // unused
  const int mh = wide ? 2 : 1;
  const void* kern = wide ? pick_sw_mh<2>(f16, tok, mode, kind) : pick_sw_mh<1>(f16, tok, mode, kind);
  set_smem_limit(kern, (int)kSmemBytes);
  const int n_ftiles = mode == kSwPlain ? (N + 2 * ROWS * mh - 1) / (2 * ROWS * mh)
                                        : (N + ROWS * mh - 1) / (ROWS * mh);
  const long long max_tiles = (long long)((M + NMAX - 1) / NMAX + E) * n_ftiles;
  const int pairs = (int)std::max<long long>(1, std::min<long long>(max_tiles, num_sms() / 2));

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(tok == kTokTiled && wide ? NUM_THREADS + 256
                      : tok == kTokCpAsync    ? NUM_THREADS_LOAD
                                              : NUM_THREADS);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pdl
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const __nv_bfloat16* bias_p = static_cast<const __nv_bfloat16*>(bias);
  __nv_bfloat16* out_p = static_cast<__nv_bfloat16*>(out);
  const __nv_bfloat16* a_p = static_cast<const __nv_bfloat16*>(a);
  void* args[] = {&mw, &ma, &mo, &tma_out, &bias_p, &seg_end, &M, &N, &N1, &K, &E, &inter,
                  &limit, &alpha, &beta, &out_p, &status, &a_p, &gather_rows, &gather_div,
                  &gather_src_rows, &seg_stride};
  cudaError_t e = cudaLaunchKernelExC(&cfg, kern, args);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
