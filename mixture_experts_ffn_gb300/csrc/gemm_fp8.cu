// Block-scaled FP8 grouped GEMM over a masked slab (TileOPs "MoE Operators",
// MoEGroupedGemmFP8FwdOp): out[g, :m_g] = a[g, :m_g] @ b[g]^T with a [E, max_m, K]
// and b [E, N, K] in float8_e4m3fn, one fp32 scale per row and 128 K-columns of
// a (a_scale [E, max_m, K/128]) and one per 128 x 128 block of b
// (b_scale [E, N/128, K/128]); m_g = layout_metadata[g] read as
// min(max(m_g, 0), max_m).  Each 128-wide K block is contracted from the raw
// FP8 values, then multiplied by its two scales and added to an fp32
// accumulator; the result is written in bf16.
//
// Work decomposition (SM pairs, tcgen05.mma.cta_group::2)
//   pair tile = 256 rows of one expert's slab x 256 columns: CTA r of the
//   pair holds rows m0 + 128 r .. (its A half) and weight rows n0 + 128 r ..
//   (its B half), so each SM loads 16 KB of A and 16 KB of B per 128-wide K
//   block for an M256 x N256 product: half the operand bytes per FLOP of a
//   one-SM M128 x N128 tile, which is what bounds the contraction (its
//   operand stream, not the tensor pipe, set the pace of the one-SM form).
//   K block = 128 e4m3 values = one 128-byte swizzle row; 6-stage ring of
//   32 KB per CTA.
//   Per K block the leader issues four kind::f8f6f4 M256 N256 K32 MMAs into
//   a fresh partial sum in one of two 256-column TMEM buffers and multicasts
//   the commit to both CTAs.  Each CTA's promotion warps read its own 128
//   lanes, scale them by a_scale[row, kb] * b_scale[column block, kb] (one
//   column block per warp, so one scale per thread and K block) and add them
//   into fp32 registers, then release the buffer on the leader, while the
//   MMAs of the next block fill the other buffer.
// Roles (320 threads per CTA)
//   warp 0 lane 0 : TMA producer of this CTA's halves (both CTAs' copies
//                   complete on the leader's barrier)
//   warp 1        : TMEM allocation (pair); lane 0 of the leader issues MMAs
//   warps 2..9    : promotion and epilogue; warp w owns TMEM lanes
//                   32*(w%4).. (rows) and columns 128*((w-2)/4).. (128 fp32
//                   registers of accumulator per thread), and writes its rows
//                   as bf16 through staged 32 x 32 TMA stores
// Tiles go round-robin over the pairs; inside an expert the row tiles of one
// column tile are consecutive, so pairs that share a weight tile run
// together and the L2 serves its re-reads.  A tile whose second row half is
// past the expert's count still runs the M256 MMA (the peer's rows are not
// written).
// Every mbarrier wait is bounded (2 s): a wait that runs out sets the timeout
// bit and the block's abort flag, and the block drains its copies and MMAs
// in flight before the pair frees TMEM.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "gemm_epilogue.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128;            // rows per CTA (256 per pair)
constexpr int BN = 256;            // columns per pair tile (128 weight rows per CTA)
constexpr int BKB = 128;           // K per block (one scale block)
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BKB;  // 16 KB of e4m3
constexpr int B_BYTES = (BN / 2) * BKB;  // 16 KB: this CTA's half of the weight rows
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;  // two partial-sum buffers
constexpr int kEpiWarps = 8;
constexpr int kEpiWarp0 = 2;  // promotion warps 2..9
// ten warps: three share an SM sub-partition's 16384 registers, so a thread
// gets at most 168 (the 128 accumulators and two 16-column chunks in flight)
constexpr int NUM_THREADS = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kColsPerWarp = BN / 2;  // accumulator columns of one promotion warp
// kind::f8f6f4 instruction descriptor: fp32 D (bit 4), e4m3 A and B (format
// 0 in bits 7..9 and 10..12), both K-major, N / 8 at bit 17, M / 16 at bit 24
// (M = 256 across the pair)
constexpr uint32_t kIdescFp8 =
    (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((2 * BM) >> 4) << 24);

struct Fp8Shared {
  uint64_t full[STAGES];   // leader: both CTAs' copies of a stage complete here
  uint64_t empty[STAGES];  // both: the leader's MMA commit frees the stage
  uint64_t pfull[2];       // both: partial sum of a K block ready (multicast commit)
  uint64_t pempty[2];      // leader: every promotion warp of the pair read it
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int prefix[kMaxExperts + 1];
  int scan_tmp[33];
};
constexpr size_t kSmemBytes = (size_t)STAGES * STAGE_BYTES + OUT_BYTES + sizeof(Fp8Shared) + 1024;
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
// arrival on a barrier of either CTA of the pair (shared::cluster address),
// released at CTA scope: it orders this thread's earlier tcgen05 loads (after
// tcgen05.fence::before_thread_sync) without waiting for the SM's copies
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}
// A TMA load into this CTA's shared memory that completes on the leader's
// barrier (shared::cluster address); coordinates innermost first.
__device__ __forceinline__ void tma2_3d(void* dst, const CUtensorMap* m, uint32_t bar, int c0,
                                        int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// The four K32 MMAs of one 128-wide K block into a fresh partial sum (M256
// across the pair), then the commits that free the stage and publish the
// partial sum in both CTAs.
__device__ __forceinline__ void umma2_fp8_block(uint32_t d_tmem, uint64_t ad, uint64_t bd,
                                                uint32_t empty_bar, uint32_t pfull_bar) {
  asm volatile(
      "{\n\t.reg .pred f, t;\n\t"
      "setp.ne.b32 f, %3, %3;\n\t"
      "setp.eq.b32 t, %3, %3;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, f;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %4, %5, %3, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %6, %7, %3, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %8, %9, %3, t;\n\t"
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%10], %12;\n\t"
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%11], %12;\n\t}" ::"r"(d_tmem),
      "l"(ad), "l"(bd), "r"(kIdescFp8), "l"(ad + 2), "l"(bd + 2), "l"(ad + 4), "l"(bd + 4),
      "l"(ad + 6), "l"(bd + 6), "r"(empty_bar), "r"(pfull_bar), "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void umma2_commit_self(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          su32(bar))
      : "memory");
}
// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// tcgen05.wait::ld with r as in-out operands, so that no use of r can be
// scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld_regs16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ int valid_rows(const int32_t* __restrict__ counts, int g, int max_m) {
  return min(max(counts[g], 0), max_m);
}

// Block-wide exclusive prefix of the pair tiles of each expert
// (ceil(m_g / 256) row tiles x n_tiles column tiles); prefix has E + 1
// entries.  Returns the total.
__device__ int build_masked_prefix(const int32_t* __restrict__ counts, int E, int max_m,
                                   int n_tiles, int* prefix, int* scratch) {
  const int nthr = blockDim.x, tid = threadIdx.x;
  const int per = (E + nthr - 1) / nthr;
  const int lo = tid * per, hi = min(E, lo + per);
  int local = 0;
  for (int e = lo; e < hi; ++e)
    local += ((valid_rows(counts, e, max_m) + 2 * BM - 1) / (2 * BM)) * n_tiles;
  const int lane = tid & 31, wid = tid >> 5, nw = (nthr + 31) >> 5;
  int v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) scratch[wid] = v;
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int w = 0; w < nw; ++w) {
      const int x = scratch[w];
      scratch[w] = acc;
      acc += x;
    }
    scratch[32] = acc;
  }
  __syncthreads();
  int run = scratch[wid] + v - local;
  for (int e = lo; e < hi; ++e) {
    prefix[e] = run;
    run += ((valid_rows(counts, e, max_m) + 2 * BM - 1) / (2 * BM)) * n_tiles;
  }
  if (tid == 0) prefix[E] = scratch[32];
  __syncthreads();
  return scratch[32];
}

struct MaskedTile {
  int g;      // expert
  int m0;     // first row of the pair tile inside the expert's slab
  int m_end;  // valid rows of the expert
  int n_idx;  // column tile (256 columns)
};

// Tile t -> (expert, row tile, column tile); inside an expert the row tiles
// of a column tile are consecutive.
__device__ __forceinline__ MaskedTile decode_masked(int t, const int* prefix,
                                                    const int32_t* __restrict__ counts, int E,
                                                    int max_m) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  MaskedTile r;
  r.g = lo;
  r.m_end = valid_rows(counts, lo, max_m);
  const int mt = (r.m_end + 2 * BM - 1) / (2 * BM);
  const int local = t - prefix[lo];
  r.n_idx = local / mt;
  r.m0 = (local % mt) * (2 * BM);
  return r;
}

__global__ void __launch_bounds__(NUM_THREADS)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b, const float* __restrict__ a_scale,
                    const float* __restrict__ b_scale, const int32_t* __restrict__ counts, int E,
                    int max_m, int N, int K, const __grid_constant__ CUtensorMap tm_out,
                    int tma_out, __nv_bfloat16* __restrict__ out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* out_stage = smem + (size_t)STAGES * STAGE_BYTES;
  Fp8Shared* sh = reinterpret_cast<Fp8Shared*>(out_stage + OUT_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  volatile int* abort_flag = &sh->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh->full[s], 1);  // the leader's expect-tx arrival (+ both CTAs' bytes)
      mbar_init(&sh->empty[s], 1);
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(&sh->pfull[p], 1);
      mbar_init(&sh->pempty[p], 2 * kEpiWarps);  // one arrival per promotion warp of the pair
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(&sh->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  const int n_tiles = (N + BN - 1) / BN;
  const int nkb = K / BKB;
  const int nsb = N / 128;  // column blocks of b_scale
  pdl_wait();  // the operands, scales and counts are read only after this
  const int total = build_masked_prefix(counts, E, max_m, n_tiles, sh->prefix, sh->scan_tmp);
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp >= kEpiWarp0) {
    // ------------------------------------------------ promotion + epilogue
    const int quad = warp & 3;                  // TMEM lanes (tile rows) 32*quad ..
    const int half = (warp - kEpiWarp0) >> 2;   // partial-sum columns 128*half ..
    uint8_t* obufs = out_stage + (warp - kEpiWarp0) * OUT_BUF_BYTES;
    int obuf = 0, pb = 0;
    uint32_t pph = 0;
    bool ok = true;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const uint32_t pempty_leader0 = map_to_rank(su32(&sh->pempty[0]), 0);
    const uint32_t pempty_leader1 = map_to_rank(su32(&sh->pempty[1]), 0);
    for (int tile = pair; tile < total && ok; tile += npairs) {
      const MaskedTile st = decode_masked(tile, sh->prefix, counts, E, max_m);
      const int row = st.m0 + BM * (int)rank + quad * 32 + lane;  // row inside the slab
      const bool in_slab = row < max_m;
      const int nb = st.n_idx * 2 + half;  // b_scale column block of this warp's columns
      const bool col_ok = nb < nsb;        // warp-uniform
      const float* sa = a_scale + ((size_t)st.g * max_m + (in_slab ? row : 0)) * nkb;
      const float* sb = b_scale + ((size_t)st.g * nsb + (col_ok ? nb : 0)) * nkb;
      // column pairs, added with the packed two-wide fp32 FMA (each half
      // rounds as its own fmaf does)
      float2 acc[kColsPerWarp / 2];
#pragma unroll
      for (int i = 0; i < kColsPerWarp / 2; ++i) acc[i] = make_float2(0.f, 0.f);
      // scales two K blocks ahead of their use
      float sa0 = in_slab ? __ldg(sa) : 0.f, sb0 = col_ok ? __ldg(sb) : 0.f;
      float sa1 = 0.f, sb1 = 0.f;
      if (nkb > 1) {
        sa1 = in_slab ? __ldg(sa + 1) : 0.f;
        sb1 = col_ok ? __ldg(sb + 1) : 0.f;
      }
#pragma unroll 1
      for (int kb = 0; kb < nkb; ++kb) {
        const float s = sa0 * sb0;
        const float2 s2 = make_float2(s, s);
        sa0 = sa1;
        sb0 = sb1;
        if (kb + 2 < nkb) {
          sa1 = in_slab ? __ldg(sa + kb + 2) : 0.f;
          sb1 = col_ok ? __ldg(sb + kb + 2) : 0.f;
        }
        if (!wait_fast(&sh->pfull[pb], pph, abort_flag, status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t taddr =
            tmem_base + lane_addr + (uint32_t)(pb * BN + half * kColsPerWarp);
        // 16-column chunks, the load of chunk c + 1 in flight while chunk c
        // is added; the buffer is released once the last chunk has landed
        uint32_t p[2][16];
        tmem_ld16(taddr, p[0]);
#pragma unroll
        for (int c = 0; c < kColsPerWarp / 16; ++c) {
          tmem_wait_ld_regs16(p[c & 1]);
          if (c + 1 < kColsPerWarp / 16) {
            tmem_ld16(taddr + (uint32_t)(16 * (c + 1)), p[(c + 1) & 1]);
          } else {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(pb ? pempty_leader1 : pempty_leader0);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i)
            acc[8 * c + i] = __ffma2_rn(make_float2(__uint_as_float(p[c & 1][2 * i]),
                                                    __uint_as_float(p[c & 1][2 * i + 1])),
                                        s2, acc[8 * c + i]);
        }
        if (++pb == 2) { pb = 0; pph ^= 1u; }
      }
      if (!ok || !col_ok) continue;
      // rows of the flattened [E * max_m, N] output; rows at or past the
      // expert's count are not written
      const int wrow0 = st.g * max_m + st.m0 + BM * (int)rank + quad * 32;
      const int m_end = st.g * max_m + st.m_end;
      const bool boxed = tma_out && m_end - wrow0 >= OUT_BOX;
      const bool row_ok = wrow0 + lane < m_end;
      __nv_bfloat16* orow = out + (row_ok ? (size_t)(wrow0 + lane) * N : 0);
#pragma unroll
      for (int c = 0; c < kColsPerWarp / 32; ++c) {
        const int col0 = nb * 128 + c * 32;
        float v[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          v[2 * i] = acc[c * 16 + i].x;
          v[2 * i + 1] = acc[c * 16 + i].y;
        }
        emit_chunk32<1>(v, col0, wrow0, boxed, row_ok, orow, N - col0, &tm_out, obufs, obuf,
                        lane);
      }
    }
    if (lane == 0) bulk_wait_all();  // every staged box written before the block exits
  } else {
    if (warp == 0) {
      if (lane == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued[STAGES];
        for (int s = 0; s < STAGES; ++s) issued[s] = 0;
        bool ok = true;
        for (int tile = pair; tile < total && ok; tile += npairs) {
          const MaskedTile st = decode_masked(tile, sh->prefix, counts, E, max_m);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_fast(&sh->empty[stage], phase ^ 1u, abort_flag, status)) { ok = false; break; }
            uint8_t* a_dst = smem + (size_t)stage * STAGE_BYTES;
            const uint32_t bar = map_to_rank(su32(&sh->full[stage]), 0);
            if (leader) mbar_expect_tx(&sh->full[stage], 2 * STAGE_BYTES);
            // rows past max_m or N read as zeros (and count in full)
            tma2_3d(a_dst, &tm_a, bar, kb * BKB, st.m0 + BM * (int)rank, st.g);
            tma2_3d(a_dst + A_BYTES, &tm_b, bar, kb * BKB, st.n_idx * BN + (BN / 2) * (int)rank,
                    st.g);
            ++issued[stage];
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
        if (!ok && leader) {  // both CTAs' copies complete on the leader's barriers
          for (int s = 0; s < STAGES; ++s)
            if (issued[s]) drain_wait(&sh->full[s], (issued[s] - 1u) & 1u);
        }
      }
    } else if (warp == 1) {
      if (lane == 0 && leader) {
        // ------------------------------------------------ MMA issuer (leader)
        int stage = 0, pb = 0;
        uint32_t phase = 0, pph = 0;
        bool ok = true, any = false;
        const uint64_t adesc0 = sw128_desc(su32(smem));
        const uint64_t bdesc0 = sw128_desc(su32(smem + A_BYTES));
        for (int tile = pair; tile < total && ok; tile += npairs) {
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_fast(&sh->pempty[pb], pph ^ 1u, abort_flag, status)) { ok = false; break; }
            if (!wait_fast(&sh->full[stage], phase, abort_flag, status)) { ok = false; break; }
            tc_fence_after();
            const uint64_t off = (uint64_t)((stage * STAGE_BYTES) >> 4);
            umma2_fp8_block(tmem_base + (uint32_t)(pb * BN), adesc0 + off, bdesc0 + off,
                            su32(&sh->empty[stage]), su32(&sh->pfull[pb]));
            any = true;
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            if (++pb == 2) { pb = 0; pph ^= 1u; }
          }
        }
        if (!ok && any) {  // every MMA issued so far done before TMEM is freed
          umma2_commit_self(&sh->drain);
          drain_wait(&sh->drain, 0);
        }
      }
    }
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

cudaError_t launch_gemm_fp8(const void* a, const float* a_scale, const void* b,
                            const float* b_scale, const int32_t* counts, int E, int max_m, int N,
                            int K, void* out, int* status, cudaStream_t s) {
  if (E == 0 || max_m == 0) return cudaSuccess;
  CUtensorMap ma, mb, mo;
  {
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)max_m, (cuuint64_t)E};
    cuuint64_t str[2] = {(cuuint64_t)K, (cuuint64_t)max_m * K};
    cuuint32_t box[3] = {BKB, BM, 1};
    if (!tmap::encode_u8(&ma, a, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)N, (cuuint64_t)E};
    cuuint64_t str[2] = {(cuuint64_t)K, (cuuint64_t)N * K};
    cuuint32_t box[3] = {BKB, BN / 2, 1};
    if (!tmap::encode_u8(&mb, b, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  int tma_out = 0;
  if ((reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)E * max_m};
    cuuint64_t str[1] = {(cuuint64_t)N * 2};
    cuuint32_t box[2] = {OUT_BOX, OUT_BOX};
    tma_out = tmap::encode_bf16(&mo, out, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B) ? 1 : 0;
  }
  if (!tma_out) mo = mb;  // unused
  set_smem_limit((const void*)gemm_fp8_kernel, (int)kSmemBytes);
  const long long max_tiles =
      (long long)E * ((max_m + 2 * BM - 1) / (2 * BM)) * ((N + BN - 1) / BN);
  const int pairs = (int)std::max<long long>(1, std::min<long long>(max_tiles, num_sms() / 2));

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(NUM_THREADS);
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
  __nv_bfloat16* out_p = static_cast<__nv_bfloat16*>(out);
  void* args[] = {&ma, &mb, &a_scale, &b_scale, &counts, &E, &max_m, &N, &K, &mo, &tma_out,
                  &out_p, &status};
  cudaError_t e = cudaLaunchKernelExC(&cfg, (const void*)gemm_fp8_kernel, args);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
