// Two-SM variant of the tcgen05 grouped GEMM (same contract as gemm_tc.cu and
// the same epilogue, gemm_epilogue.cuh; TileOPs "MoE Operators",
// MoEGroupedGemmFwdOp).
//
// A cluster of two CTAs on a pair of SMs computes a 256-row x 256-column tile
// with tcgen05.mma.cta_group::2 (M256 N256 K16): each CTA loads its own 128
// rows of A and HALF of the 256 B rows (stacked gated layouts: the leader
// loads the 128 gate rows, the peer the 128 up rows; otherwise the lower and
// upper 128 rows), so an SM ingests 32 KB per 64-wide k-block instead of the
// 48 KB of the one-SM 128x256 tile -- a third fewer bytes per MMA, and the
// one-SM kernel is bound by its per-SM load stream.  The price is the 256-row
// pair tile: on ragged expert segments the padded rows cost MMA time and
// loads, which on routed workloads cancels the gain.
//
// Roles (192 threads in each CTA of the pair):
//   warp 0 lane 0 (both CTAs): TMA producer for its own A rows and B half; the
//     copies of both CTAs complete on the LEADER's full barrier (expect-tx of
//     the whole 64 KB by the leader).
//   warp 1 (both CTAs): TMEM allocation (cta_group::2); in the leader, lane 0
//     issues the MMAs and multicasts its commits to both CTAs' empty / tfull
//     barriers.
//   warps 2..5 (both CTAs): epilogue of the CTA's 128 rows from its own TMEM;
//     each thread arrives on the leader's tempty barrier (256 arrivals).
// Every wait is bounded (2 s) as in gemm_tc.cu; on a timeout the leader drains
// the copies and MMAs in flight before the pair frees TMEM.
#include <cuda.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "gemm_epilogue.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moe {
namespace {

using namespace tc;

constexpr int BMP = 256;                        // rows per CTA pair
constexpr int BMC = 128;                        // rows per CTA
constexpr int BMS = 64;                         // rows per CTA of a short (128-row) pair tile
constexpr int BN = 256;                         // accumulator columns
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int A_BYTES = BMC * BK * 2;           // 16 KB
constexpr int BH_BYTES = (BN / 2) * BK * 2;     // 16 KB: this CTA's half of B
constexpr int STAGE_BYTES = A_BYTES + BH_BYTES; // 32 KB
constexpr int TMEM_COLS = 512;
constexpr int NUM_THREADS = 192;
// Gathered-row mode: four more warps per CTA copy the CTA's A rows from the
// token-ordered hidden states through the permutation with cp.async (as in
// the one-SM kernel).  Their completions can only arrive on a barrier of
// their own CTA, so in the peer they arrive on afull and warp 1 of the peer
// (idle otherwise) forwards each completed stage to the leader's full barrier.
constexpr int NUM_THREADS_GATHER = NUM_THREADS + 128;
constexpr int kLoaderWarp0 = NUM_THREADS / 32;
constexpr uint32_t kIdesc2 = idesc_bf16(BMP, BN);
constexpr uint32_t kIdesc2s = idesc_bf16(2 * BMS, BN);

struct Tc2Shared {
  uint64_t full[STAGES];   // leader: both CTAs' copies of a stage complete here
  uint64_t afull[STAGES];  // peer, gathered rows: the peer's A copies of a stage
  uint64_t empty[STAGES];  // both: the leader's MMA commit frees the stage
  uint64_t tfull[2];       // both: accumulator ready
  uint64_t tempty[2];      // leader: both epilogues have drained the accumulator
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int prefix[kMaxExperts + 1];
  int scan_tmp[33];
};
// The 16 KB output staging area follows the ring directly, so it also keeps
// every operand read of a stage inside this CTA's shared memory, whatever the
// MMA reads past its half-tile (the MMA never writes shared memory).
static_assert(OUT_BYTES >= 16 * 1024, "staging doubles as the guard after the ring");
constexpr size_t kSmemBytes =
    (size_t)STAGES * STAGE_BYTES + OUT_BYTES + sizeof(Tc2Shared) + 1024;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared variable in CTA `rank` of the cluster
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
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote_cta(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}
// TMA load into this CTA's shared memory, completing on a barrier of either
// CTA of the pair (shared::cluster address)
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
// the four K16 MMAs of a k-block plus the commit that frees the stage in both CTAs
__device__ __forceinline__ void umma2_kblock(uint32_t d_tmem, uint64_t ad, uint64_t bd,
                                             uint32_t idesc, uint32_t accumulate, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %6, %7, %3, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %8, %9, %3, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %10, %11, %3, t;\n\t"
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%5], %12;\n\t}" ::"r"(d_tmem),
      "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate), "r"(bar), "l"(ad + 2), "l"(bd + 2),
      "l"(ad + 4), "l"(bd + 4), "l"(ad + 6), "l"(bd + 6), "h"((uint16_t)3)
      : "memory");
}
// arrive (once) on the barrier at this offset in both CTAs when the MMAs issued
// so far have completed
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

// GATHER: row r of A is row grows[r] / gdiv of gsrc (the hidden states, gsrc_rows
// rows; grows is row_to_route, gdiv = top_k); tm_a and tm_a_s are unused.
template <int MODE, int ACT, bool GATHER>
__global__ void __launch_bounds__(GATHER ? NUM_THREADS_GATHER : NUM_THREADS, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_a_s,
                    const __grid_constant__ CUtensorMap tm_b_s,
                    const __nv_bfloat16* __restrict__ bias, const int32_t* __restrict__ seg_end,
                    int M, int Nout, int N1, int K, int E, float limit, float alpha, float beta,
                    const __grid_constant__ CUtensorMap tm_out, int tma_out,
                    __nv_bfloat16* __restrict__ out, int* status,
                    const __nv_bfloat16* __restrict__ gsrc, const int32_t* __restrict__ grows,
                    int gdiv, int gsrc_rows, int seg_stride) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* out_stage = smem + (size_t)STAGES * STAGE_BYTES;  // 1024-byte aligned
  Tc2Shared* sh = reinterpret_cast<Tc2Shared*>(out_stage + OUT_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  volatile int* abort_flag = &sh->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // the leader's expect-tx arrival; gathered rows: plus one per leader
      // A-loader thread and the peer's forwarded arrival
      mbar_init(&sh->full[s], GATHER ? 1 + 128 + 1 : 1);
      mbar_init(&sh->afull[s], 128);
      mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->tfull[a], 1);
      mbar_init(&sh->tempty[a], 2 * 128);
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_a_s)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b_s)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(&sh->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  const int n_tiles = MODE == kTcPlain ? (Nout + BN - 1) / BN : (Nout + BN / 2 - 1) / (BN / 2);
  // barrier init, tensor-map prefetch and TMEM allocation above overlap the
  // previous launch; seg_end and the operands are read only after this
  pdl_wait();
  const int total = build_tile_prefix(seg_end, E, M, BMP, n_tiles, sh->prefix, sh->scan_tmp, seg_stride);
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  const int nkb = (K + BK - 1) / BK;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = 0;
      bool ok = true;
      for (int tile = pair; tile < total && ok; tile += npairs) {
        const SegTile st = decode_tile(tile, sh->prefix, seg_end, E, M, BMP, n_tiles, seg_stride);
        const bool tall = st.m_end - st.m0 > BMC;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_fast(&sh->empty[stage], phase ^ 1u, abort_flag, status)) { ok = false; break; }
          uint8_t* a_dst = smem + (size_t)stage * STAGE_BYTES;
          uint8_t* b_dst = a_dst + A_BYTES;
          if (leader) {  // A comes from the loader warps in gather mode
            const int a_bytes = GATHER ? 0 : tall ? A_BYTES : A_BYTES / 2;
            mbar_expect_tx(&sh->full[stage], 2 * (a_bytes + BH_BYTES));
          }
          const uint32_t bar = map_to_rank(su32(&sh->full[stage]), 0);
          const int k0 = kb * BK;
          if (tall) {
            if constexpr (!GATHER) tma2_2d(a_dst, &tm_a, bar, k0, st.m0 + BMC * (int)rank);
            if constexpr (MODE == kTcStacked)
              tma2_4d(b_dst, &tm_b, bar, k0, st.n_idx * (BN / 2), (int)rank, st.e);
          } else {
            // short tile: 64 rows per CTA; a stacked B half holds the gate
            // and the up rows of this CTA's 64 activation columns
            if constexpr (!GATHER) tma2_2d(a_dst, &tm_a_s, bar, k0, st.m0 + BMS * (int)rank);
            if constexpr (MODE == kTcStacked)
              tma2_4d(b_dst, &tm_b_s, bar, k0, st.n_idx * (BN / 2) + BMS * (int)rank, 0, st.e);
          }
          if constexpr (MODE != kTcStacked)
            tma2_3d(b_dst, &tm_b, bar, k0, st.n_idx * BN + (BN / 2) * (int)rank, st.e);
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
      int stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      bool ok = true, any = false;
      const uint64_t adesc0 = sw128_desc(su32(smem));
      const uint64_t bdesc0 = sw128_desc(su32(smem + A_BYTES));
      uint32_t empty_addr[STAGES];
      for (int s = 0; s < STAGES; ++s) empty_addr[s] = su32(&sh->empty[s]);
      for (int tile = pair; tile < total && ok; tile += npairs) {
        const SegTile st = decode_tile(tile, sh->prefix, seg_end, E, M, BMP, n_tiles, seg_stride);
        const uint32_t idesc = st.m_end - st.m0 > BMC ? kIdesc2 : kIdesc2s;
        if (!wait_fast(&sh->tempty[acc], aphase ^ 1u, abort_flag, status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_fast(&sh->full[stage], phase, abort_flag, status)) { ok = false; break; }
          // the leader's A rows were written by cp.async through the generic
          // proxy; tcgen05.mma reads them through the async proxy (the peer's
          // forwarder fences its own CTA's rows)
          if constexpr (GATHER) fence_proxy_async_smem();
          tc_fence_after();
          const uint64_t off = (uint64_t)((stage * STAGE_BYTES) >> 4);
          umma2_kblock(d_tmem, adesc0 + off, bdesc0 + off, idesc, kb != 0 ? 1u : 0u,
                       empty_addr[stage]);
          any = true;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma2_commit_both(&sh->tfull[acc]);
        if (++acc == 2) { acc = 0; aphase ^= 1u; }
      }
      if (!ok && any) {
        umma2_commit_self(&sh->drain);
        drain_wait(&sh->drain, 0);
      }
    }
    if constexpr (GATHER) {
      if (lane == 0 && !leader) {
        // ---------------------------------------------- forwarder (peer)
        int stage = 0;
        uint32_t phase = 0;
        const uint32_t full_remote0 = map_to_rank(su32(&sh->full[0]), 0);
        bool ok = true;
        for (int tile = pair; tile < total && ok; tile += npairs) {
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_fast(&sh->afull[stage], phase, abort_flag, status)) { ok = false; break; }
            // This CTA's A rows are read by this CTA's own tensor core when the
            // leader's MMAs run: order them for the async proxy here, and
            // release at CTA scope only (a cluster-scope release waits for the
            // SM's copies in flight and serialises the ring).
            fence_proxy_async_smem();
            mbar_arrive_remote_cta(full_remote0 + (uint32_t)(stage * sizeof(uint64_t)));
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
      }
    }
  } else if (GATHER && warp >= kLoaderWarp0) {
    // ------------------------------------------------ A loaders (gather mode)
    // 128 threads copy this CTA's 128 (64 in a short tile) rows x 128 bytes
    // of a k-block: thread lt owns 16-byte chunk lt % 8 of rows lt / 8 + 16 i,
    // in the 128-byte swizzle of the TMA boxes (chunk ch of row r at chunk
    // ch ^ (r % 8)); rows outside the tile's segment are zero-filled.
    const int lt = threadIdx.x - kLoaderWarp0 * 32;
    const int ch = lt & 7, r0 = lt >> 3;
    const uint32_t dst0 = (uint32_t)(r0 * 128 + ((ch ^ (r0 & 7)) << 4));
    uint64_t* arrive_bar = leader ? sh->full : sh->afull;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    constexpr int kRows = BMC / 16;  // rows per loader thread in a 256-row pair tile
    for (int tile = pair; tile < total && ok; tile += npairs) {
      const SegTile st = decode_tile(tile, sh->prefix, seg_end, E, M, BMP, n_tiles, seg_stride);
      const bool tall = st.m_end - st.m0 > BMC;
      const int rbase = st.m0 + (tall ? BMC : BMS) * (int)rank;
      const int nrows = tall ? kRows : kRows / 2;
      const __nv_bfloat16* src[kRows];
      uint32_t valid = 0;
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        // only rows of the tile's own segment are read (the map holds defined
        // entries below seg_end[E-1] only)
        const int row = rbase + r0 + 16 * i;
        const int rt = i < nrows && row < st.m_end ? grows[row] : -1;
        int t = 0;
        if (rt >= 0 && rt / gdiv < gsrc_rows) {
          t = rt / gdiv;
          valid |= 1u << i;
        }
        src[i] = gsrc + (size_t)t * K + ch * 8;
      }
      for (int kb = 0; kb < nkb; ++kb) {
        if (!wait_fast(&sh->empty[stage], phase ^ 1u, abort_flag, status)) { ok = false; break; }
        const uint32_t a_dst = su32(smem + (size_t)stage * STAGE_BYTES) + dst0;
        const int k0 = kb * BK;
        const bool kin = k0 + ch * 8 < K;
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
          if (i >= nrows) break;
          const bool v = kin && ((valid >> i) & 1u);
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(a_dst + i * 16 * 128),
                       "l"(v ? src[i] + k0 : gsrc), "r"(v ? 16 : 0)
                       : "memory");
        }
        // arrives on this CTA's stage barrier once this thread's copies land
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
    int acc = 0;
    uint32_t aphase = 0;
    const uint32_t tempty_remote[2] = {map_to_rank(su32(&sh->tempty[0]), 0),
                                       map_to_rank(su32(&sh->tempty[1]), 0)};
    uint8_t* obufs = out_stage + quad * 2 * OUT_BUF_BYTES;
    int obuf = 0;
    for (int tile = pair; tile < total; tile += npairs) {
      const SegTile st = decode_tile(tile, sh->prefix, seg_end, E, M, BMP, n_tiles, seg_stride);
      if (!wait_fast(&sh->tfull[acc], aphase, abort_flag, status)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN);
      if (st.m_end - st.m0 > BMC) {
        drain_acc<MODE, ACT>(tbase, st.m0 + BMC * (int)rank + quad * 32, st.m_end, st.n_idx,
                             st.e, bias, nullptr, N1, Nout, limit, alpha, beta, &tm_out, tma_out, out,
                             obufs, obuf, lane);
      } else {
        // short tile (M128 over the pair): TMEM lane 64h + r holds row
        // 64 * rank + r with accumulator columns 128h.. in columns 0..127
        const int wrow0 = st.m0 + BMS * (int)rank + 32 * (quad & 1);
        const int h = quad >> 1;
        if (wrow0 < st.m_end) {  // warp-uniform
          if constexpr (MODE == kTcPlain)
            drain_cols<MODE, ACT>(tbase, wrow0, st.m_end, st.n_idx * BN + (BN / 2) * h,
                                  BN / 2 / 32, 0, st.e, bias, nullptr, N1, Nout, limit, alpha, beta,
                                  &tm_out, tma_out, out, obufs, obuf, lane);
          else
            drain_cols<MODE, ACT>(tbase, wrow0, st.m_end, st.n_idx * (BN / 2) + BMS * h,
                                  BMS / 32, BMS, st.e, bias, nullptr, N1, Nout, limit, alpha, beta,
                                  &tm_out, tma_out, out, obufs, obuf, lane);
        }
      }
      tc_fence_before();
      mbar_arrive_remote(tempty_remote[acc]);
      if (++acc == 2) { acc = 0; aphase ^= 1u; }
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

cudaError_t launch_gemm_tc2(const void* a, const void* w, const void* bias,
                            const int32_t* seg_end, int M, int N, int K, int E,
                            const moe_act_params* act, void* out, int* status, cudaStream_t s,
                            const int32_t* gather_rows, int gather_div, int gather_src_rows,
                            int seg_stride) {
  if (M == 0 || N == 0) return cudaSuccess;
  int mode = kTcPlain, kind = MOE_ACT_IDENTITY, N1 = N;
  float limit = 0.f, alpha = 1.f, beta = 0.f;
  if (act) kind = act->kind;
  if (act && act_is_gated(act->kind)) {
    mode = (kind == MOE_ACT_SWIGLU && act->swiglu_fusion == 1) ? kTcInterleaved : kTcStacked;
    N1 = 2 * N;
    limit = act->limit;
    alpha = act->alpha;
    beta = act->beta;
  }
  // ma / mb: 128 A rows and one 128-row half of B per CTA (256-row pair
  // tiles); ma_s / mb_s: 64 A rows, and for stacked weights 64 gate rows then
  // the 64 matching up rows (128-row pair tiles)
  const bool gather = gather_rows != nullptr;
  CUtensorMap ma, mb, ma_s, mb_s;
  if (!gather) {  // (gathered rows of A are loaded without a tensor map)
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t str[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {BK, BMC};
    if (!tmap::encode_bf16(&ma, a, 2, dims, str, box)) return cudaErrorInvalidValue;
    cuuint32_t box_s[2] = {BK, BMS};
    if (!tmap::encode_bf16(&ma_s, a, 2, dims, str, box_s)) return cudaErrorInvalidValue;
  }
  if (mode == kTcStacked) {
    cuuint64_t dims[4] = {(cuuint64_t)K, (cuuint64_t)N, 2, (cuuint64_t)E};
    cuuint64_t str[3] = {(cuuint64_t)K * 2, (cuuint64_t)N * K * 2, (cuuint64_t)2 * N * K * 2};
    cuuint32_t box[4] = {BK, BN / 2, 1, 1};
    if (!tmap::encode_bf16(&mb, w, 4, dims, str, box)) return cudaErrorInvalidValue;
    cuuint32_t box_s[4] = {BK, BMS, 2, 1};
    if (!tmap::encode_bf16(&mb_s, w, 4, dims, str, box_s)) return cudaErrorInvalidValue;
  } else {
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)N1, (cuuint64_t)E};
    cuuint64_t str[2] = {(cuuint64_t)K * 2, (cuuint64_t)N1 * K * 2};
    cuuint32_t box[3] = {BK, BN / 2, 1};
    if (!tmap::encode_bf16(&mb, w, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  if (mode != kTcStacked) mb_s = mb;  // unused
  if (gather) ma = ma_s = mb;           // unused
  {
    for (const void* fn : {(const void*)gemm_tc2_kernel<kTcPlain, MOE_ACT_IDENTITY, false>,
                           (const void*)gemm_tc2_kernel<kTcPlain, MOE_ACT_RELU, false>,
                           (const void*)gemm_tc2_kernel<kTcPlain, MOE_ACT_GELU, false>,
                           (const void*)gemm_tc2_kernel<kTcPlain, MOE_ACT_SILU, false>,
                           (const void*)gemm_tc2_kernel<kTcStacked, MOE_ACT_GELU_AND_MUL, false>,
                           (const void*)gemm_tc2_kernel<kTcStacked, MOE_ACT_SILU_AND_MUL, false>,
                           (const void*)gemm_tc2_kernel<kTcStacked, MOE_ACT_SWIGLU, false>,
                           (const void*)gemm_tc2_kernel<kTcInterleaved, MOE_ACT_SWIGLU, false>,
                           (const void*)gemm_tc2_kernel<kTcPlain, MOE_ACT_IDENTITY, true>,
                           (const void*)gemm_tc2_kernel<kTcPlain, MOE_ACT_RELU, true>,
                           (const void*)gemm_tc2_kernel<kTcPlain, MOE_ACT_GELU, true>,
                           (const void*)gemm_tc2_kernel<kTcPlain, MOE_ACT_SILU, true>,
                           (const void*)gemm_tc2_kernel<kTcStacked, MOE_ACT_GELU_AND_MUL, true>,
                           (const void*)gemm_tc2_kernel<kTcStacked, MOE_ACT_SILU_AND_MUL, true>,
                           (const void*)gemm_tc2_kernel<kTcStacked, MOE_ACT_SWIGLU, true>,
                           (const void*)gemm_tc2_kernel<kTcInterleaved, MOE_ACT_SWIGLU, true>})
      set_smem_limit(fn, (int)kSmemBytes);
  }
  // output map for the staged TMA stores (rows stored directly when the
  // output's base or pitch is not 16-byte aligned)
  CUtensorMap mo;
  int tma_out = 0;
  if (N % 8 == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t str[1] = {(cuuint64_t)N * 2};
    cuuint32_t box[2] = {OUT_BOX, OUT_BOX};
    tma_out = tmap::encode_bf16(&mo, out, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B) ? 1 : 0;
  }
  if (!tma_out) mo = mb;  // unused
  const int n_tiles = mode == kTcPlain ? (N + BN - 1) / BN : (N + BN / 2 - 1) / (BN / 2);
  const long long max_tiles = (long long)((M + BMP - 1) / BMP + E) * n_tiles;
  const int pairs = (int)std::max<long long>(1, std::min<long long>(max_tiles, num_sms() / 2));

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(gather ? NUM_THREADS_GATHER : NUM_THREADS);
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
  auto pick = [&](auto g) {
    constexpr bool G = decltype(g)::value;
    return mode == kTcPlain ? (kind == MOE_ACT_RELU   ? gemm_tc2_kernel<kTcPlain, MOE_ACT_RELU, G>
                               : kind == MOE_ACT_GELU ? gemm_tc2_kernel<kTcPlain, MOE_ACT_GELU, G>
                               : kind == MOE_ACT_SILU ? gemm_tc2_kernel<kTcPlain, MOE_ACT_SILU, G>
                                                      : gemm_tc2_kernel<kTcPlain, MOE_ACT_IDENTITY, G>)
           : mode == kTcInterleaved ? gemm_tc2_kernel<kTcInterleaved, MOE_ACT_SWIGLU, G>
           : kind == MOE_ACT_SWIGLU ? gemm_tc2_kernel<kTcStacked, MOE_ACT_SWIGLU, G>
           : kind == MOE_ACT_GELU_AND_MUL ? gemm_tc2_kernel<kTcStacked, MOE_ACT_GELU_AND_MUL, G>
                                    : gemm_tc2_kernel<kTcStacked, MOE_ACT_SILU_AND_MUL, G>;
  };
  auto* kern = gather ? pick(std::true_type{}) : pick(std::false_type{});
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, ma_s, mb_s,
                                     static_cast<const __nv_bfloat16*>(bias),
                                     seg_end, M, N, N1, K, E, limit, alpha, beta, mo, tma_out,
                                     static_cast<__nv_bfloat16*>(out), status,
                                     static_cast<const __nv_bfloat16*>(a), gather_rows,
                                     gather_div, gather_src_rows, seg_stride);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
