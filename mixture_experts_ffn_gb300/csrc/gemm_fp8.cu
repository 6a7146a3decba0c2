// Block-scaled FP8 grouped GEMM over a masked slab (TileOPs "MoE Operators",
// MoEGroupedGemmFP8FwdOp): out[g, :m_g] = a[g, :m_g] @ b[g]^T with a [E, max_m, K]
// and b [E, N, K] in float8_e4m3fn, one fp32 scale per row and 128 K-columns of
// a (a_scale [E, max_m, K/128]) and one per 128 x 128 block of b
// (b_scale [E, N/128, K/128]); m_g = layout_metadata[g] read as
// min(max(m_g, 0), max_m).  Each 128-wide K block is contracted from the raw
// FP8 values, then multiplied by its two scales and added to an fp32
// accumulator; the result is written in bf16.
//
// Work decomposition
//   tile = 128 rows x 128 columns of one expert (so one b scale per tile and
//   K block); K block = 128 e4m3 values = one 128-byte swizzle row; 6-stage
//   shared-memory ring of A (16 KB) + B (16 KB).
//   Per K block the MMA warp writes a fresh partial sum with four
//   tcgen05.mma.kind::f8f6f4 M128 N128 K32 into one of two 128-column TMEM
//   buffers; the epilogue warps read it, scale it by a_scale[row, kb] *
//   b_scale[n-block, kb] and add it into a register accumulator ("promotion"),
//   then free the buffer, so the MMAs of the next block run meanwhile.
// Roles (320 threads, one CTA per SM)
//   warp 0 lane 0 : TMA producer
//   warp 1        : TMEM allocator; lane 0 issues the MMAs
//   warps 2..9    : promotion and epilogue; warp w owns TMEM lanes 32*(w%4)..
//                   (tile rows) and accumulator columns 64*((w-2)/4).. (64
//                   fp32 registers of accumulator per thread), and writes its
//                   rows as bf16 through staged 32 x 32 TMA stores
// Every mbarrier wait is bounded (as in gemm_tc.cu): a wait that runs out sets
// the timeout bit, raises the block's abort flag, and the block drains its
// copies and MMAs in flight before freeing TMEM.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "gemm_epilogue.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128, BN = 128, BKB = 128;  // tile rows, tile columns, K per block
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BKB;  // 16 KB of e4m3
constexpr int B_BYTES = BN * BKB;  // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;  // two partial-sum buffers
constexpr int kEpiWarps = 8;
constexpr int NUM_THREADS = 64 + 32 * kEpiWarps;
constexpr int kColsPerWarp = BN / 2;  // accumulator columns of one epilogue warp
// kind::f8f6f4 instruction descriptor: fp32 D (bit 4), e4m3 A and B (format
// 0 in bits 7..9 and 10..12), N / 8 at bit 17, M / 16 at bit 24
constexpr uint32_t kIdescFp8 =
    (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

struct Fp8Shared {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t pfull[2];   // partial sum of a K block ready (MMA commit)
  uint64_t pempty[2];  // partial sum read by every epilogue thread
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int prefix[kMaxExperts + 1];
  int scan_tmp[33];
};
constexpr size_t kSmemBytes = (size_t)STAGES * STAGE_BYTES + OUT_BYTES + sizeof(Fp8Shared) + 1024;

__device__ __forceinline__ int valid_rows(const int32_t* __restrict__ counts, int g, int max_m) {
  return min(max(counts[g], 0), max_m);
}

// Block-wide exclusive prefix of the tiles of each expert (ceil(m_g / BM) row
// tiles x n_tiles column tiles); prefix has E + 1 entries.  Returns the total.
__device__ int build_masked_prefix(const int32_t* __restrict__ counts, int E, int max_m,
                                   int n_tiles, int* prefix, int* scratch) {
  const int nthr = blockDim.x, tid = threadIdx.x;
  const int per = (E + nthr - 1) / nthr;
  const int lo = tid * per, hi = min(E, lo + per);
  int local = 0;
  for (int e = lo; e < hi; ++e) local += ((valid_rows(counts, e, max_m) + BM - 1) / BM) * n_tiles;
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
    run += ((valid_rows(counts, e, max_m) + BM - 1) / BM) * n_tiles;
  }
  if (tid == 0) prefix[E] = scratch[32];
  __syncthreads();
  return scratch[32];
}

struct MaskedTile {
  int g;      // expert
  int m0;     // first row of the tile inside the expert's slab
  int m_end;  // valid rows of the expert
  int n_idx;  // column tile
};

// Tile t -> (expert, row tile, column tile); inside an expert the column tiles
// are the outer loop, so concurrent CTAs share each weight tile through L2.
__device__ __forceinline__ MaskedTile decode_masked(int t, const int* prefix,
                                                    const int32_t* __restrict__ counts, int E,
                                                    int max_m, int n_tiles) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  MaskedTile r;
  r.g = lo;
  r.m_end = valid_rows(counts, lo, max_m);
  const int mt = (r.m_end + BM - 1) / BM;
  const int local = t - prefix[lo];
  r.n_idx = local / mt;
  r.m0 = (local % mt) * BM;
  return r;
}

// The four K32 MMAs of one 128-wide K block into a fresh partial sum.
__device__ __forceinline__ void umma_fp8_block(uint32_t d_tmem, uint64_t ad, uint64_t bd) {
  asm volatile(
      "{\n\t.reg .pred f, t;\n\t"
      "setp.ne.b32 f, %3, %3;\n\t"
      "setp.eq.b32 t, %3, %3;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, f;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %4, %5, %3, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %6, %7, %3, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %8, %9, %3, t;\n\t}" ::"r"(d_tmem),
      "l"(ad), "l"(bd), "r"(kIdescFp8), "l"(ad + 2), "l"(bd + 2), "l"(ad + 4), "l"(bd + 4),
      "l"(ad + 6), "l"(bd + 6)
      : "memory");
}
__device__ __forceinline__ void commit_to(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          su32(bar))
      : "memory");
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
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
  volatile int* abort_flag = &sh->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], 1);
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(&sh->pfull[p], 1);
      mbar_init(&sh->pempty[p], kEpiWarps * 32);
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
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(&sh->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  const int n_tiles = N / BN;
  const int nkb = K / BKB;
  pdl_wait();  // the operands, scales and counts are read only after this
  const int total = build_masked_prefix(counts, E, max_m, n_tiles, sh->prefix, sh->scan_tmp);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const MaskedTile st = decode_masked(tile, sh->prefix, counts, E, max_m, n_tiles);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_fast(&sh->empty[stage], phase ^ 1u, abort_flag, status)) { ok = false; break; }
          uint8_t* a_dst = smem + (size_t)stage * STAGE_BYTES;
          mbar_expect_tx(&sh->full[stage], STAGE_BYTES);
          tma_3d(a_dst, &tm_a, &sh->full[stage], kb * BKB, st.m0, st.g);
          tma_3d(a_dst + A_BYTES, &tm_b, &sh->full[stage], kb * BKB, st.n_idx * BN, st.g);
          ++issued[stage];
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        for (int s = 0; s < STAGES; ++s)
          if (issued[s]) drain_wait(&sh->full[s], (issued[s] - 1u) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0, pb = 0;
      uint32_t phase = 0, pph = 0;
      bool ok = true, any = false;
      const uint64_t adesc0 = sw128_desc(su32(smem));
      const uint64_t bdesc0 = sw128_desc(su32(smem + A_BYTES));
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_fast(&sh->pempty[pb], pph ^ 1u, abort_flag, status)) { ok = false; break; }
          if (!wait_fast(&sh->full[stage], phase, abort_flag, status)) { ok = false; break; }
          tc_fence_after();
          const uint64_t off = (uint64_t)((stage * STAGE_BYTES) >> 4);
          umma_fp8_block(tmem_base + (uint32_t)(pb * BN), adesc0 + off, bdesc0 + off);
          commit_to(&sh->empty[stage]);  // the stage is free once these MMAs finish
          commit_to(&sh->pfull[pb]);     // and the partial sum is ready
          any = true;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          if (++pb == 2) { pb = 0; pph ^= 1u; }
        }
      }
      if (!ok && any) {  // every MMA issued so far done before TMEM is freed
        commit_to(&sh->drain);
        drain_wait(&sh->drain, 0);
      }
    }
  } else {
    // ------------------------------------------------ promotion + epilogue
    const int quad = warp & 3;                // TMEM lanes (tile rows) 32*quad ..
    const int half = (warp - 2) >> 2;         // accumulator columns 64*half ..
    uint8_t* obufs = out_stage + (warp - 2) * OUT_BUF_BYTES;
    int obuf = 0, pb = 0;
    uint32_t pph = 0;
    bool ok = true;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const MaskedTile st = decode_masked(tile, sh->prefix, counts, E, max_m, n_tiles);
      const int row = st.m0 + quad * 32 + lane;  // row inside the expert's slab
      const bool in_slab = row < max_m;
      const float* sa = a_scale + ((size_t)st.g * max_m + (in_slab ? row : 0)) * nkb;
      const float* sb = b_scale + ((size_t)st.g * n_tiles + st.n_idx) * nkb;
      float acc[kColsPerWarp];
#pragma unroll
      for (int i = 0; i < kColsPerWarp; ++i) acc[i] = 0.f;
      float sa_next = in_slab ? __ldg(sa) : 0.f, sb_next = __ldg(sb);
      for (int kb = 0; kb < nkb; ++kb) {
        const float s = sa_next * sb_next;
        if (kb + 1 < nkb) {
          sa_next = in_slab ? __ldg(sa + kb + 1) : 0.f;
          sb_next = __ldg(sb + kb + 1);
        }
        if (!wait_fast(&sh->pfull[pb], pph, abort_flag, status)) { ok = false; break; }
        tc_fence_after();
        uint32_t p0[32], p1[32];
        const uint32_t taddr = tmem_base + lane_addr + (uint32_t)(pb * BN + half * kColsPerWarp);
        tmem_ld32(taddr, p0);
        tmem_ld32(taddr + 32, p1);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&sh->pempty[pb]);  // the MMAs may refill this buffer now
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          acc[i] = fmaf(__uint_as_float(p0[i]), s, acc[i]);
          acc[32 + i] = fmaf(__uint_as_float(p1[i]), s, acc[32 + i]);
        }
        if (++pb == 2) { pb = 0; pph ^= 1u; }
      }
      if (!ok) break;
      // rows of the flattened [E * max_m, N] output; rows at or past the
      // expert's count are not written
      const int wrow0 = st.g * max_m + st.m0 + quad * 32;
      const int m_end = st.g * max_m + st.m_end;
      const bool boxed = tma_out && m_end - wrow0 >= OUT_BOX;
      const bool row_ok = wrow0 + lane < m_end;
      __nv_bfloat16* orow = out + (size_t)(wrow0 + lane) * N;
#pragma unroll
      for (int c = 0; c < kColsPerWarp / 32; ++c) {
        const int col0 = st.n_idx * BN + half * kColsPerWarp + c * 32;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = acc[c * 32 + i];
        emit_chunk32<1>(v, col0, wrow0, boxed, row_ok, orow, N - col0, &tm_out, obufs, obuf,
                        lane);
      }
    }
    if (lane == 0) bulk_wait_all();  // every staged box written before the block exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
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
    cuuint32_t box[3] = {BKB, BN, 1};
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
  const long long max_tiles = (long long)E * ((max_m + BM - 1) / BM) * (N / BN);
  const int grid = (int)std::max<long long>(1, std::min<long long>(max_tiles, num_sms()));
  launch_pdl(gemm_fp8_kernel, grid, NUM_THREADS, kSmemBytes, s, ma, mb, a_scale, b_scale, counts,
             E, max_m, N, K, mo, tma_out, static_cast<__nv_bfloat16*>(out), status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
