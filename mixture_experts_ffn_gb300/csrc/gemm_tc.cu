// Persistent tcgen05 grouped GEMM for bf16 operands with fp32 accumulators in
// tensor memory, fed by TMA, over the expert-segmented row layout
// ("contiguous · physical_psum") of TileOPs "MoE Operators",
// MoEGroupedGemmFwdOp: out[rows of e] = a[rows of e] @ b[e]^T, with the gated
// activation (silu_and_mul over stacked rows, clamped SwiGLU over interleaved
// or concatenated rows) and the optional bias fused into the epilogue, so the
// [M, 2F] product never leaves the SM.
//
// Work decomposition
//   tile = 128 rows x 256 accumulator columns; k-block = 64 (one 128-byte
//   swizzle atom of bf16); 4-stage shared-memory ring of A (16 KB) + B (32 KB).
//   Gated modes use the 256 accumulator columns as 128 gate + 128 up columns
//   (stacked: one 4-D box of gate rows j0.. then up rows F+j0..; interleaved:
//   256 consecutive rows 2*j0..), giving 128 activation columns per tile.
//   With the gate and up projections in two tensors (SwiGLU fusion 0), two
//   3-D boxes of 128 rows each land in the same shared-memory layout.
// Roles (192 threads, one CTA per SM)
//   warp 0 lane 0 : TMA producer
//   warp 1        : TMEM allocator; lane 0 issues tcgen05.mma (M128 N256 K16)
//   warps 2..5    : epilogue; warp w reads TMEM lanes 32*(w%4).., one row per
//                   thread, applies bias + activation, rounds to bf16 and
//                   writes 32x32 boxes through swizzled shared memory and TMA
//                   stores (gemm_epilogue.cuh)
//   Two 256-column accumulators (all 512 TMEM columns) let the epilogue of one
//   tile overlap the main loop of the next.
// What bounds it: shared-memory traffic per SM.  Each 64-wide k-block writes
// 48 KB into shared memory (A 16 KB + B 32 KB) and the four M128 N256 K16 MMAs
// read the same 48 KB back; at 128 bytes per cycle that is >= 750 cycles per
// k-block against 512 cycles of MMA, and the measured ~950 cycles put shared
// memory about 79% busy.  Timed apart, the MMAs alone and the loads alone each
// run faster than the whole kernel, and deeper rings do not help.
// Every mbarrier wait is bounded: a wait that runs out sets MOE's timeout bit
// in the status word, raises a block-wide abort flag, and the block drains its
// in-flight copies and MMAs (again bounded) before freeing TMEM and returning.
#include <cuda.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "gemm_epilogue.cuh"
#include "tmap.h"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int NUM_THREADS = 192;
// With the row gather (A rows read from the token-ordered hidden states through
// the permutation, so the permuted copy of the activations is never written),
// four more warps load A with cp.async: TMA copies only whole boxes of a
// tensor, not rows picked by an index.
constexpr int NUM_THREADS_GATHER = NUM_THREADS + 128;
constexpr int kLoaderWarp0 = NUM_THREADS / 32;

struct TcShared {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int prefix[kMaxExperts + 1];
  int scan_tmp[33];
};
constexpr size_t kSmemBytes =
    (size_t)STAGES * STAGE_BYTES + OUT_BYTES + sizeof(TcShared) + 1024;


constexpr uint32_t kIdesc = idesc_bf16(BM, BN);
constexpr uint32_t kIdescF16 = idesc_f16(BM, BN);

// The four K16 MMAs of one 64-wide k-block and the commit that frees its stage,
// in one block: descriptors advance by 32 bytes (2 in 16-byte units) per K16.
__device__ __forceinline__ void umma_kblock(uint32_t d_tmem, uint64_t ad, uint64_t bd,
                                            uint32_t idesc, uint32_t accumulate, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %7, %3, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %9, %3, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %10, %11, %3, t;\n\t"
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t}" ::"r"(
          d_tmem),
      "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate), "r"(bar), "l"(ad + 2), "l"(bd + 2),
      "l"(ad + 4), "l"(bd + 4), "l"(ad + 6), "l"(bd + 6)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          su32(bar))
      : "memory");
}


// GATHER: row r of A is row grows[r] / gdiv of gsrc (the hidden states, gsrc_rows
// rows; grows is row_to_route, gdiv = top_k); tm_a is unused.
template <int MODE, int ACT, bool GATHER>
__global__ void __launch_bounds__(GATHER ? NUM_THREADS_GATHER : NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __nv_bfloat16* __restrict__ bias, const int32_t* __restrict__ seg_end,
                   int M, int Nout, int N1, int K, int E, float limit, float alpha, float beta,
                   const __grid_constant__ CUtensorMap tm_out, int tma_out,
                   __nv_bfloat16* __restrict__ out, int* status,
                   const __nv_bfloat16* __restrict__ gsrc, const int32_t* __restrict__ grows,
                   int gdiv, int gsrc_rows, int seg_stride,
                   const __grid_constant__ CUtensorMap tm_b_up, int split,
                   const __nv_bfloat16* __restrict__ bias_up, int f16) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* out_stage = smem + (size_t)STAGES * STAGE_BYTES;  // 1024-byte aligned
  TcShared* sh = reinterpret_cast<TcShared*>(out_stage + OUT_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &sh->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // the producer's expect-tx arrival, plus one per A-loader thread
      mbar_init(&sh->full[s], GATHER ? 1 + 128 : 1);
      mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->tfull[a], 1);
      mbar_init(&sh->tempty[a], 128);
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b)) : "memory");
    if (split)
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b_up))
                   : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(&sh->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  const int n_tiles = MODE == kTcPlain ? (Nout + BN - 1) / BN : (Nout + BN / 2 - 1) / (BN / 2);
  // barrier init, tensor-map prefetch and TMEM allocation above overlap the
  // previous launch; seg_end and the operands are read only after this
  pdl_wait();
  const int total = build_tile_prefix(seg_end, E, M, BM, n_tiles, sh->prefix, sh->scan_tmp, seg_stride);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  const int nkb = (K + BK - 1) / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = 0;
      bool ok = true;
      int tile = blockIdx.x;
      SegTile st{}, nx{};
      if (tile < total) st = decode_tile(tile, sh->prefix, seg_end, E, M, BM, n_tiles, seg_stride);
      for (; tile < total && ok; tile += gridDim.x) {
        if (tile + (int)gridDim.x < total)
          nx = decode_tile(tile + gridDim.x, sh->prefix, seg_end, E, M, BM, n_tiles, seg_stride);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_fast(&sh->empty[stage], phase ^ 1u, abort_flag, status)) { ok = false; break; }
          uint8_t* a_dst = smem + (size_t)stage * STAGE_BYTES;
          uint8_t* b_dst = a_dst + A_BYTES;
          const int k0 = kb * BK;
          if constexpr (GATHER) {
            mbar_expect_tx(&sh->full[stage], B_BYTES);  // A comes from the loader warps
          } else {
            mbar_expect_tx(&sh->full[stage], STAGE_BYTES);
            tma_2d(a_dst, &tm_a, &sh->full[stage], k0, st.m0);
          }
          if constexpr (MODE == kTcStacked) {  // gate rows j0.. then up rows F+j0..
            if (split) {
              tma_3d(b_dst, &tm_b, &sh->full[stage], k0, st.n_idx * (BN / 2), st.e);
              tma_3d(b_dst + B_BYTES / 2, &tm_b_up, &sh->full[stage], k0, st.n_idx * (BN / 2),
                     st.e);
            } else {
              tma_4d(b_dst, &tm_b, &sh->full[stage], k0, st.n_idx * (BN / 2), 0, st.e);
            }
          } else {
            tma_3d(b_dst, &tm_b, &sh->full[stage], k0, st.n_idx * BN, st.e);
          }
          ++issued[stage];
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        st = nx;
      }
      if (!ok) {  // let every copy already in flight land before the block exits
        for (int s = 0; s < STAGES; ++s)
          if (issued[s]) drain_wait(&sh->full[s], (issued[s] - 1u) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      bool ok = true, any = false;
      // descriptors of stage 0; stage s adds s * STAGE_BYTES to the address field
      const uint64_t adesc0 = sw128_desc(su32(smem));
      const uint64_t bdesc0 = sw128_desc(su32(smem + A_BYTES));
      const uint32_t idesc = f16 ? kIdescF16 : kIdesc;  // A and B of one type
      uint32_t empty_addr[STAGES];
      for (int s = 0; s < STAGES; ++s) empty_addr[s] = su32(&sh->empty[s]);
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        if (!wait_fast(&sh->tempty[acc], aphase ^ 1u, abort_flag, status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_fast(&sh->full[stage], phase, abort_flag, status)) { ok = false; break; }
          // cp.async wrote A through the generic proxy; tcgen05.mma reads it
          // through the async proxy
          if constexpr (GATHER) fence_proxy_async_smem();
          tc_fence_after();
          const uint64_t off = (uint64_t)((stage * STAGE_BYTES) >> 4);
          umma_kblock(d_tmem, adesc0 + off, bdesc0 + off, idesc, kb != 0 ? 1u : 0u,
                      empty_addr[stage]);
          any = true;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&sh->tfull[acc]);  // accumulator ready for the epilogue
        if (++acc == 2) { acc = 0; aphase ^= 1u; }
      }
      if (!ok && any) {  // wait for every MMA issued so far before TMEM is freed
        umma_commit(&sh->drain);
        drain_wait(&sh->drain, 0);
      }
    }
  } else if (GATHER && warp >= kLoaderWarp0) {
    // ------------------------------------------------ A loaders (gather mode)
    // 128 threads copy the 128 rows x 128 bytes of a k-block: thread lt owns
    // 16-byte chunk lt % 8 of rows lt / 8 + 16 i (i < 8), so 8 neighbouring
    // lanes read one 128-byte row piece; the destination follows the 128-byte
    // swizzle of the TMA boxes (chunk ch of row r at chunk ch ^ (r % 8)).
    const int lt = threadIdx.x - kLoaderWarp0 * 32;
    const int ch = lt & 7, r0 = lt >> 3;
    const uint32_t dst0 = (uint32_t)(r0 * 128 + ((ch ^ (r0 & 7)) << 4));
    // The hidden rows are read again by every column tile of their experts:
    // kept in L2 ahead of the weight stream that passes through it
    // (DeepSeek-V3-style gate_up 3339 vs 3363 us, Qwen3-style 196.6 vs 202.8
    // us; marking the weights evict-first as well was slower on the former).
    uint64_t keep_policy;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep_policy));
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    // The row map entries of a tile are loaded one tile ahead, so their
    // latency never delays the first copies of the next tile.
    auto load_map = [&](int tile, int (&r)[8]) {
      const SegTile t = decode_tile(tile, sh->prefix, seg_end, E, M, BM, n_tiles, seg_stride);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        // Only rows of the tile's own expert segment are read: the map holds
        // defined entries for rows below seg_end[E-1] only (routes with an
        // out-of-range id get no row); padding rows are zero-filled.
        const int row = t.m0 + r0 + 16 * i;
        r[i] = row < t.m_end ? grows[row] : -1;
      }
    };
    int cur[8], nxt[8];
    if (blockIdx.x < total) load_map(blockIdx.x, cur);
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      if (tile + (int)gridDim.x < total) load_map(tile + gridDim.x, nxt);
      const __nv_bfloat16* src[8];
      uint32_t valid = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        int t = 0;
        if (cur[i] >= 0 && cur[i] / gdiv < gsrc_rows) {
          t = cur[i] / gdiv;
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
        for (int i = 0; i < 8; ++i) {
          const bool v = kin && ((valid >> i) & 1u);
          asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(
                           a_dst + i * 16 * 128),
                       "l"(v ? src[i] + k0 : gsrc), "r"(v ? 16 : 0), "l"(keep_policy)
                       : "memory");
        }
        // arrives on the stage's full barrier once this thread's copies land
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                         su32(&sh->full[stage]))
                     : "memory");
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // nothing in flight at exit
  } else {
    // ------------------------------------------------ epilogue (warps 2..5)
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    int acc = 0;
    uint32_t aphase = 0;
    uint8_t* obufs = out_stage + quad * 2 * OUT_BUF_BYTES;
    int obuf = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const SegTile st = decode_tile(tile, sh->prefix, seg_end, E, M, BM, n_tiles, seg_stride);
      if (!wait_fast(&sh->tfull[acc], aphase, abort_flag, status)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN);
      if (f16)
        drain_acc<MODE, ACT, true>(tb, st.m0 + quad * 32, st.m_end, st.n_idx, st.e, bias, bias_up,
                                   N1, Nout, limit, alpha, beta, &tm_out, tma_out, out, obufs,
                                   obuf, lane);
      else
        drain_acc<MODE, ACT, false>(tb, st.m0 + quad * 32, st.m_end, st.n_idx, st.e, bias,
                                    bias_up, N1, Nout, limit, alpha, beta, &tm_out, tma_out, out,
                                    obufs, obuf, lane);
      tc_fence_before();
      mbar_arrive(&sh->tempty[acc]);
      if (++acc == 2) { acc = 0; aphase ^= 1u; }
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

// ------------------------------------------------------------ host side
}  // namespace

cudaError_t launch_gemm_tc(const void* a, const void* w, const void* bias, const int32_t* seg_end,
                           int M, int N, int K, int E, const moe_act_params* act, void* out,
                           int* status, cudaStream_t s, const int32_t* gather_rows,
                           int gather_div, int gather_src_rows, int seg_stride,
                           const SplitUp* split, bool f16) {
  if (M == 0 || N == 0) return cudaSuccess;
  // The weights-as-M kernel on SM pairs (gemm_sw.cu) pads an expert's rows to
  // 16 instead of 128.  Its wide form (256 weight rows per CTA, two M256
  // accumulators) is the default for products with long K and segments
  // averaging >= 128 rows, gathered or not, plain or gated: measured on the
  // DeepSeek-V3-style GEMMs 2.87 vs 3.32 ms (gathered gate_up) and 1.61 vs
  // 1.75 ms (down), on the Qwen3-style gate_up 195 vs 197 us; with short K
  // (Qwen3-style down, 136 vs 111 us) or 64-row segments (gpt-oss-style, 674
  // vs 640 us) this kernel is faster.
  // MOE_TC_KERNEL=1sm keeps every call on this kernel, =sw sends every call
  // the pair kernel can take to its 128-row form, =wide to its wide form
  // (the settings exist to check the kernels against each other).
  static const int which = [] {
    const char* v = getenv("MOE_TC_KERNEL");
    return v && v[0] == '1' ? 1 : v && v[0] == 's' ? 2 : v && v[0] == 'w' ? 3 : 0;
  }();
  const bool gather = gather_rows != nullptr;
  const bool sw_ok = !split && num_sms() >= 2 && N % 8 == 0 && K % 8 == 0;
  const bool wide_pick = which == 0 && K >= 2048 && (long long)M >= 128LL * E;
  if (sw_ok && (which >= 2 || wide_pick))
    return launch_gemm_sw(a, w, bias, seg_end, M, N, K, E, act, out, status, s, gather_rows,
                          gather_div, gather_src_rows, seg_stride, f16, which != 2);
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
  // split weights: w is the gate projection [E, N, K], split->w_up the up
  // projection, both read by 128-row boxes (only with a stacked gated mode)
  if (split && mode != kTcStacked) return cudaErrorInvalidValue;
  if (split) N1 = N;
  CUtensorMap ma, mb, mb_up;
  if (!gather) {  // (gathered rows of A are loaded without a tensor map)
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t str[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {BK, BM};
    if (!tmap::encode_bf16(&ma, a, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B, f16))
      return cudaErrorInvalidValue;
  }
  if (split) {
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)N, (cuuint64_t)E};
    cuuint64_t str[2] = {(cuuint64_t)K * 2, (cuuint64_t)N * K * 2};
    cuuint32_t box[3] = {BK, BN / 2, 1};
    if (!tmap::encode_bf16(&mb, w, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B, f16) ||
        !tmap::encode_bf16(&mb_up, split->w_up, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B,
                           f16))
      return cudaErrorInvalidValue;
  } else if (mode == kTcStacked) {
    cuuint64_t dims[4] = {(cuuint64_t)K, (cuuint64_t)N, 2, (cuuint64_t)E};
    cuuint64_t str[3] = {(cuuint64_t)K * 2, (cuuint64_t)N * K * 2, (cuuint64_t)2 * N * K * 2};
    cuuint32_t box[4] = {BK, BN / 2, 2, 1};  // 128 gate rows then 128 up rows
    if (!tmap::encode_bf16(&mb, w, 4, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B, f16))
      return cudaErrorInvalidValue;
  } else {
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)N1, (cuuint64_t)E};
    cuuint64_t str[2] = {(cuuint64_t)K * 2, (cuuint64_t)N1 * K * 2};
    cuuint32_t box[3] = {BK, BN, 1};
    if (!tmap::encode_bf16(&mb, w, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B, f16))
      return cudaErrorInvalidValue;
  }
  if (gather) ma = mb;  // unused by the kernel
  if (!split) mb_up = mb;  // unused
  {
    for (const void* fn : {(const void*)gemm_tc_kernel<kTcPlain, MOE_ACT_IDENTITY, false>,
                           (const void*)gemm_tc_kernel<kTcPlain, MOE_ACT_RELU, false>,
                           (const void*)gemm_tc_kernel<kTcPlain, MOE_ACT_GELU, false>,
                           (const void*)gemm_tc_kernel<kTcPlain, MOE_ACT_SILU, false>,
                           (const void*)gemm_tc_kernel<kTcStacked, MOE_ACT_GELU_AND_MUL, false>,
                           (const void*)gemm_tc_kernel<kTcStacked, MOE_ACT_SILU_AND_MUL, false>,
                           (const void*)gemm_tc_kernel<kTcStacked, MOE_ACT_SWIGLU, false>,
                           (const void*)gemm_tc_kernel<kTcInterleaved, MOE_ACT_SWIGLU, false>,
                           (const void*)gemm_tc_kernel<kTcPlain, MOE_ACT_IDENTITY, true>,
                           (const void*)gemm_tc_kernel<kTcPlain, MOE_ACT_RELU, true>,
                           (const void*)gemm_tc_kernel<kTcPlain, MOE_ACT_GELU, true>,
                           (const void*)gemm_tc_kernel<kTcPlain, MOE_ACT_SILU, true>,
                           (const void*)gemm_tc_kernel<kTcStacked, MOE_ACT_GELU_AND_MUL, true>,
                           (const void*)gemm_tc_kernel<kTcStacked, MOE_ACT_SILU_AND_MUL, true>,
                           (const void*)gemm_tc_kernel<kTcStacked, MOE_ACT_SWIGLU, true>,
                           (const void*)gemm_tc_kernel<kTcInterleaved, MOE_ACT_SWIGLU, true>})
      set_smem_limit(fn, (int)kSmemBytes);
  }
  const int n_tiles = mode == kTcPlain ? (N + BN - 1) / BN : (N + BN / 2 - 1) / (BN / 2);
  const long long max_tiles = (long long)((M + BM - 1) / BM + E) * n_tiles;
  const int grid = (int)std::max<long long>(1, std::min<long long>(max_tiles, num_sms()));
  // Output map for the staged stores: rows of Nout bf16, 32 x 32 boxes.  TMA
  // needs a 16-byte aligned base and row pitch; otherwise rows are stored
  // directly from registers.
  CUtensorMap mo;
  int tma_out = 0;
  if (N % 8 == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t str[1] = {(cuuint64_t)N * 2};
    cuuint32_t box[2] = {OUT_BOX, OUT_BOX};
    tma_out = tmap::encode_bf16(&mo, out, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B, f16) ? 1 : 0;
  }
  if (!tma_out) mo = mb;  // unused
  const auto* bias_p = static_cast<const __nv_bfloat16*>(bias);
  auto* out_p = static_cast<__nv_bfloat16*>(out);
  auto pick = [&](auto g) {
    constexpr bool G = decltype(g)::value;
    return mode == kTcPlain ? (kind == MOE_ACT_RELU   ? gemm_tc_kernel<kTcPlain, MOE_ACT_RELU, G>
                               : kind == MOE_ACT_GELU ? gemm_tc_kernel<kTcPlain, MOE_ACT_GELU, G>
                               : kind == MOE_ACT_SILU ? gemm_tc_kernel<kTcPlain, MOE_ACT_SILU, G>
                                                      : gemm_tc_kernel<kTcPlain, MOE_ACT_IDENTITY, G>)
           : mode == kTcInterleaved ? gemm_tc_kernel<kTcInterleaved, MOE_ACT_SWIGLU, G>
           : kind == MOE_ACT_SWIGLU ? gemm_tc_kernel<kTcStacked, MOE_ACT_SWIGLU, G>
           : kind == MOE_ACT_GELU_AND_MUL ? gemm_tc_kernel<kTcStacked, MOE_ACT_GELU_AND_MUL, G>
                                    : gemm_tc_kernel<kTcStacked, MOE_ACT_SILU_AND_MUL, G>;
  };
  auto* kern = gather ? pick(std::true_type{}) : pick(std::false_type{});
  launch_pdl(kern, grid, gather ? NUM_THREADS_GATHER : NUM_THREADS, kSmemBytes, s, ma, mb,
             bias_p, seg_end, M, N, N1, K, E, limit, alpha, beta, mo, tma_out, out_p, status,
             static_cast<const __nv_bfloat16*>(a), gather_rows, gather_div, gather_src_rows,
             seg_stride, mb_up, split ? 1 : 0,
             split ? static_cast<const __nv_bfloat16*>(split->b_up) : nullptr, f16 ? 1 : 0);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
