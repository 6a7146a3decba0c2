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
//   (stacked: two TMA boxes, gate rows j0.. and up rows F+j0..; interleaved:
//   256 consecutive rows 2*j0..), giving 128 activation columns per tile.
// Roles (192 threads, one CTA per SM)
//   warp 0 lane 0 : TMA producer
//   warp 1        : TMEM allocator; lane 0 issues tcgen05.mma (M128 N256 K16)
//   warps 2..5    : epilogue; warp w reads TMEM lanes 32*(w%4).., one row per
//                   thread, applies bias + activation and stores bf16
//   Two 256-column accumulators (all 512 TMEM columns) let the epilogue of one
//   tile overlap the main loop of the next.
// Every mbarrier wait is bounded: a wait that runs out sets MOE's timeout bit
// in the status word, raises a block-wide abort flag, and the block drains its
// in-flight copies and MMAs (again bounded) before freeing TMEM and returning.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int NUM_THREADS = 192;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

enum TcMode { kTcPlain = 0, kTcStacked = 1, kTcInterleaved = 2 };

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
constexpr size_t kSmemBytes = (size_t)STAGES * STAGE_BYTES + sizeof(TcShared) + 1024;

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of parity `parity`; false on abort or timeout.
__device__ __noinline__ bool wait_bar(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                      int* status) {
  const uint32_t addr = su32(b);
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(addr, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kTimeoutNs) {
      *abort_flag = 1;
      latch_error(status, kDevTimeout);
      return false;
    }
  }
}
// Bounded wait used while draining after an abort (ignores the abort flag).
__device__ __noinline__ void drain_wait(uint64_t* b, uint32_t parity) {
  const uint32_t addr = su32(b);
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(addr, parity)) {
    if (global_ns() - t0 > kTimeoutNs) return;
  }
}

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0,
                                       int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(su32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0,
                                       int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(su32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_4d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0,
                                       int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(su32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row core groups 1024 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                    // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset
  d |= (uint64_t)1 << 46;                    // descriptor version
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: D f32, A/B bf16, both K-major, M x N.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t ad, uint64_t bd, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(ad), "l"(bd), "r"(kIdesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          su32(bar))
      : "memory");
}

#define MOE_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                  "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : MOE_R8(0), MOE_R8(8), MOE_R8(16), MOE_R8(24)
      : "r"(taddr));
}
#undef MOE_R8
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// store 32 bf16 values (64 bytes) of one row; vector path when all columns valid
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const float (&v)[32], int n_valid) {
  if (n_valid >= 32) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 u;
      u.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
      u.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
      u.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
      u.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
      d4[q] = u;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < n_valid) dst[i] = __float2bfloat16_rn(v[i]);
  }
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __nv_bfloat16* __restrict__ bias, const int32_t* __restrict__ seg_end,
                   int M, int Nout, int N1, int K, int E, int mode, int act_kind, float limit,
                   float alpha, float beta, __nv_bfloat16* __restrict__ out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  TcShared* sh = reinterpret_cast<TcShared*>(smem + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &sh->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh->full[s], 1);
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
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(&sh->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  const int n_tiles = mode == kTcPlain ? (Nout + BN - 1) / BN : (Nout + BN / 2 - 1) / (BN / 2);
  const int total = build_tile_prefix(seg_end, E, M, BM, n_tiles, sh->prefix, sh->scan_tmp);
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
      uint32_t issued[STAGES] = {0, 0, 0, 0};
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const SegTile st = decode_tile(tile, sh->prefix, seg_end, E, M, BM, n_tiles);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bar(&sh->empty[stage], phase ^ 1u, abort_flag, status)) { ok = false; break; }
          uint8_t* a_dst = smem + (size_t)stage * STAGE_BYTES;
          uint8_t* b_dst = a_dst + A_BYTES;
          mbar_expect_tx(&sh->full[stage], STAGE_BYTES);
          const int k0 = kb * BK;
          tma_2d(a_dst, &tm_a, &sh->full[stage], k0, st.m0);
          if (mode == kTcStacked) {
            const int j0 = st.n_idx * (BN / 2);
            tma_4d(b_dst, &tm_b, &sh->full[stage], k0, j0, 0, st.e);
            tma_4d(b_dst + B_BYTES / 2, &tm_b, &sh->full[stage], k0, j0, 1, st.e);
          } else {
            tma_3d(b_dst, &tm_b, &sh->full[stage], k0, st.n_idx * BN, st.e);
          }
          ++issued[stage];
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
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
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        if (!wait_bar(&sh->tempty[acc], aphase ^ 1u, abort_flag, status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bar(&sh->full[stage], phase, abort_flag, status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = su32(smem + (size_t)stage * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            umma(d_tmem, sw128_desc(a_addr + k * 32), sw128_desc(b_addr + k * 32),
                 (kb | k) != 0 ? 1u : 0u);
          }
          any = true;
          umma_commit(&sh->empty[stage]);  // frees the slot once these MMAs retire
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
  } else {
    // ------------------------------------------------ epilogue (warps 2..5)
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    int acc = 0;
    uint32_t aphase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const SegTile st = decode_tile(tile, sh->prefix, seg_end, E, M, BM, n_tiles);
      if (!wait_bar(&sh->tfull[acc], aphase, abort_flag, status)) break;
      tc_fence_after();
      const int row = st.m0 + quad * 32 + lane;
      const bool row_ok = row < st.m_end;
      const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN);
      const __nv_bfloat16* be = bias ? bias + (size_t)st.e * N1 : nullptr;
      __nv_bfloat16* orow = out + (size_t)row * Nout;
      if (mode == kTcPlain) {
        const int n0 = st.n_idx * BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int col0 = n0 + c * 32;
          if (col0 >= Nout) break;  // warp-uniform
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          tmem_wait_ld();
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float b = (be && col0 + i < Nout) ? __bfloat162float(be[col0 + i]) : 0.f;
            v[i] = __uint_as_float(r[i]) + b;
          }
          if (row_ok) store_row32(orow + col0, v, Nout - col0);
        }
      } else {
        const int j0 = st.n_idx * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          const int col0 = j0 + c * 32;  // activation column
          if (col0 >= Nout) break;
          uint32_t g[32], u[32];
          if (mode == kTcStacked) {
            tmem_ld32(tbase + c * 32, g);             // gate columns
            tmem_ld32(tbase + BN / 2 + c * 32, u);    // up columns
          } else {
            tmem_ld32(tbase + c * 64, g);             // (gate, up) pairs
            tmem_ld32(tbase + c * 64 + 32, u);
          }
          tmem_wait_ld();
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float gv, uv;
            int rg, ru;
            if (mode == kTcStacked) {
              gv = __uint_as_float(g[i]);
              uv = __uint_as_float(u[i]);
              rg = col0 + i;
              ru = Nout + col0 + i;
            } else {
              // pair i lives in columns 2i, 2i+1 of the 64 loaded
              const int p = 2 * i;
              gv = __uint_as_float(p < 32 ? g[p] : u[p - 32]);
              uv = __uint_as_float(p + 1 < 32 ? g[p + 1] : u[p + 1 - 32]);
              rg = 2 * (col0 + i);
              ru = rg + 1;
            }
            if (be && col0 + i < Nout) {
              gv += __bfloat162float(be[rg]);
              uv += __bfloat162float(be[ru]);
            }
            v[i] = act_kind == MOE_ACT_SILU_AND_MUL ? silu_mul(gv, uv)
                                                    : swiglu_f(gv, uv, limit, alpha, beta);
          }
          if (row_ok) store_row32(orow + col0, v, Nout - col0);
        }
      }
      tc_fence_before();
      mbar_arrive(&sh->tempty[acc]);
      if (++acc == 2) { acc = 0; aphase ^= 1u; }
    }
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
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

bool encode(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeFn fn = get_encode();
  if (!fn) return false;
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(ptr),
                  dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm_tc(const void* a, const void* w, const void* bias, const int32_t* seg_end,
                           int M, int N, int K, int E, const moe_act_params* act, void* out,
                           int* status, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  int mode = kTcPlain, kind = MOE_ACT_IDENTITY, N1 = N;
  float limit = 0.f, alpha = 1.f, beta = 0.f;
  if (act && act->kind != MOE_ACT_IDENTITY) {
    kind = act->kind;
    mode = (kind == MOE_ACT_SWIGLU && act->swiglu_fusion == 1) ? kTcInterleaved : kTcStacked;
    N1 = 2 * N;
    limit = act->limit;
    alpha = act->alpha;
    beta = act->beta;
  }
  CUtensorMap ma, mb;
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t str[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {BK, BM};
    if (!encode(&ma, a, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  if (mode == kTcStacked) {
    cuuint64_t dims[4] = {(cuuint64_t)K, (cuuint64_t)N, 2, (cuuint64_t)E};
    cuuint64_t str[3] = {(cuuint64_t)K * 2, (cuuint64_t)N * K * 2, (cuuint64_t)2 * N * K * 2};
    cuuint32_t box[4] = {BK, BN / 2, 1, 1};
    if (!encode(&mb, w, 4, dims, str, box)) return cudaErrorInvalidValue;
  } else {
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)N1, (cuuint64_t)E};
    cuuint64_t str[2] = {(cuuint64_t)K * 2, (cuuint64_t)N1 * K * 2};
    cuuint32_t box[3] = {BK, BN, 1};
    if (!encode(&mb, w, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  static std::once_flag attr_once;
  std::call_once(attr_once, [] {
    cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)kSmemBytes);
  });
  const int n_tiles = mode == kTcPlain ? (N + BN - 1) / BN : (N + BN / 2 - 1) / (BN / 2);
  const long long max_tiles = (long long)((M + BM - 1) / BM + E) * n_tiles;
  const int grid = (int)std::max<long long>(1, std::min<long long>(max_tiles, num_sms()));
  gemm_tc_kernel<<<grid, NUM_THREADS, kSmemBytes, s>>>(
      ma, mb, static_cast<const __nv_bfloat16*>(bias), seg_end, M, N, N1, K, E, mode, kind, limit,
      alpha, beta, static_cast<__nv_bfloat16*>(out), status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
