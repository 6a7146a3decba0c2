// Epilogue shared by the tcgen05 grouped-GEMM kernels: the accumulator layout
// modes, the gated activations, and the drain of one 128-lane x 256-column
// accumulator to bf16 output rows through swizzled shared-memory staging and
// TMA stores.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

// How the accumulator columns of a tile map to output columns: plain GEMM
// columns; gate rows j0.. then up rows F+j0.. (stacked halves); or (gate, up)
// pairs in consecutive columns (interleaved rows of the weight).
enum TcMode { kTcPlain = 0, kTcStacked = 1, kTcInterleaved = 2 };

constexpr int kEpiCols = 256;  // accumulator columns of one tile

// Output staging: each epilogue warp owns two 2 KB buffers (32 rows x 32 bf16
// columns, 64-byte swizzle) that it fills from registers and hands to a TMA
// store, so the output leaves the SM as whole boxes instead of 32 scattered
// row segments per store instruction (those flood the L1/shared-memory data
// path that tcgen05.mma reads its operands through).
constexpr int OUT_BOX = 32;                        // rows and columns of one staged box
constexpr int OUT_BUF_BYTES = OUT_BOX * OUT_BOX * 2;  // 2 KB
constexpr int OUT_BYTES = 8 * OUT_BUF_BYTES;          // 4 warps x 2 buffers, or 8 x 1

// Epilogue activation math.  The exponential and the quotient use the fast
// hardware approximations (relative error about 1e-6 over the arguments an
// activation sees), far below the bf16 rounding of the stored result; every
// branch on the mode and the activation is resolved at compile time so the 32
// columns of a chunk are independent instruction streams.
__device__ __forceinline__ float fast_sigmoid(float x) {
  return __fdividef(1.0f, 1.0f + __expf(-x));
}
template <int ACT>
__device__ __forceinline__ float gated(float g, float u, float limit, float alpha, float beta) {
  if constexpr (ACT == MOE_ACT_SILU_AND_MUL) {
    return g * fast_sigmoid(g) * u;
  } else if constexpr (ACT == MOE_ACT_GELU_AND_MUL) {
    return gelu_f(g) * u;
  } else {
    if (limit > 0.0f) {
      g = fminf(g, limit);
      u = fmaxf(fminf(u, limit), -limit);
    }
    return g * fast_sigmoid(alpha * g) * (u + beta);
  }
}

// One 32-column chunk of the calling warp's 32 output rows (row wrow0 + lane,
// columns col0..): a whole 32 x 32 box staged in shared memory and written by
// one TMA store when `boxed` (all 32 rows inside the segment), else row by
// row for the rows that are (row_ok).  obufs holds NBUF 2 KB buffers of the
// warp; obuf is the next one.  F16: the output is float16, else bfloat16.
template <int NBUF, bool F16 = false>
__device__ __forceinline__ void emit_chunk32(const float (&v)[32], int col0, int wrow0,
                                             bool boxed, bool row_ok,
                                             __nv_bfloat16* __restrict__ orow, int ncols_left,
                                             const CUtensorMap* tm_out, uint8_t* obufs,
                                             int& obuf, int lane) {
  if (boxed) {
    uint8_t* buf = obufs + obuf * OUT_BUF_BYTES;
    if (lane == 0) bulk_wait_read<NBUF - 1>();  // the last store from this buffer
    __syncwarp();
    // row `lane`, 16-byte chunk q lands at chunk q ^ ((lane >> 1) & 3)
    // (the 64-byte swizzle the output map describes): conflict-free
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 u;
      u.x = pack2<F16>(v[8 * q + 0], v[8 * q + 1]);
      u.y = pack2<F16>(v[8 * q + 2], v[8 * q + 3]);
      u.z = pack2<F16>(v[8 * q + 4], v[8 * q + 5]);
      u.w = pack2<F16>(v[8 * q + 6], v[8 * q + 7]);
      *reinterpret_cast<uint4*>(buf + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4)) = u;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tm_out, buf, col0, wrow0);
      bulk_commit();
    }
    obuf = NBUF == 1 ? 0 : obuf ^ 1;
  } else if (row_ok) {
    store_row32<F16>(orow + col0, v, ncols_left);
  }
}

// Epilogue of nchunks x 32 output columns for the 32 rows of the calling
// warp (TMEM lanes 32*(warp%4).., row wrow0 + lane), starting at output (or,
// gated, activation) column col_base: bias, activation, bf16 rounding and the
// store.  TMEM column layout from tbase: plain, chunk c at 32c; stacked, gate
// at 32c and up at up_off + 32c; interleaved, (gate, up) pairs at 64c.  Rows
// at or past m_end (the end of the tile's expert segment) are not written.
// Bias rows are N1 wide; the up bias of a stacked tile is column Nout + j of
// the expert's row, or column j of bias_up's row when the up projection is a
// tensor of its own (bias_up != nullptr, N1 = Nout).  F16: bias and output
// are float16 (the pointers' bfloat16 type is nominal), else bfloat16.
template <int MODE, int ACT, bool F16 = false>
__device__ __forceinline__ void drain_cols(uint32_t tbase, int wrow0, int m_end, int col_base,
                                           int nchunks, int up_off, int e,
                                           const __nv_bfloat16* __restrict__ bias,
                                           const __nv_bfloat16* __restrict__ bias_up, int N1,
                                           int Nout, float limit, float alpha, float beta,
                                           const CUtensorMap* tm_out, int tma_out,
                                           __nv_bfloat16* __restrict__ out, uint8_t* obufs,
                                           int& obuf, int lane) {
  const int row = wrow0 + lane;
  const bool row_ok = row < m_end;
  const __nv_bfloat16* be = bias ? bias + (size_t)e * N1 : nullptr;
  const __nv_bfloat16* bu = bias_up ? bias_up + (size_t)e * N1 : be ? be + Nout : nullptr;
  __nv_bfloat16* orow = out + (size_t)row * Nout;
  // Whole-box TMA stores only where all 32 rows of this warp belong to the
  // tile's expert segment; a ragged tail stores row by row instead so it
  // never writes rows of the next segment.
  const bool boxed = tma_out && m_end - wrow0 >= OUT_BOX;
  auto emit = [&](const float (&v)[32], int col0) {
    emit_chunk32<2, F16>(v, col0, wrow0, boxed, row_ok, orow, Nout - col0, tm_out, obufs, obuf,
                         lane);
  };
  if constexpr (MODE == kTcPlain) {
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int col0 = col_base + c * 32;
      if (col0 >= Nout) break;  // warp-uniform
      uint32_t r[32];
      tmem_ld32(tbase + c * 32, r);
      tmem_wait_ld();
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
      if (be) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (col0 + i < Nout) v[i] += ld16<F16>(be + col0 + i);
      }
      if constexpr (ACT == MOE_ACT_RELU) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = fmaxf(v[i], 0.0f);
      } else if constexpr (ACT == MOE_ACT_GELU) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = gelu_f(v[i]);
      } else if constexpr (ACT == MOE_ACT_SILU) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = v[i] * fast_sigmoid(v[i]);
      }
      emit(v, col0);
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int col0 = col_base + c * 32;  // activation column
      if (col0 >= Nout) break;
      uint32_t g[32], u[32];
      if constexpr (MODE == kTcStacked) {
        tmem_ld32(tbase + c * 32, g);           // gate columns
        tmem_ld32(tbase + up_off + c * 32, u);  // up columns
      } else {
        tmem_ld32(tbase + c * 64, g);             // (gate, up) pairs
        tmem_ld32(tbase + c * 64 + 32, u);
      }
      tmem_wait_ld();
      float gv[32], uv[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if constexpr (MODE == kTcStacked) {
          gv[i] = __uint_as_float(g[i]);
          uv[i] = __uint_as_float(u[i]);
        } else {  // pair i lives in columns 2i, 2i+1 of the 64 loaded
          gv[i] = __uint_as_float(2 * i < 32 ? g[2 * i] : u[2 * i - 32]);
          uv[i] = __uint_as_float(2 * i + 1 < 32 ? g[2 * i + 1] : u[2 * i + 1 - 32]);
        }
      }
      if (be) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (col0 + i < Nout) {
            if constexpr (MODE == kTcStacked) {
              gv[i] += ld16<F16>(be + col0 + i);
              uv[i] += ld16<F16>(bu + col0 + i);
            } else {
              gv[i] += ld16<F16>(be + 2 * (col0 + i));
              uv[i] += ld16<F16>(be + 2 * (col0 + i) + 1);
            }
          }
        }
      }
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = gated<ACT>(gv[i], uv[i], limit, alpha, beta);
      emit(v, col0);
    }
  }
}

// The whole 128-lane x 256-column accumulator of a tile: 256 output columns
// (plain) or 128 activation columns (gated, up columns 128 to the right when
// stacked) of column tile n_idx.
template <int MODE, int ACT, bool F16 = false>
__device__ __forceinline__ void drain_acc(uint32_t tbase, int wrow0, int m_end, int n_idx, int e,
                                          const __nv_bfloat16* __restrict__ bias,
                                          const __nv_bfloat16* __restrict__ bias_up, int N1, int Nout,
                                          float limit, float alpha, float beta,
                                          const CUtensorMap* tm_out, int tma_out,
                                          __nv_bfloat16* __restrict__ out, uint8_t* obufs,
                                          int& obuf, int lane) {
  if constexpr (MODE == kTcPlain)
    drain_cols<MODE, ACT, F16>(tbase, wrow0, m_end, n_idx * kEpiCols, kEpiCols / 32, 0, e, bias,
                          bias_up, N1,
                          Nout, limit, alpha, beta, tm_out, tma_out, out, obufs, obuf, lane);
  else
    drain_cols<MODE, ACT, F16>(tbase, wrow0, m_end, n_idx * (kEpiCols / 2), kEpiCols / 64,
                          kEpiCols / 2, e, bias, bias_up, N1, Nout, limit, alpha, beta, tm_out, tma_out,
                          out, obufs, obuf, lane);
}

}  // namespace tc
}  // namespace moe
