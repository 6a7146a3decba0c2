// Device-side helpers shared by the kernels of libmoe.so (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace moe {

// Wait for the grids this one depends on (the previous kernel of the stream
// under programmatic stream serialization, see launch_pdl) to complete and
// their memory to be visible; a no-op when launched without it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- element I/O
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float load(const float* p) { return *p; }
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  // round to nearest even, as every cast to the operand dtype in this library
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

template <> struct Elem<__half> {
  static __device__ __forceinline__ float load(const __half* p) { return __half2float(*p); }
  static __device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
  // round to nearest even; past 65520 in magnitude, infinity (IEEE binary16)
  static __device__ __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float f16_lo(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}
// the two 16-bit element types by a flag: true = float16, false = bfloat16
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) return pack_f16x2(lo, hi); else return pack_bf16x2(lo, hi);
}
template <bool F16>
__device__ __forceinline__ float lo16(uint32_t v) {
  if constexpr (F16) return f16_lo(v); else return bf16_lo(v);
}
template <bool F16>
__device__ __forceinline__ float hi16(uint32_t v) {
  if constexpr (F16) return f16_hi(v); else return bf16_hi(v);
}

// ---------------------------------------------------------------- math
__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

// silu(g) * u  (silu_and_mul)
__device__ __forceinline__ float silu_mul(float g, float u) { return g * sigmoidf_(g) * u; }

// gelu(x) = x * Phi(x) = x/2 * (1 + erf(x / sqrt 2))
__device__ __forceinline__ float gelu_f(float x) {
  return 0.5f * x * (1.0f + erff(x * 0.7071067811865476f));
}

// the gated kinds read 2F rows (gate and up), the others F
__host__ __device__ constexpr bool act_is_gated(int kind) {
  return kind == MOE_ACT_SILU_AND_MUL || kind == MOE_ACT_SWIGLU || kind == MOE_ACT_GELU_AND_MUL;
}

// non-gated activation of one value (identity, relu, gelu, silu)
__device__ __forceinline__ float act_plain(int kind, float x) {
  return kind == MOE_ACT_RELU ? fmaxf(x, 0.0f)
         : kind == MOE_ACT_GELU ? gelu_f(x)
         : kind == MOE_ACT_SILU ? x * sigmoidf_(x)
                                : x;
}

// clamped SwiGLU; limit <= 0 disables both clamps
__device__ __forceinline__ float swiglu_f(float g, float l, float limit, float alpha, float beta) {
  if (limit > 0.0f) {
    g = fminf(g, limit);
    l = fmaxf(fminf(l, limit), -limit);
  }
  return g * sigmoidf_(alpha * g) * (l + beta);
}

// ---------------------------------------------------------------- warp reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------- status word
__device__ __forceinline__ void latch_error(int* status, int bit) {
  if (status) atomicOr(status, bit);
}

// wall-clock nanoseconds (for bounded waits)
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- segment tiles
// Tiles of an expert-segmented ("physical_psum") row space: expert e owns rows
// [seg_end[e-1], seg_end[e]) and ceil(rows / BM) row tiles, each crossed with
// `n_tiles` column tiles.  The per-expert tile prefix is built in shared
// memory by the whole block (E <= kMaxExperts), so no extra launch or host
// round trip is needed.
// Block-wide exclusive prefix of tiles; prefix has E + 1 entries.  Returns the
// total tile count.  All threads of the block must call it.
// Rows [s, t) of expert e: with stride 0, the segment between seg_end[e-1]
// and seg_end[e] (clamped to [0, M]); with stride > 0 (a masked slab), the
// first min(max(seg_end[e], 0), stride) rows from e * stride (seg_end then
// holds the valid-row counts).
__device__ __forceinline__ void seg_bounds(const int32_t* __restrict__ seg_end, int e, int M,
                                           int stride, int& s, int& t) {
  if (stride > 0) {
    s = e * stride;
    t = s + min(max(seg_end[e], 0), stride);
  } else {
    s = e == 0 ? 0 : seg_end[e - 1];
    t = seg_end[e];
    s = max(0, min(s, M));
    t = max(s, min(t, M));
  }
}

__device__ inline int build_tile_prefix(const int32_t* __restrict__ seg_end, int E, int M, int BM,
                                        int n_tiles, int* prefix, int* scratch /*>= 33 ints*/,
                                        int stride = 0) {
  const int nthr = blockDim.x, tid = threadIdx.x;
  const int per = (E + nthr - 1) / nthr;
  const int lo = tid * per, hi = min(E, lo + per);
  int local = 0;
  for (int e = lo; e < hi; ++e) {
    int s, t;
    seg_bounds(seg_end, e, M, stride, s, t);
    int mt = (t - s + BM - 1) / BM;
    local += mt * n_tiles;
  }
  // inclusive scan of `local` across the block
  const int lane = tid & 31, wid = tid >> 5, nw = (nthr + 31) >> 5;
  int v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) scratch[wid] = v;
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int w = 0; w < nw; ++w) {
      int x = scratch[w];
      scratch[w] = acc;
      acc += x;
    }
    scratch[32] = acc;
  }
  __syncthreads();
  int run = scratch[wid] + v - local;  // exclusive prefix of this thread
  for (int e = lo; e < hi; ++e) {
    prefix[e] = run;
    int s, t;
    seg_bounds(seg_end, e, M, stride, s, t);
    run += ((t - s + BM - 1) / BM) * n_tiles;
  }
  if (tid == 0) prefix[E] = scratch[32];
  __syncthreads();
  return scratch[32];
}

struct SegTile {
  int e;       // expert
  int m0;      // first row of the tile
  int m_end;   // one past the last valid row (segment end)
  int n_idx;   // column tile index
};

// Tile t -> (expert, row tile, column tile).  Inside an expert, column tiles
// are the outer loop and row tiles the inner one, so concurrent CTAs share
// each weight tile through L2.
__device__ __forceinline__ SegTile decode_tile(int t, const int* prefix, const int32_t* seg_end,
                                               int E, int M, int BM, int n_tiles,
                                               int stride = 0) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {  // last e with prefix[e] <= t (skips empty experts)
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  SegTile r;
  r.e = lo;
  int s, e_end;
  seg_bounds(seg_end, lo, M, stride, s, e_end);
  int mt = (e_end - s + BM - 1) / BM;
  int local = t - prefix[lo];
  r.n_idx = local / mt;
  r.m0 = s + (local % mt) * BM;
  r.m_end = e_end;
  return r;
}

}  // namespace moe
