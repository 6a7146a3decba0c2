// Indexed small-route expert MLP (TileOPs "MoE Operators",
// IndexedExpertMLPFwdOp): routes that share an expert are grouped and the
// expert's weights are streamed from HBM once for all of them, so DRAM traffic
// is one read of each distinct expert's w_gate_up and w_down.  The arithmetic
// and rounding points are those of the staged pipeline: fp32 dot products,
// silu(gate) * up rounded to bf16, down product rounded to bf16, fp32 weighted
// combine in fixed k order.
//
//   gate_up : work item = (active expert, 32 activation columns); each warp
//             streams 4 (gate row, up row) pairs with 16-byte loads and dots
//             them with every route's hidden row of that expert
//   down    : work item = (active expert, 32 rows of w_down); each warp
//             streams 4 rows and dots them with every route's activation row
//   combine : the deterministic gather-combine of the staged pipeline
// Both streaming kernels are persistent (one resident round of CTAs) over a
// device-side list of the experts that have routes, so no host
// synchronisation is needed.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kNR = 8;          // routes of one expert handled per pass
constexpr int kColsPerItem = 32;
constexpr int kWarps = 8;

__device__ __forceinline__ void fma8(float& acc, const uint4& w, const uint4& x) {
  acc = fmaf(bf16_lo(w.x), bf16_lo(x.x), acc);
  acc = fmaf(bf16_hi(w.x), bf16_hi(x.x), acc);
  acc = fmaf(bf16_lo(w.y), bf16_lo(x.y), acc);
  acc = fmaf(bf16_hi(w.y), bf16_hi(x.y), acc);
  acc = fmaf(bf16_lo(w.z), bf16_lo(x.z), acc);
  acc = fmaf(bf16_hi(w.z), bf16_hi(x.z), acc);
  acc = fmaf(bf16_lo(w.w), bf16_lo(x.w), acc);
  acc = fmaf(bf16_hi(w.w), bf16_hi(x.w), acc);
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// act[row, j] = bf16(silu(W1[e, j] . x_t) * (W1[e, F + j] . x_t)) for the rows of e
__global__ void __launch_bounds__(kWarps * 32) indexed_gate_up(
    const __nv_bfloat16* __restrict__ hidden, const __nv_bfloat16* __restrict__ w1,
    const int32_t* __restrict__ seg_end, const int32_t* __restrict__ row_to_route,
    const int* __restrict__ active, const int* __restrict__ num_active, int T, int H, int F,
    int K, __nv_bfloat16* __restrict__ act) {
  pdl_wait();  // everything below reads results of earlier launches
  const int D = *num_active;
  const int items_per_e = F / kColsPerItem;
  const int n_items = D * items_per_e;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = H / 8;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int d = item / items_per_e;
    const int e = active[d];
    const int r_begin = e == 0 ? 0 : seg_end[e - 1];
    const int r_end = seg_end[e];
    const int jbase = (item % items_per_e) * kColsPerItem;
    for (int r0 = r_begin; r0 < r_end; r0 += kNR) {
      const int nr = min(kNR, r_end - r0);
      const uint4* xr[kNR];
#pragma unroll
      for (int q = 0; q < kNR; ++q) {
        int t = q < nr ? row_to_route[r0 + q] / K : 0;
        t = min(max(t, 0), T - 1);
        xr[q] = reinterpret_cast<const uint4*>(hidden + (size_t)t * H);
      }
      for (int jj = warp; jj < kColsPerItem; jj += kWarps) {
        const int j = jbase + jj;
        const uint4* wg = reinterpret_cast<const uint4*>(w1 + ((size_t)e * 2 * F + j) * H);
        const uint4* wu = reinterpret_cast<const uint4*>(w1 + ((size_t)e * 2 * F + F + j) * H);
        float ag[kNR], au[kNR];
#pragma unroll
        for (int q = 0; q < kNR; ++q) ag[q] = au[q] = 0.f;
        int v = lane;
        for (; v + 96 < nvec; v += 128) {
          uint4 g0 = ldg_stream(wg + v), g1 = ldg_stream(wg + v + 32);
          uint4 g2 = ldg_stream(wg + v + 64), g3 = ldg_stream(wg + v + 96);
          uint4 u0 = ldg_stream(wu + v), u1 = ldg_stream(wu + v + 32);
          uint4 u2 = ldg_stream(wu + v + 64), u3 = ldg_stream(wu + v + 96);
#pragma unroll
          for (int q = 0; q < kNR; ++q) {
            if (q < nr) {
              uint4 x0 = __ldg(xr[q] + v), x1 = __ldg(xr[q] + v + 32);
              uint4 x2 = __ldg(xr[q] + v + 64), x3 = __ldg(xr[q] + v + 96);
              fma8(ag[q], g0, x0); fma8(ag[q], g1, x1); fma8(ag[q], g2, x2); fma8(ag[q], g3, x3);
              fma8(au[q], u0, x0); fma8(au[q], u1, x1); fma8(au[q], u2, x2); fma8(au[q], u3, x3);
            }
          }
        }
        for (; v < nvec; v += 32) {
          uint4 g0 = ldg_stream(wg + v), u0 = ldg_stream(wu + v);
#pragma unroll
          for (int q = 0; q < kNR; ++q) {
            if (q < nr) {
              uint4 x0 = __ldg(xr[q] + v);
              fma8(ag[q], g0, x0);
              fma8(au[q], u0, x0);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < kNR; ++q) {
          if (q < nr) {
            float g = warp_sum(ag[q]);
            float u = warp_sum(au[q]);
            if (lane == 0) act[(size_t)(r0 + q) * F + j] = __float2bfloat16_rn(silu_mul(g, u));
          }
        }
      }
    }
  }
}

// y[row, h] = bf16(W2[e, h] . act[row]) for the rows of e
__global__ void __launch_bounds__(kWarps * 32) indexed_down(
    const __nv_bfloat16* __restrict__ w2, const __nv_bfloat16* __restrict__ act,
    const int32_t* __restrict__ seg_end, const int* __restrict__ active,
    const int* __restrict__ num_active, int H, int F, __nv_bfloat16* __restrict__ y) {
  pdl_wait();  // everything below reads results of earlier launches
  const int D = *num_active;
  const int items_per_e = H / kColsPerItem;
  const int n_items = D * items_per_e;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = F / 8;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int d = item / items_per_e;
    const int e = active[d];
    const int r_begin = e == 0 ? 0 : seg_end[e - 1];
    const int r_end = seg_end[e];
    const int hbase = (item % items_per_e) * kColsPerItem;
    for (int r0 = r_begin; r0 < r_end; r0 += kNR) {
      const int nr = min(kNR, r_end - r0);
      for (int hh = warp; hh < kColsPerItem; hh += kWarps) {
        const int h = hbase + hh;
        const uint4* wr = reinterpret_cast<const uint4*>(w2 + ((size_t)e * H + h) * F);
        float acc[kNR];
#pragma unroll
        for (int q = 0; q < kNR; ++q) acc[q] = 0.f;
        int v = lane;
        for (; v + 96 < nvec; v += 128) {
          uint4 w0 = ldg_stream(wr + v), w1v = ldg_stream(wr + v + 32);
          uint4 w2v = ldg_stream(wr + v + 64), w3 = ldg_stream(wr + v + 96);
#pragma unroll
          for (int q = 0; q < kNR; ++q) {
            if (q < nr) {
              const uint4* ar = reinterpret_cast<const uint4*>(act + (size_t)(r0 + q) * F);
              fma8(acc[q], w0, __ldg(ar + v));
              fma8(acc[q], w1v, __ldg(ar + v + 32));
              fma8(acc[q], w2v, __ldg(ar + v + 64));
              fma8(acc[q], w3, __ldg(ar + v + 96));
            }
          }
        }
        for (; v < nvec; v += 32) {
          uint4 w0 = ldg_stream(wr + v);
#pragma unroll
          for (int q = 0; q < kNR; ++q) {
            if (q < nr) {
              const uint4* ar = reinterpret_cast<const uint4*>(act + (size_t)(r0 + q) * F);
              fma8(acc[q], w0, __ldg(ar + v));
            }
          }
        }
#pragma unroll
        for (int q = 0; q < kNR; ++q) {
          if (q < nr) {
            float s = warp_sum(acc[q]);
            if (lane == 0) y[(size_t)(r0 + q) * H + h] = __float2bfloat16_rn(s);
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_indexed(const void* hidden, const void* w1, const void* w2, const float* w,
                           const int32_t* ids, int T, int H, int F, int E, int K, float scale,
                           void* out, void* ws, const ForwardWs& L, cudaStream_t s,
                           bool maps_ready) {
  const int M = T * K;
  if (M == 0) return cudaSuccess;
  char* base = static_cast<char*>(ws);
  int32_t* seg_end = reinterpret_cast<int32_t*>(base + L.seg_end);
  int32_t* r2r = reinterpret_cast<int32_t*>(base + L.row_to_route);
  int32_t* route_to_row = reinterpret_cast<int32_t*>(base + L.route_to_row);
  __nv_bfloat16* act = reinterpret_cast<__nv_bfloat16*>(base + L.act);
  __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(base + L.y);
  PermuteWs P(M, E);
  const int* active = reinterpret_cast<const int*>(base + P.active);
  const int* num_active = reinterpret_cast<const int*>(base + P.num_active);

  cudaError_t err = cudaSuccess;
  if (!maps_ready) {
    err = launch_permute(nullptr, 2, ids, T, H, E, K, nullptr, seg_end, r2r, route_to_row, ws, s);
    if (err != cudaSuccess) return err;
  }
  // One resident round of CTAs per kernel (its occupancy x the SM count):
  // CTAs beyond what the SMs hold at once would start only when whole CTAs
  // of the first round finish all their items, and that second round is
  // what sets the tail (measured on the Kimi-K2-style decode: 1250 vs
  // 1400 us with the grid at 4 CTAs per SM, which registers cap at 2 for
  // the gate_up kernel and 3 for the down kernel; 32-column items instead
  // of 64 then 1241 us).
  const int per_sm_gu = resident_ctas((const void*)indexed_gate_up, kWarps * 32);
  const int per_sm_dn = resident_ctas((const void*)indexed_down, kWarps * 32);
  launch_pdl(indexed_gate_up, num_sms() * per_sm_gu, kWarps * 32, 0, s,
      static_cast<const __nv_bfloat16*>(hidden),
      static_cast<const __nv_bfloat16*>(w1), seg_end, r2r, active, num_active, T, H, F, K, act);
  launch_pdl(indexed_down, num_sms() * per_sm_dn, kWarps * 32, 0, s,
      static_cast<const __nv_bfloat16*>(w2), act,
      seg_end, active, num_active, H, F, y);
  count_launch(2);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  return launch_combine(y, w, route_to_row, T, K, H, MOE_BF16, scale, out, s);
}

}  // namespace moe
