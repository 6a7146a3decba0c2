// Device pieces of the deterministic permute, shared by the permute kernels
// and the fused route + permute kernel (TileOPs "MoE Operators",
// MoEPrePermuteFwdOp; layout "contiguous · physical_psum").  Routes are cut
// into chunks of kPermuteChunk consecutive route indices.
#pragma once

#include "common.cuh"

namespace moe {
namespace pm {

// Exclusive block scan of one value per thread (blockDim.x <= 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot /*>= 33*/, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) warp_tot[wid] = x;
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int w = 0; w < nw; ++w) {
      int t = warp_tot[w];
      warp_tot[w] = acc;
      acc += t;
    }
    warp_tot[32] = acc;
  }
  __syncthreads();
  int r = warp_tot[wid] + x - v;
  *total = warp_tot[32];
  __syncthreads();
  return r;
}

// Histogram of chunk c's expert ids in shared memory (hist: E ints), written
// to counts_row[E].  Out-of-range ids are skipped and latch kDevBadIndex.
__device__ __forceinline__ void count_chunk(const int32_t* __restrict__ ids, int M, int E, int c,
                                            int* hist, int* __restrict__ counts_row,
                                            int* status) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int r0 = c * kPermuteChunk, r1 = min(M, r0 + kPermuteChunk);
  bool bad = false;
  for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    const int id = ids[r];
    if (id >= 0 && id < E) atomicAdd(&hist[id], 1);
    else bad = true;
  }
  if (bad) latch_error(status, kDevBadIndex);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts_row[e] = hist[e];
  __syncthreads();
}

// Scatter of chunk c by the W = blockDim.x / 32 warps of the CTA (W a power of
// two, kPermuteChunk / W a multiple of 32): warp w ranks its routes with
// match-any (one round per 32 routes), the per-warp expert counts are prefixed
// across warps in shared memory (wcnt: W x E ints), then every route gets
// row = off[e] (chunk c's first row of expert e) + routes of e in earlier
// warps + its rank in the warp.  Rows inside an expert follow ascending route
// index; routes with an out-of-range id get route_to_row = -1 and no row.
__device__ __forceinline__ void scatter_chunk(const int32_t* __restrict__ ids, int M, int E, int c,
                                              const int* off, int* wcnt,
                                              int32_t* __restrict__ row_to_route,
                                              int32_t* __restrict__ route_to_row) {
  const int W = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_warp = kPermuteChunk / W;
  for (int i = threadIdx.x; i < W * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int r0 = c * kPermuteChunk + warp * per_warp;
  const int r1 = min(M, min(c * kPermuteChunk + kPermuteChunk, r0 + per_warp));
  const uint32_t lt = (1u << lane) - 1u;
  int* mine = wcnt + (size_t)warp * E;
  constexpr int kMaxRounds = kPermuteChunk / 32;
  int rank_of[kMaxRounds];  // rank of this lane's route in round j
  for (int j = 0; j * 32 < per_warp; ++j) {
    const int r = r0 + j * 32 + lane;
    const bool valid = r < r1;
    const int id = valid ? ids[r] : -1;
    const bool ok = valid && id >= 0 && id < E;
    const int key = ok ? id : -1 - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    const int before = ok ? mine[id] : 0;
    __syncwarp();
    if (ok && __popc(peers & lt) == 0) mine[id] = before + __popc(peers);
    __syncwarp();
    rank_of[j & (kMaxRounds - 1)] = before + __popc(peers & lt);
  }
  __syncthreads();
  // exclusive prefix over warps, per expert, seeded with the chunk's start row
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = off[e];
    for (int w = 0; w < W; ++w) {
      const int n = wcnt[(size_t)w * E + e];
      wcnt[(size_t)w * E + e] = run;
      run += n;
    }
  }
  __syncthreads();
  for (int j = 0; j * 32 < per_warp; ++j) {
    const int r = r0 + j * 32 + lane;
    if (r >= r1) break;
    const int id = ids[r];
    if (id >= 0 && id < E) {
      const int row = mine[id] + rank_of[j & (kMaxRounds - 1)];
      row_to_route[row] = r;
      route_to_row[r] = row;
    } else {
      route_to_row[r] = -1;
    }
  }
  __syncthreads();
}

}  // namespace pm
}  // namespace moe
