// Fused route + permute index maps: one persistent launch (one CTA of 16
// warps per SM) instead of the router and the three permute launches, whose
// cost on the forward is mostly the fixed latency of each launch.
//
//   A  route: warp per token, grid-stride over tokens (route_dev.cuh)
//   -- grid barrier (every token's ids written)
//   B  count: CTA per chunk of kPermuteChunk routes, histogram -> counts[c][E]
//   -- grid barrier (every chunk counted)
//   C  scan:  every CTA that owns a chunk reads all counts, scans the expert
//             totals into expert start rows (CTA 0 writes seg_end and the
//             active-expert list) and, for its chunks, the first row of each
//             expert in the chunk
//   D  scatter: the chunk's routes get their rows (permute_dev.cuh)
// The result is bit-identical to moe_route followed by moe_permute (same
// routing code, same chunking, same in-order ranks).
//
// The grid barriers spin on two counters in the status area of the
// workspace (zero when the status area is cleared) and reset them for the
// next launch: a third counter counts the CTAs past the second barrier, and
// the last one zeroes all three (no CTA reads them again in this launch; the
// next launch reads them after the grids in between have completed).  The
// launch is cooperative (one CTA per SM), so all CTAs of the grid are
// resident together, and every spin is bounded: a barrier that runs out
// latches the timeout bit and the CTA stops, leaving the counters for the
// status clear that the error requires.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "permute_dev.cuh"
#include "route_dev.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using rt::RouteArgs;

constexpr int kFusedWarps = 16;  // kPermuteChunk / 16 = 64 routes per warp in the scatter
// Large batches (more than two tokens a warp at 16 warps per SM) with at most
// eight registers of scores a lane run 32 warps per CTA: the routing phase
// then takes at most two tokens a warp on the DeepSeek-V3-style batch (the
// launch 43.7 vs 47.7 us); smaller batches keep 16 (more registers a thread,
// and 32 warps measured slower on the gpt-oss-style batch).
constexpr int kFusedWarpsLarge = 32;

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Barrier parameters: the arrivals a barrier waits for beyond the grid's
// own CTAs (0; 1 only under the test hook, so that the wait cannot end) and
// the limit of each wait.
struct BarrierArgs {
  int extra;
  uint64_t limit_ns;
};

// All CTAs of the grid meet here; false (and the timeout bit) if one never came.
__device__ bool grid_barrier(int* ctr, int* status, BarrierArgs b) {
  __shared__ int ok_s;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's writes before its arrival
    atomicAdd(ctr, 1);
    const uint64_t t0 = global_ns();
    int ok = 1;
    while (ld_acquire(ctr) < (int)gridDim.x + b.extra) {
      if (global_ns() - t0 > b.limit_ns) {
        latch_error(status, kDevTimeout);
        ok = 0;
        break;
      }
      __nanosleep(128);
    }
    __threadfence();
    ok_s = ok;
  }
  __syncthreads();
  return ok_s != 0;
}

// counts[0..n)[e] summed (all) and counts[0..c)[e] summed (before), one
// pass with 16 loads in flight
__device__ __forceinline__ void column_sums(const int* __restrict__ counts, int E, int e, int n,
                                            int c, int& all, int& before) {
  int sa = 0, sb = 0;
  for (int c0 = 0; c0 < n; c0 += 16) {
    int v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = c0 + j < n ? counts[(size_t)(c0 + j) * E + e] : 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      sa += v[j];
      sb += c0 + j < c ? v[j] : 0;
    }
  }
  all = sa;
  before = sb;
}
// counts[0..n)[e] summed
__device__ __forceinline__ int column_sum(const int* __restrict__ counts, int E, int e, int n) {
  int all, before;
  column_sums(counts, E, e, n, 0, all, before);
  return all;
}

template <int NPL, int W>
__global__ void __launch_bounds__(W * 32, 1) route_permute_kernel(
    const void* __restrict__ logits, const float* __restrict__ bias,
    const int32_t* __restrict__ ids_in, int T, int E, RouteArgs a, float* __restrict__ w_out,
    int32_t* __restrict__ id_out, void* __restrict__ probs, float* __restrict__ wscale,
    int C, int* __restrict__ counts, int32_t* __restrict__ seg_end, int* __restrict__ active,
    int* __restrict__ num_active, int32_t* __restrict__ row_to_route,
    int32_t* __restrict__ route_to_row, int* status, int* bar, BarrierArgs ba) {
  extern __shared__ int smem[];  // [E] expert start | [E] chunk offsets / histogram | [W][E]
  pdl_wait();  // everything below reads results of earlier launches
  const int warp = threadIdx.x >> 5, tid = threadIdx.x;  // W warps (blockDim.x == 32 W)
  const int M = T * a.K;
  // ---- A: route (the next token's logits are loaded before this one is routed)
  {
    const int stride = gridDim.x * W;
    int t = blockIdx.x * W + warp;
    float z[NPL], zn[NPL];
    if (t < T) rt::load_logits<NPL>(t, logits, E, a.dt, z);
    for (; t < T; t += stride) {
      if (t + stride < T) rt::load_logits<NPL>(t + stride, logits, E, a.dt, zn);
      rt::route_loaded<NPL>(t, z, bias, ids_in, E, a, w_out, id_out, probs, wscale);
#pragma unroll
      for (int i = 0; i < NPL; ++i) z[i] = zn[i];
    }
  }
  if (!grid_barrier(&bar[0], status, ba)) return;
  // ---- B: count
  int* start = smem;
  int* offs = smem + E;
  int* wcnt = smem + 2 * E;
  for (int c = blockIdx.x; c < C; c += gridDim.x)
    pm::count_chunk(id_out, M, E, c, offs, counts + (size_t)c * E, status);
  if (!grid_barrier(&bar[1], status, ba)) return;
  if (threadIdx.x == 0 && atomicAdd(&bar[2], 1) == (int)gridDim.x - 1) {
    // every CTA is past both barriers: ready for the next launch
    bar[0] = 0;
    bar[1] = 0;
    bar[2] = 0;
  }
  if ((int)blockIdx.x >= C) return;  // no chunk of its own
  // ---- C: expert start rows (one thread per expert, E <= blockDim.x); the
  // same pass sums the counts of the chunks before this CTA's first chunk
  int tot = 0, before = 0;
  if (tid < E) column_sums(counts, E, tid, C, blockIdx.x, tot, before);
  __shared__ int wt[33];
  int total, n_act;
  const int first = pm::block_exclusive_scan(tot, wt, &total);
  const int afirst = pm::block_exclusive_scan(tid < E && tot > 0 ? 1 : 0, wt, &n_act);
  if (tid < E) {
    start[tid] = first;
    if (blockIdx.x == 0) {
      seg_end[tid] = first + tot;
      if (tot > 0) active[afirst] = tid;
    }
  }
  if (blockIdx.x == 0 && tid == 0) *num_active = n_act;
  __syncthreads();
  // ---- D: this CTA's chunks
  for (int c = blockIdx.x; c < C; c += gridDim.x) {
    if (tid < E)
      offs[tid] = start[tid] + (c == (int)blockIdx.x ? before : column_sum(counts, E, tid, c));
    __syncthreads();
    pm::scatter_chunk(id_out, M, E, c, offs, wcnt, row_to_route, route_to_row);
  }
}

template <int NPL, int W>
cudaError_t launch_npl(const void* logits, const float* bias, const int32_t* ids_in, int T,
                       int E, const RouteArgs& a, float* w, int32_t* ids, void* probs,
                       float* wscale, int C, int* counts, int32_t* seg_end, int* active,
                       int* num_active, int32_t* r2r, int32_t* route_to_row, int* status, int* bar,
                       size_t smem, int grid, BarrierArgs ba, cudaStream_t s) {
  set_smem_limit((const void*)route_permute_kernel<NPL, W>, (2 + W) * kFusedWarps * 32 * 4);
  // A cooperative launch: the scheduler starts the grid only when all of its
  // CTAs can be resident at once, so two of these kernels running on two
  // streams never each hold part of the GPU while waiting at a barrier for
  // CTAs the other one keeps out.  Programmatic serialisation is asked for too
  // (the kernel waits on the previous grid before it reads anything); a driver
  // that refuses the pair gets the cooperative launch alone.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  static std::atomic<int> n_attrs{2};
  cfg.numAttrs = n_attrs.load();
  cudaError_t e = cudaLaunchKernelEx(&cfg, route_permute_kernel<NPL, W>, logits, bias, ids_in, T, E,
                                     a, w, ids, probs, wscale, C, counts, seg_end, active,
                                     num_active, r2r, route_to_row, status, bar, ba);
  if (e == cudaErrorInvalidValue || e == cudaErrorNotSupported) {
    (void)cudaGetLastError();
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, route_permute_kernel<NPL, W>, logits, bias, ids_in, T, E, a, w, ids,
                           probs, wscale, C, counts, seg_end, active, num_active, r2r,
                           route_to_row, status, bar, ba);
    if (e == cudaSuccess) n_attrs.store(1);
  }
  return e;
}

// Test hook state (see moe_test_force_wait_timeout): off by default.
std::atomic<int> g_force_timeout{0};
std::atomic<long long> g_force_timeout_ns{0};

}  // namespace

int set_wait_timeout_test(int enable, long long limit_ns) {
  if (enable) g_force_timeout_ns.store(limit_ns > 0 ? limit_ns : 1);
  return g_force_timeout.exchange(enable ? 1 : 0);
}

bool route_permute_ok(int E) { return E >= 1 && E <= kFusedWarps * 32; }

cudaError_t launch_route_permute(const void* logits, const float* bias, const int32_t* ids_in,
                                 int T, int E, const moe_route_params& p, float* w, int32_t* ids,
                                 void* probs, float* wscale, int32_t* seg_end,
                                 int32_t* row_to_route, int32_t* route_to_row, void* ws,
                                 cudaStream_t s) {
  const int K = p.top_k;
  const int M = T * K;
  if (M == 0 || !route_permute_ok(E)) return cudaErrorInvalidValue;
  PermuteWs L(M, E);
  char* base = static_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(base);
  int* bar = reinterpret_cast<int*>(base + 16);  // barrier counters in the status area
  int* counts = reinterpret_cast<int*>(base + L.counts);
  int* active = reinterpret_cast<int*>(base + L.active);
  int* num_active = reinterpret_cast<int*>(base + L.num_active);
  const int C = (M + kPermuteChunk - 1) / kPermuteChunk;
  const int grid = num_sms();
  const int npl = (E + 31) / 32;
  const bool large = npl <= 8 && T > 2 * kFusedWarps * grid;
  const size_t smem = (size_t)(2 + (large ? kFusedWarpsLarge : kFusedWarps)) * E * 4;
  cudaError_t e = cudaSuccess;
  const RouteArgs a = rt::route_args(p, probs, wscale);
  BarrierArgs ba{0, tc::kTimeoutNs};
  if (g_force_timeout.load()) ba = BarrierArgs{1, (uint64_t)g_force_timeout_ns.load()};
  auto go = [&](auto tag) {
    constexpr int N = decltype(tag)::value;
    return launch_npl<N, kFusedWarps>(logits, bias, ids_in, T, E, a, w, ids, probs, wscale, C,
                                      counts, seg_end, active, num_active, row_to_route,
                                      route_to_row, status, bar, smem, grid, ba, s);
  };
  auto go_large = [&](auto tag) {
    constexpr int N = decltype(tag)::value;
    return launch_npl<N, kFusedWarpsLarge>(logits, bias, ids_in, T, E, a, w, ids, probs, wscale,
                                           C, counts, seg_end, active, num_active, row_to_route,
                                           route_to_row, status, bar, smem, grid, ba, s);
  };
  if (large) {
    if (npl <= 1) e = go_large(std::integral_constant<int, 1>{});
    else if (npl <= 2) e = go_large(std::integral_constant<int, 2>{});
    else if (npl <= 4) e = go_large(std::integral_constant<int, 4>{});
    else e = go_large(std::integral_constant<int, 8>{});
  } else if (npl <= 1) e = go(std::integral_constant<int, 1>{});
  else if (npl <= 2) e = go(std::integral_constant<int, 2>{});
  else if (npl <= 4) e = go(std::integral_constant<int, 4>{});
  else if (npl <= 8) e = go(std::integral_constant<int, 8>{});
  else if (npl <= 12) e = go(std::integral_constant<int, 12>{});
  else e = go(std::integral_constant<int, 16>{});
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
