// Permutation into the tight expert-contiguous layout and the inverse
// weighted combine.  TileOPs "MoE Operators": MoEPrePermuteFwdOp (rows grouped
// by expert, layout "contiguous · physical_psum" = segment end rows),
// MoEPostPermuteFwdOp (restore token order, apply the routing weights once,
// reduce over k, cast) and FusedMoEExpertsFwdOp (the weighted sum).
//
// Permute = 4 launches, all deterministic:
//   count   : one CTA per chunk of kPermuteChunk routes, shared-memory histogram
//   scan    : one CTA; per-expert totals, exclusive scan -> seg_end, per-chunk
//             start offsets, list of experts that have routes
//   scatter : one warp per chunk; routes of a chunk are ranked in order with
//             warp match-any, so rows inside an expert follow ascending route
//   gather  : one warp per row copies the hidden row with 128-bit accesses
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "permute_dev.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) perm_count(const int32_t* __restrict__ ids, int M, int E,
                                                  int* __restrict__ counts, int* status) {
  pdl_wait();  // everything below reads results of earlier launches
  extern __shared__ int hist[];
  pm::count_chunk(ids, M, E, blockIdx.x, hist, counts + (size_t)blockIdx.x * E, status);
}

// One CTA.  Thread i owns a contiguous run of experts; for each it sums the
// expert's count over the chunks (coalesced across the warp, 16 loads in
// flight), the totals are scanned across the block into segment starts, and
// counts[c][e] is overwritten with the first row of expert e's routes in chunk
// c (start + routes of e in earlier chunks).  The experts that have routes are
// listed in ascending order.
constexpr int kScanBatch = 16;

__global__ void __launch_bounds__(1024) perm_scan(int* __restrict__ counts, int C, int E,
                                                  int32_t* __restrict__ seg_end,
                                                  int* __restrict__ active,
                                                  int* __restrict__ num_active) {
  pdl_wait();  // everything below reads results of earlier launches
  __shared__ int wt[33];
  const int nthr = blockDim.x, tid = threadIdx.x;
  const int per = (E + nthr - 1) / nthr;
  const int lo = min(E, tid * per), hi = min(E, lo + per);
  int tot_local = 0, act_local = 0;
  for (int e = lo; e < hi; ++e) {
    int s = 0;
    for (int c0 = 0; c0 < C; c0 += kScanBatch) {
      int v[kScanBatch];
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j)
        v[j] = c0 + j < C ? counts[(size_t)(c0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j) s += v[j];
    }
    tot_local += s;
    act_local += s > 0;
  }
  int total, n_act;
  int start = pm::block_exclusive_scan(tot_local, wt, &total);
  int astart = pm::block_exclusive_scan(act_local, wt, &n_act);
  for (int e = lo; e < hi; ++e) {
    int run = start;
    for (int c0 = 0; c0 < C; c0 += kScanBatch) {
      int v[kScanBatch];
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j)
        v[j] = c0 + j < C ? counts[(size_t)(c0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j) {
        if (c0 + j < C) counts[(size_t)(c0 + j) * E + e] = run;
        run += v[j];
      }
    }
    seg_end[e] = run;
    if (run > start) active[astart++] = e;
    start = run;
  }
  if (tid == 0) *num_active = n_act;
}

__global__ void __launch_bounds__(32) perm_scatter(const int32_t* __restrict__ ids, int M, int E,
                                                   const int* __restrict__ offsets,
                                                   int32_t* __restrict__ row_to_route,
                                                   int32_t* __restrict__ route_to_row) {
  pdl_wait();  // everything below reads results of earlier launches
  extern __shared__ int cur[];
  const int lane = threadIdx.x;
  const int* off = offsets + (size_t)blockIdx.x * E;
  for (int e = lane; e < E; e += 32) cur[e] = off[e];
  __syncwarp();
  const int r0 = blockIdx.x * kPermuteChunk, r1 = min(M, r0 + kPermuteChunk);
  constexpr int J = kPermuteChunk / 32;
  int idv[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    int r = r0 + j * 32 + lane;
    idv[j] = r < r1 ? __ldg(ids + r) : -1;
  }
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int r = r0 + j * 32 + lane;
    if (r0 + j * 32 >= r1) break;  // warp-uniform
    const bool valid = r < r1;
    const int id = idv[j];
    const bool ok = valid && id >= 0 && id < E;
    const int key = ok ? id : -1 - lane;  // invalid lanes never group
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    const int rank = __popc(peers & lt);
    const int b = ok ? cur[id] : 0;
    __syncwarp();
    if (ok) {
      const int row = b + rank;
      row_to_route[row] = r;
      route_to_row[r] = row;
      if (rank == 0) cur[id] = b + __popc(peers);
    } else if (valid) {
      route_to_row[r] = -1;
    }
    __syncwarp();
  }
}

// Scatter of one chunk per CTA (pm::scatter_chunk).
__global__ void __launch_bounds__(1024) perm_scatter_cta(const int32_t* __restrict__ ids, int M,
                                                         int E, const int* __restrict__ offsets,
                                                         int32_t* __restrict__ row_to_route,
                                                         int32_t* __restrict__ route_to_row) {
  pdl_wait();  // everything below reads results of earlier launches
  extern __shared__ int wcnt[];  // [W][E]
  pm::scatter_chunk(ids, M, E, blockIdx.x, offsets + (size_t)blockIdx.x * E, wcnt, row_to_route,
                    route_to_row);
}

// expert_input[row] = hidden[row_to_route[row] / K], rows < seg_end[E-1]
template <int VEC_BYTES>
__global__ void __launch_bounds__(256) perm_gather(const char* __restrict__ hidden,
                                                   const int32_t* __restrict__ row_to_route,
                                                   const int32_t* __restrict__ seg_end, int E,
                                                   int K, int T, size_t row_bytes,
                                                   char* __restrict__ out, int* status) {
  pdl_wait();  // everything below reads results of earlier launches
  const int warps = blockDim.x >> 5;
  const int row = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int n_rows = seg_end[E - 1];
  if (row >= n_rows) return;
  const int r = row_to_route[row];
  const int t = r / K;
  if (r < 0 || t >= T) {
    if (lane == 0) latch_error(status, kDevBadIndex);
    return;
  }
  const char* src = hidden + (size_t)t * row_bytes;
  char* dst = out + (size_t)row * row_bytes;
  if constexpr (VEC_BYTES == 16) {
    const int4* s4 = reinterpret_cast<const int4*>(src);
    int4* d4 = reinterpret_cast<int4*>(dst);
    const int n = (int)(row_bytes / 16);
    int i = lane;
    for (; i + 96 < n; i += 128) {
      int4 a = __ldg(s4 + i), b = __ldg(s4 + i + 32), c = __ldg(s4 + i + 64), d = __ldg(s4 + i + 96);
      d4[i] = a;
      d4[i + 32] = b;
      d4[i + 64] = c;
      d4[i + 96] = d;
    }
    for (; i < n; i += 32) d4[i] = __ldg(s4 + i);
  } else {
    const uint16_t* s2 = reinterpret_cast<const uint16_t*>(src);
    uint16_t* d2 = reinterpret_cast<uint16_t*>(dst);
    for (size_t i = lane; i < row_bytes / 2; i += 32) d2[i] = s2[i];
  }
}

// out[t] = scale * sum_k w[t,k] * y[route_to_row[t*K+k]], fixed k order, fp32.
// One item = VEC consecutive columns of one token; persistent grid-stride
// threads take items i, i + stride, ..., so that each thread keeps several
// rows' loads in flight and no block is launched for a few loads only.
template <typename T, int VEC>
__device__ __forceinline__ void combine_item(const T* __restrict__ y, const float* __restrict__ w,
                                             const int32_t* __restrict__ r2r, int K, int H,
                                             int M, float scale, T* __restrict__ out, int t,
                                             int v, const float* __restrict__ tscale) {
  if (tscale) scale *= __ldg(tscale + t);
  float acc[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
  const int32_t* rr = r2r + (size_t)t * K;
  const float* ww = w + (size_t)t * K;
  for (int k0 = 0; k0 < K; k0 += 8) {
    // all index and weight loads of the group first, then the row loads
    int row[8];
    float wk[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool in = k0 + j < K;
      row[j] = in ? __ldg(rr + k0 + j) : -1;
      wk[j] = in ? __ldg(ww + k0 + j) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool ok = row[j] >= 0 && row[j] < M;
      const T* src = y + (size_t)(ok ? row[j] : 0) * H + (size_t)v * VEC;
      if constexpr (VEC == 8) {  // bf16 or f16 x 8 = 16 bytes
        constexpr bool H16 = std::is_same<T, __half>::value;
        int4 q = ok ? __ldg(reinterpret_cast<const int4*>(src)) : make_int4(0, 0, 0, 0);
        const uint32_t u[4] = {(uint32_t)q.x, (uint32_t)q.y, (uint32_t)q.z, (uint32_t)q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(wk[j], lo16<H16>(u[i]), acc[2 * i]);
          acc[2 * i + 1] = fmaf(wk[j], hi16<H16>(u[i]), acc[2 * i + 1]);
        }
      } else if constexpr (VEC == 4) {  // f32 x 4
        float4 q = ok ? __ldg(reinterpret_cast<const float4*>(src)) : make_float4(0, 0, 0, 0);
        acc[0] = fmaf(wk[j], q.x, acc[0]);
        acc[1] = fmaf(wk[j], q.y, acc[1]);
        acc[2] = fmaf(wk[j], q.z, acc[2]);
        acc[3] = fmaf(wk[j], q.w, acc[3]);
      } else {
        if (ok) {
#pragma unroll
          for (int i = 0; i < VEC; ++i) acc[i] = fmaf(wk[j], Elem<T>::to_f(src[i]), acc[i]);
        }
      }
    }
  }
  T* dst = out + (size_t)t * H + (size_t)v * VEC;
  if constexpr (VEC == 8) {
    constexpr bool H16 = std::is_same<T, __half>::value;
    int4 q;
    q.x = (int)pack2<H16>(scale * acc[0], scale * acc[1]);
    q.y = (int)pack2<H16>(scale * acc[2], scale * acc[3]);
    q.z = (int)pack2<H16>(scale * acc[4], scale * acc[5]);
    q.w = (int)pack2<H16>(scale * acc[6], scale * acc[7]);
    *reinterpret_cast<int4*>(dst) = q;
  } else if constexpr (VEC == 4) {
    *reinterpret_cast<float4*>(dst) =
        make_float4(scale * acc[0], scale * acc[1], scale * acc[2], scale * acc[3]);
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) dst[i] = Elem<T>::from_f(scale * acc[i]);
  }
}

template <typename T, int VEC>
__global__ void __launch_bounds__(256) combine_kernel(const T* __restrict__ y,
                                                      const float* __restrict__ w,
                                                      const int32_t* __restrict__ r2r, int Tn,
                                                      int K, int H, int M, float scale,
                                                      T* __restrict__ out,
                                                      const float* __restrict__ tscale) {
  pdl_wait();  // everything below reads results of earlier launches
  const int nvec = H / VEC;
  const long long items = (long long)Tn * nvec;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < items; i += stride) {
    const int t = (int)(i / nvec), v = (int)(i - (long long)t * nvec);
    combine_item<T, VEC>(y, w, r2r, K, H, M, scale, out, t, v, tscale);
  }
}

// Plain copy by the SMs, 16 bytes per thread and step (a grid-stride loop over
// one CTA per SM): used to bring page-locked host activations in, where the
// SMs' reads over the host link outrun a copy engine.
__global__ void __launch_bounds__(256) copy16_kernel(const int4* __restrict__ src,
                                                     int4* __restrict__ dst, long long n) {
  long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const int4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n; i += stride) dst[i] = src[i];
}

// ---- padded permute-align layout (TileOPs "MoE Operators",
// MoEPermuteAlignFwdOp), built from the tight layout's maps: every expert's
// range is its segment of the tight layout moved to a start rounded up to
// block_size, the rest of the range numel.

// sorted_token_ids[0, L) = numel, expert_ids[0, nb) = -1
__global__ void align_fill_kernel(int32_t* __restrict__ sorted_ids, long long L, int32_t numel,
                                  int32_t* __restrict__ expert_ids, int nb) {
  pdl_wait();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < L; i += stride)
    sorted_ids[i] = numel;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nb; i += stride)
    expert_ids[i] = -1;
}

// One CTA: padded starts (exclusive prefix of the counts rounded up to
// block_size) into pstart, the owner of every block of the ranges into
// expert_ids, and the padded total.
__global__ void __launch_bounds__(1024) align_scan_kernel(const int32_t* __restrict__ seg_end,
                                                          int E, int block_size,
                                                          int32_t* __restrict__ pstart,
                                                          int32_t* __restrict__ expert_ids,
                                                          int32_t* __restrict__ num_post_pad) {
  pdl_wait();
  __shared__ int wt[33];
  int base = 0;
  for (int e0 = 0; e0 < E; e0 += blockDim.x) {
    const int e = e0 + (int)threadIdx.x;
    int padded = 0;
    if (e < E) {
      const int cnt = seg_end[e] - (e == 0 ? 0 : seg_end[e - 1]);
      padded = (cnt + block_size - 1) / block_size * block_size;
    }
    int total;
    const int first = base + pm::block_exclusive_scan(padded, wt, &total);
    if (e < E) {
      pstart[e] = first;
      for (int b = first / block_size; b < (first + padded) / block_size; ++b) expert_ids[b] = e;
    }
    base += total;
  }
  if (threadIdx.x == 0) *num_post_pad = base;
}

// Row i of the tight layout (expert e) goes to pstart[e] + (i - start of e).
__global__ void align_scatter_kernel(const int32_t* __restrict__ seg_end, int E,
                                     const int32_t* __restrict__ row_to_route,
                                     const int32_t* __restrict__ pstart,
                                     int32_t* __restrict__ sorted_ids) {
  pdl_wait();
  const int n = seg_end[E - 1];
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    int lo = 0, hi = E - 1;  // first expert whose segment ends past i
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (seg_end[mid] > i) hi = mid; else lo = mid + 1;
    }
    const int start = lo == 0 ? 0 : seg_end[lo - 1];
    sorted_ids[pstart[lo] + (i - start)] = row_to_route[i];
  }
}

// seg_end[e] = number of rows whose id is <= e, for ids grouped in ascending
// expert order (the per_row layout): an upper-bound search per expert.
__global__ void ids_to_seg_end_kernel(const int32_t* __restrict__ ids, int M, int E,
                                      int32_t* __restrict__ seg_end) {
  pdl_wait();
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
    int lo = 0, hi = M;  // first row whose id exceeds e
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (ids[mid] <= e) lo = mid + 1; else hi = mid;
    }
    seg_end[e] = lo;
  }
}

__global__ void fill_i32_kernel(int32_t* __restrict__ p, int32_t v, int n) {
  pdl_wait();  // the buffer may still be read by the previous launch
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = v;
}

}  // namespace

cudaError_t launch_permute_align(const int32_t* ids, int T, int K, int E, int block_size,
                                 int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_pad,
                                 int32_t* seg_end, int32_t* row_to_route, int32_t* route_to_row,
                                 int32_t* pstart, void* ws, cudaStream_t s) {
  const int M = T * K;
  const long long L = (long long)M + (long long)(E + 1) * (block_size - 1);
  const int nb = (int)((L + block_size - 1) / block_size);
  cudaError_t e = launch_permute(nullptr, 4, ids, T, 0, E, K, nullptr, seg_end, row_to_route,
                                 route_to_row, ws, s);
  if (e != cudaSuccess) return e;
  const int fill_grid = (int)std::min<long long>((L + 255) / 256, (long long)num_sms() * 4);
  launch_pdl(align_fill_kernel, std::max(fill_grid, 1), 256, 0, s, sorted_ids, L, (int32_t)M,
             expert_ids, nb);
  launch_pdl(align_scan_kernel, 1, 1024, 0, s, (const int32_t*)seg_end, E, block_size, pstart,
             expert_ids, num_post_pad);
  const int sc_grid = std::max(1, std::min((M + 255) / 256, num_sms() * 4));
  launch_pdl(align_scatter_kernel, sc_grid, 256, 0, s, (const int32_t*)seg_end, E,
             (const int32_t*)row_to_route, (const int32_t*)pstart, sorted_ids);
  count_launch(3);
  return cudaGetLastError();
}

cudaError_t launch_ids_to_seg_end(const int32_t* ids, int M, int E, int32_t* seg_end,
                                  cudaStream_t s) {
  launch_pdl(ids_to_seg_end_kernel, (E + 255) / 256, 256, 0, s, ids, M, E, seg_end);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_fill_i32(int32_t* p, int32_t v, int n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  launch_pdl(fill_i32_kernel, (n + 255) / 256, 256, 0, s, p, v, n);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  if (bytes % 16 || (uintptr_t)src % 16 || (uintptr_t)dst % 16) return cudaErrorInvalidValue;
  copy16_kernel<<<num_sms(), 256, 0, s>>>(static_cast<const int4*>(src), static_cast<int4*>(dst),
                                          (long long)(bytes / 16));
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_permute(const void* hidden, int esz, const int32_t* ids, int T, int H, int E,
                           int K, void* expert_input, int32_t* seg_end, int32_t* row_to_route,
                           int32_t* route_to_row, void* ws, cudaStream_t s) {
  const int M = T * K;
  PermuteWs L(M, E);
  char* w = static_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(w);
  int* counts = reinterpret_cast<int*>(w + L.counts);
  int* active = reinterpret_cast<int*>(w + L.active);
  int* num_active = reinterpret_cast<int*>(w + L.num_active);
  if (M == 0) {
    cudaMemsetAsync(seg_end, 0, (size_t)E * 4, s);
    cudaMemsetAsync(num_active, 0, 4, s);
    return cudaGetLastError();
  }
  const int C = (M + kPermuteChunk - 1) / kPermuteChunk;
  const size_t hist_smem = (size_t)E * 4;
  launch_pdl(perm_count, C, 256, hist_smem, s, ids, M, E, counts, status);
  launch_pdl(perm_scan, 1, 1024, 0, s, counts, C, E, seg_end, active, num_active);
  // one CTA of W warps per chunk while W x E counts fit in 96 KB of shared
  // memory; otherwise one warp per chunk
  int W = 32;
  while (W > 1 && (size_t)W * E * 4 > 96 * 1024) W >>= 1;
  if (W >= 4) {
    const size_t sm = (size_t)W * E * 4;
    set_smem_limit((const void*)perm_scatter_cta, 96 * 1024);
    launch_pdl(perm_scatter_cta, C, W * 32, sm, s, ids, M, E, counts, row_to_route, route_to_row);
  } else {
    launch_pdl(perm_scatter, C, 32, hist_smem, s, ids, M, E, counts, row_to_route, route_to_row);
  }
  count_launch(3);
  if (expert_input)
    return launch_permute_gather(hidden, esz, T, H, E, K, seg_end, row_to_route, expert_input, ws,
                                 s);
  return cudaGetLastError();
}

cudaError_t launch_permute_gather(const void* hidden, int esz, int T, int H, int E, int K,
                                  const int32_t* seg_end, const int32_t* row_to_route,
                                  void* expert_input, void* ws, cudaStream_t s) {
  const int M = T * K;
  if (M == 0) return cudaSuccess;
  int* status = static_cast<int*>(ws);
  const size_t row_bytes = (size_t)H * esz;
  const int rows_per_block = 8;
  dim3 grid((M + rows_per_block - 1) / rows_per_block);
  const bool vec = (row_bytes % 16 == 0) && ((uintptr_t)hidden % 16 == 0) &&
                   ((uintptr_t)expert_input % 16 == 0);
  if (vec)
    launch_pdl(perm_gather<16>, grid, 256, 0, s, static_cast<const char*>(hidden), row_to_route,
               seg_end, E, K, T, row_bytes, static_cast<char*>(expert_input), status);
  else
    launch_pdl(perm_gather<2>, grid, 256, 0, s, static_cast<const char*>(hidden), row_to_route,
               seg_end, E, K, T, row_bytes, static_cast<char*>(expert_input), status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* y, const float* w, const int32_t* r2r, int T, int K, int H,
                           moe_dtype dt, float scale, void* out, cudaStream_t s,
                           const float* token_scale) {
  if (T == 0 || H == 0) return cudaSuccess;
  const int M = T * K;
  const bool aligned = ((uintptr_t)y % 16 == 0) && ((uintptr_t)out % 16 == 0);
  // at most one resident round of CTAs (a grid-stride loop covers the rest)
  auto grid_for = [&](const void* kern, int vec) {
    const long long items = (long long)T * (H / vec);
    const long long cap = (long long)num_sms() * resident_ctas(kern, 256);
    return (unsigned)std::max<long long>(1, std::min<long long>(cap, (items + 255) / 256));
  };
  auto half_width = [&](auto tag) {
    using B = decltype(tag);
    if (aligned && H % 8 == 0)
      launch_pdl(combine_kernel<B, 8>, grid_for((const void*)combine_kernel<B, 8>, 8), 256, 0, s,
          static_cast<const B*>(y), w, r2r, T, K, H, M, scale, static_cast<B*>(out), token_scale);
    else
      launch_pdl(combine_kernel<B, 1>, grid_for((const void*)combine_kernel<B, 1>, 1), 256, 0, s,
          static_cast<const B*>(y), w, r2r, T, K, H, M, scale, static_cast<B*>(out), token_scale);
  };
  if (dt == MOE_BF16) {
    half_width(__nv_bfloat16{});
  } else if (dt == MOE_F16) {
    half_width(__half{});
  } else {
    if (aligned && H % 4 == 0)
      launch_pdl(combine_kernel<float, 4>, grid_for((const void*)combine_kernel<float, 4>, 4), 256,
          0, s, static_cast<const float*>(y), w, r2r, T, K, H, M, scale,
          static_cast<float*>(out), token_scale);
    else
      launch_pdl(combine_kernel<float, 1>, grid_for((const void*)combine_kernel<float, 1>, 1), 256,
          0, s, static_cast<const float*>(y), w, r2r, T, K, H, M, scale,
          static_cast<float*>(out), token_scale);
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
