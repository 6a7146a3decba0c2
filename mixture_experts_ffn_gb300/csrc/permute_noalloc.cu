// moe_permute_noalloc: the permute of moe_permute for callers that cannot
// hand the library a workspace.
//
// Some callers cannot call cudaMalloc at the point where they run the layer:
// cudaMalloc and cudaFree can synchronise the whole device and so stall every
// other stream, and serving runtimes that fix their memory budget at start-up
// (or that own all device memory through their own allocator) forbid any
// allocation afterwards.  This entry point needs no workspace from the caller:
// its scratch (the status word and the per-chunk expert counts of the
// histogram/scan/scatter permute) lives in a fixed array in device memory that
// belongs to the library and is held by every GPU that loads the library until
// the process exits.  The caller still passes every input and output buffer.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace moe {
namespace {

// Fixed scratch: 1 MiB.  Enough for M = T*K up to 131072 routes with E up to
// 1024 experts (the permute scratch is 256 B + ceil(M/1024) * E * 4 B + E * 4 B).
constexpr size_t kNoAllocScratchBytes = 1u << 20;
static __device__ __align__(256) unsigned char g_permute_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device.  In host code
// the array's name only stands for the symbol: its device address has to be
// asked for, once per device, with that device current.
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool spans_overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_permute_noalloc(const void* hidden, moe_dtype dtype,
                                          const int32_t* topk_ids, int T, int H, int E, int K,
                                          void* expert_input, int32_t* seg_end,
                                          int32_t* row_to_route, int32_t* route_to_row,
                                          cudaStream_t stream) {
  if (T < 0 || K < 1 || E < 1 || E > 12288 || (dtype != MOE_F32 && dtype != MOE_BF16 && dtype != MOE_F16))
    return MOE_ERR_INVALID_ARG;
  if ((long long)T * K >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
  if (expert_input && (!hidden || H < 1)) return MOE_ERR_INVALID_ARG;
  if (!seg_end || (T > 0 && (!topk_ids || !row_to_route || !route_to_row)))
    return MOE_ERR_INVALID_ARG;
  const int M = T * K;
  if (PermuteWs(M, E).total > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;
  const size_t esz = dtype == MOE_F32 ? 4 : 2;
  const void* outs[4] = {expert_input, seg_end, row_to_route, route_to_row};
  const size_t out_n[4] = {expert_input ? (size_t)M * H * esz : 0, (size_t)E * 4, (size_t)M * 4,
                           (size_t)M * 4};
  const void* ins[2] = {hidden, topk_ids};
  const size_t in_n[2] = {expert_input ? (size_t)T * H * esz : 0, (size_t)M * 4};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 2; ++j)
      if (spans_overlap(outs[i], out_n[i], ins[j], in_n[j])) return MOE_ERR_OVERLAP;
    for (int j = i + 1; j < 4; ++j)
      if (spans_overlap(outs[i], out_n[i], outs[j], out_n[j])) return MOE_ERR_OVERLAP;
  }
  void* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  // The status word is the only part of the scratch that must start at zero
  // (kernels OR error bits into it); the counts are fully rewritten every call.
  if (cudaMemsetAsync(scratch, 0, MOE_STATUS_BYTES, stream) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_permute(hidden, (int)esz, topk_ids, T, H, E, K, expert_input, seg_end,
                        row_to_route, route_to_row, scratch, stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
