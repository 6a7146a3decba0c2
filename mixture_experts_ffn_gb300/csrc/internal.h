// Host-side declarations shared by the translation units of libmoe.so.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// device status-word bits (first int of every workspace)
enum : int {
  kDevBadIndex = 1,  // an id / index outside its range was met and skipped
  kDevTimeout = 2,   // a bounded wait ran out
};

constexpr int kPermuteChunk = 1024;  // routes per permute chunk
constexpr int kMaxExperts = 1024;    // router / grouped GEMM limit on E

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Permute scratch: [status 256 B][chunk counts C x E][active experts E][num_active 1]
struct PermuteWs {
  size_t counts, active, num_active, total;
  PermuteWs(int M, int E) {
    size_t C = (size_t)(M + kPermuteChunk - 1) / kPermuteChunk;
    if (C == 0) C = 1;
    counts = MOE_STATUS_BYTES;
    active = align256(counts + C * (size_t)E * 4);
    num_active = align256(active + (size_t)E * 4);
    total = align256(num_active + 4);
  }
};

// Full forward workspace: the permute scratch first (sharing the status word),
// then routing, index maps and the staged intermediates.
struct ForwardWs {
  size_t topk_w, topk_ids, seg_end, row_to_route, route_to_row, expert_input, act, y, total;
  ForwardWs(int T, int H, int F, int E, int K, int esz) {
    size_t M = (size_t)T * K;
    PermuteWs p((int)M, E);
    topk_w = p.total;
    topk_ids = align256(topk_w + M * 4);
    seg_end = align256(topk_ids + M * 4);
    row_to_route = align256(seg_end + (size_t)E * 4);
    route_to_row = align256(row_to_route + M * 4);
    expert_input = align256(route_to_row + M * 4);
    act = align256(expert_input + M * (size_t)H * esz);
    y = align256(act + M * (size_t)F * esz);
    total = align256(y + M * (size_t)H * esz);
  }
};

void count_launch(int n = 1);
int num_sms();
// CTAs of `kernel` that one SM of the current device holds at once with
// `threads` threads and `smem_bytes` of dynamic shared memory (an occupancy
// query, cached per device, kernel and shape); at least 1.
int resident_ctas(const void* kernel, int threads, int smem_bytes = 0);

// Raises the dynamic shared-memory limit of `kernel` to `bytes` on the
// current device, once per (device, kernel): the setting belongs to the
// device's context, so a second GPU needs its own call.  Thread-safe.
cudaError_t set_smem_limit(const void* kernel, int bytes);

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel of the stream is still finishing, runs whatever
// does not read earlier results (shared-memory set-up, barrier init, TMEM
// allocation), and executes griddepcontrol.wait (pdl_wait) before its first
// access to global memory written by earlier work on the stream.  Every kernel
// of the library does so, so launches stay ordered transitively.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- launchers (return cudaGetLastError() of their launches) ----
cudaError_t launch_route(const void* logits, const float* bias, const int32_t* ids_in, int T,
                         int E, const moe_route_params& p, float* w, int32_t* ids, void* probs,
                         float* wscale, cudaStream_t s);

// Router + permute index maps in one launch (bit-identical to launch_route
// then launch_permute without the gather); route_permute_ok(E) says whether
// E is within its limit (E <= 512).  Uses ws's permute scratch and three
// ints of its status area (grid-barrier counters that reset themselves).
bool route_permute_ok(int E);
// Test hook behind moe_test_force_wait_timeout; returns the previous state.
int set_wait_timeout_test(int enable, long long limit_ns);
cudaError_t launch_route_permute(const void* logits, const float* bias, const int32_t* ids_in,
                                 int T, int E, const moe_route_params& p, float* w, int32_t* ids,
                                 void* probs, float* wscale, int32_t* seg_end,
                                 int32_t* row_to_route, int32_t* route_to_row, void* ws,
                                 cudaStream_t s);

cudaError_t launch_permute(const void* hidden, int esz, const int32_t* ids, int T, int H, int E,
                           int K, void* expert_input, int32_t* seg_end, int32_t* row_to_route,
                           int32_t* route_to_row, void* ws, cudaStream_t s);
// The padded permute-align layout from topk_ids (tight maps in seg_end,
// row_to_route, route_to_row; padded starts in pstart [E]; ws as the permute's).
cudaError_t launch_permute_align(const int32_t* ids, int T, int K, int E, int block_size,
                                 int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_pad,
                                 int32_t* seg_end, int32_t* row_to_route, int32_t* route_to_row,
                                 int32_t* pstart, void* ws, cudaStream_t s);

// The gather step of launch_permute alone: expert_input[row] = hidden[row_to_route[row] / K]
// for the rows below seg_end[E-1], from maps already built (launch_route_permute).
cudaError_t launch_permute_gather(const void* hidden, int esz, int T, int H, int E, int K,
                                  const int32_t* seg_end, const int32_t* row_to_route,
                                  void* expert_input, void* ws, cudaStream_t s);

// dst[0, bytes) = src[0, bytes) by the SMs (16-byte aligned pointers and
// size; cudaErrorInvalidValue otherwise); src may be page-locked host memory
// mapped for the device.
cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, cudaStream_t s);

// seg_end [E] of a per_row layout (ids [M] grouped in ascending expert order).
cudaError_t launch_ids_to_seg_end(const int32_t* ids, int M, int E, int32_t* seg_end,
                                  cudaStream_t s);

// p[0, n) = v on the stream.
cudaError_t launch_fill_i32(int32_t* p, int32_t v, int n, cudaStream_t s);

// token_scale (optional, [T] f32) multiplies token t's sum as well
cudaError_t launch_combine(const void* y, const float* w, const int32_t* route_to_row, int T,
                           int K, int H, moe_dtype dt, float scale, void* out, cudaStream_t s,
                           const float* token_scale = nullptr);

cudaError_t launch_swiglu(const void* gate, const void* up, int64_t R, int I, moe_dtype dt,
                          int fusion, float limit, float alpha, float beta, void* out,
                          cudaStream_t s);

// SwiGLU fusion 0: the gate and up projections of a gated gate_up GEMM as two
// tensors, [E, F, K] each, with optional biases [E, F] each.  The launchers'
// w / bias then hold the gate projection and its bias.
struct SplitUp {
  const void* w_up;
  const void* b_up;
};

// SIMT grouped GEMM (exact fp32 FMA; any dtype).  act == nullptr: plain GEMM
// with N output columns; otherwise N = F act columns read from N1 rows.
cudaError_t launch_gemm_simt(const void* a, const void* w, const void* bias,
                             const int32_t* seg_end, int M, int N, int K, int E, moe_dtype dt,
                             const moe_act_params* act, void* out, int* status, cudaStream_t s,
                             int seg_stride = 0, const SplitUp* split = nullptr);

// tcgen05 grouped GEMM (bf16 operands, or float16 with f16, fp32 TMEM
// accumulators).  With
// gather_rows, row r of A is row gather_rows[r] / gather_div of `a` (the
// token-ordered hidden states, gather_src_rows rows, read through row_to_route
// so the permuted copy is never materialised); only rows inside their expert's
// segment are read.
cudaError_t launch_gemm_tc(const void* a, const void* w, const void* bias, const int32_t* seg_end,
                           int M, int N, int K, int E, const moe_act_params* act, void* out,
                           int* status, cudaStream_t s, const int32_t* gather_rows = nullptr,
                           int gather_div = 1, int gather_src_rows = 0, int seg_stride = 0,
                           const SplitUp* split = nullptr, bool f16 = false);

// The weights-as-M tcgen05 grouped GEMM on SM pairs (gemm_sw.cu): the same
// contract as launch_gemm_tc without split weights; N and K multiples of 8.
// wide: 256 weight rows per CTA (two M256 accumulators) instead of 128.
cudaError_t launch_gemm_sw(const void* a, const void* w, const void* bias, const int32_t* seg_end,
                           int M, int N, int K, int E, const moe_act_params* act, void* out,
                           int* status, cudaStream_t s, const int32_t* gather_rows,
                           int gather_div, int gather_src_rows, int seg_stride, bool f16,
                           bool wide);

// block-scaled FP8 grouped GEMM over a masked slab (e4m3 operands, fp32
// scales per row x 128 K of a and per 128 x 128 block of b, bf16 out)
cudaError_t launch_gemm_fp8(const void* a, const float* a_scale, const void* b,
                            const float* b_scale, const int32_t* counts, int E, int max_m, int N,
                            int K, void* out, int* status, cudaStream_t s);

// indexed per-route decode path (bf16, silu_and_mul, no bias)
cudaError_t launch_indexed(const void* hidden, const void* w1, const void* w2, const float* w,
                           const int32_t* ids, int T, int H, int F, int E, int K, float scale,
                           void* out, void* ws, const ForwardWs& L, cudaStream_t s,
                           bool maps_ready = false);

}  // namespace moe
