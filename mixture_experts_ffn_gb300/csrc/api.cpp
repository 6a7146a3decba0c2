// C ABI of libmoe.so: argument validation, overlap checks, workspace layout and
// dispatch to the kernels.  Every check runs on the host before any launch, so
// an invalid call writes nothing.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>
#include <set>
#include <string>
#include <vector>
#include <utility>

#include "internal.h"

namespace moe {

static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

int resident_ctas(const void* kernel, int threads, int smem_bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int, int>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(dev, kernel, threads, smem_bytes);
  const auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem_bytes) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    n = 1;
  }
  n = n < 1 ? 1 : n;
  cache[key] = n;
  return n;
}

cudaError_t set_smem_limit(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(dev, kernel);
  if (done.count(key)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert(key);
  return e;
}

static int g_force_simt = 0;

// ---------------------------------------------------------------- stage profile
// With MOE_PROFILE=1 in the environment (read once), the forward brackets each
// of its stages with a pair of CUDA events on the caller's stream;
// moe_profile_report synchronises them and returns per-stage totals.  The
// events sit between the launches, so a profiled forward loses the overlap of
// one launch's start with the previous one's end.
namespace {
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
std::vector<ProfRec> g_prof;

bool profiling() {
  static const bool on = [] {
    const char* v = getenv("MOE_PROFILE");
    return v && v[0] == '1';
  }();
  return on;
}

// Brackets the launches of one stage between its construction and done().
struct StageTimer {
  const char* name;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  StageTimer(const char* n, cudaStream_t st) : name(n), s(st) {
    if (!profiling()) return;
    if (cudaEventCreate(&a) != cudaSuccess || cudaEventRecord(a, s) != cudaSuccess) a = nullptr;
  }
  void done() {
    if (!a) return;
    cudaEvent_t b = nullptr;
    if (cudaEventCreate(&b) != cudaSuccess || cudaEventRecord(b, s) != cudaSuccess) {
      cudaEventDestroy(a);
      if (b) cudaEventDestroy(b);
      a = nullptr;
      return;
    }
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof.push_back({name, a, b});
    a = nullptr;
  }
  ~StageTimer() {
    if (a) cudaEventDestroy(a);
  }
};
}  // namespace

namespace {

struct Span {
  const void* p;
  size_t bytes;
};
bool overlaps(Span a, Span b) {
  if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
  uintptr_t a0 = (uintptr_t)a.p, a1 = a0 + a.bytes;
  uintptr_t b0 = (uintptr_t)b.p, b1 = b0 + b.bytes;
  return a0 < b1 && b0 < a1;
}
// any output overlapping any input, or two outputs overlapping each other
template <size_t NO, size_t NI>
bool any_overlap(const Span (&outs)[NO], const Span (&ins)[NI]) {
  for (size_t i = 0; i < NO; ++i) {
    for (size_t j = 0; j < NI; ++j)
      if (overlaps(outs[i], ins[j])) return true;
    for (size_t j = i + 1; j < NO; ++j)
      if (overlaps(outs[i], outs[j])) return true;
  }
  return false;
}

size_t esize(moe_dtype d) { return d == MOE_F32 ? 4 : 2; }
bool dtype_ok(int d) { return d == MOE_F32 || d == MOE_BF16 || d == MOE_F16; }
// bytes of one logit / router_probs element (the MoERouter type T)
size_t rsz(const moe_route_params* p) { return esize((moe_dtype)p->dtype); }

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

moe_status check_route(const void* logits, const float* bias, int T, int E,
                       const moe_route_params* p, const float* w, const int32_t* ids,
                       const void* probs, const float* wscale) {
  if (!p || T < 0 || E < 1 || E > kMaxExperts || !dtype_ok(p->dtype)) return MOE_ERR_INVALID_ARG;
  const int K = p->top_k, G = p->num_expert_group, TG = p->topk_group;
  if (K < 1 || K > E || K > 64) return MOE_ERR_INVALID_ARG;
  if (p->scoring != MOE_SCORING_SOFTMAX && p->scoring != MOE_SCORING_SIGMOID &&
      p->scoring != MOE_SCORING_SQRT_SOFTPLUS)
    return MOE_ERR_INVALID_ARG;
  if (bias && p->scoring == MOE_SCORING_SOFTMAX) return MOE_ERR_INVALID_ARG;
  if (G < 1 || G > 32 || E % G != 0) return MOE_ERR_INVALID_ARG;
  if (TG < 1 || TG > G || (long long)TG * (E / G) < K) return MOE_ERR_INVALID_ARG;
  if (bias && G > 1 && E / G < 2) return MOE_ERR_INVALID_ARG;
  if (!(p->routed_scaling_factor > 0.f) || !std::isfinite(p->routed_scaling_factor))
    return MOE_ERR_INVALID_ARG;
  if (p->local_expert_count < 0) return MOE_ERR_INVALID_ARG;
  if (p->local_expert_count > 0) {
    if (p->local_expert_start < 0 || p->local_expert_start + p->local_expert_count > E)
      return MOE_ERR_INVALID_ARG;
    if (!probs || !wscale) return MOE_ERR_INVALID_ARG;
  } else if (probs || wscale) {
    return MOE_ERR_INVALID_ARG;
  }
  if (T > 0 && (!logits || !w || !ids)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// the gated kinds read 2F gate_up rows, the others F
bool gated_kind(int k) {
  return k == MOE_ACT_SILU_AND_MUL || k == MOE_ACT_SWIGLU || k == MOE_ACT_GELU_AND_MUL;
}

bool act_ok(const moe_act_params* a) {
  if (!a) return false;
  if (a->kind == MOE_ACT_SWIGLU) return a->swiglu_fusion == 1 || a->swiglu_fusion == 2;
  return a->kind >= MOE_ACT_SILU_AND_MUL && a->kind <= MOE_ACT_SILU;
}

// SwiGLU fusion 0 (gate and up projections in two tensors): a gated kind, with
// swiglu_fusion 0 for the clamped SwiGLU.  The launchers get a copy marked
// stacked, the layout whose accumulator they share.
bool split_act(const moe_act_params* a, moe_act_params* stacked) {
  if (!a || !gated_kind(a->kind)) return false;
  if (a->kind == MOE_ACT_SWIGLU && a->swiglu_fusion != 0) return false;
  *stacked = *a;
  stacked->swiglu_fusion = 2;
  return true;
}

bool ws_ok(const void* ws, size_t have, size_t need) {
  return ws && ((uintptr_t)ws & 255u) == 0 && have >= need;
}

bool tc_ok(const void* a, const void* w, const void* out, int Nout, int Kd, int M) {
  return !g_force_simt && Nout % 8 == 0 && Kd % 8 == 0 && aligned16(a) && aligned16(w) &&
         aligned16(out) && M < (1 << 30);
}

// grouped GEMM dispatch; act == nullptr for the plain (down) GEMM
cudaError_t grouped_gemm(const void* a, const void* w, const void* bias, const int32_t* seg_end,
                         int M, int Nout, int Kd, int E, moe_dtype dt, const moe_act_params* act,
                         void* out, int* status, cudaStream_t s, int seg_stride = 0,
                         const SplitUp* split = nullptr) {
  if (dt != MOE_F32 && tc_ok(a, w, out, Nout, Kd, M) && (!split || aligned16(split->w_up)))
    return launch_gemm_tc(a, w, bias, seg_end, M, Nout, Kd, E, act, out, status, s, nullptr, 1, 0,
                          seg_stride, split, dt == MOE_F16);
  return launch_gemm_simt(a, w, bias, seg_end, M, Nout, Kd, E, dt, act, out, status, s,
                          seg_stride, split);
}

bool indexed_rule(int T, int H, int F, int E, int K, moe_dtype dt, const moe_act_params* act,
                  const void* b1, const void* b2, const void* hidden, const void* w1,
                  const void* w2) {
  return (long long)T * K <= 2LL * E && act->kind == MOE_ACT_SILU_AND_MUL && !b1 && !b2 &&
         dt == MOE_BF16 && H % 128 == 0 && F % 256 == 0 && aligned16(hidden) &&
         aligned16(w1) && aligned16(w2);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_route(const void* logits, const float* correction_bias, const int32_t* expert_ids,
                     int T, int E, const moe_route_params* p, float* topk_weights,
                     int32_t* topk_ids, void* router_probs, float* weight_scale,
                     cudaStream_t stream) {
  moe_status st = check_route(logits, correction_bias, T, E, p, topk_weights, topk_ids,
                              router_probs, weight_scale);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  const size_t TK = (size_t)T * p->top_k, lc = (size_t)p->local_expert_count;
  Span outs[] = {{topk_weights, TK * 4}, {topk_ids, TK * 4}, {router_probs, T * lc * rsz(p)},
                 {weight_scale, (size_t)T * 4}};
  Span ins[] = {{logits, (size_t)T * E * rsz(p)}, {correction_bias, (size_t)E * 4},
                {expert_ids, TK * 4}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  return cuda_status(launch_route(logits, correction_bias, expert_ids, T, E, *p, topk_weights,
                                  topk_ids, router_probs, weight_scale, stream));
}

moe_status moe_route_permute(const void* logits, const float* correction_bias,
                             const int32_t* expert_ids, int T, int E, const moe_route_params* p,
                             float* topk_weights, int32_t* topk_ids, void* router_probs,
                             float* weight_scale, int32_t* seg_end, int32_t* row_to_route,
                             int32_t* route_to_row, void* ws, size_t ws_bytes,
                             cudaStream_t stream) {
  moe_status st = check_route(logits, correction_bias, T, E, p, topk_weights, topk_ids,
                              router_probs, weight_scale);
  if (st != MOE_OK) return st;
  const long long TKl = (long long)T * p->top_k;
  if (TKl >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
  if (!seg_end || (T > 0 && (!row_to_route || !route_to_row))) return MOE_ERR_INVALID_ARG;
  if (!route_permute_ok(E)) return MOE_ERR_UNSUPPORTED;
  const int M = (int)TKl;
  if (!ws_ok(ws, ws_bytes, PermuteWs(M, E).total)) return MOE_ERR_WORKSPACE;
  const size_t TK = (size_t)M, lc = (size_t)p->local_expert_count;
  Span outs[] = {{topk_weights, TK * 4}, {topk_ids, TK * 4}, {router_probs, T * lc * rsz(p)},
                 {weight_scale, (size_t)T * 4}, {seg_end, (size_t)E * 4},
                 {row_to_route, TK * 4}, {route_to_row, TK * 4}, {ws, PermuteWs(M, E).total}};
  Span ins[] = {{logits, (size_t)T * E * rsz(p)}, {correction_bias, (size_t)E * 4},
                {expert_ids, TK * 4}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  if (T == 0) return cuda_status(cudaMemsetAsync(seg_end, 0, (size_t)E * 4, stream));
  return cuda_status(launch_route_permute(logits, correction_bias, expert_ids, T, E, *p,
                                          topk_weights, topk_ids, router_probs, weight_scale,
                                          seg_end, row_to_route, route_to_row, ws, stream));
}

size_t moe_permute_workspace_size(int M, int E) {
  if (M < 0 || E < 1) return 0;
  return PermuteWs(M, E).total;
}

moe_status moe_permute(const void* hidden, moe_dtype dtype, const int32_t* topk_ids, int T, int H,
                       int E, int K, void* expert_input, int32_t* seg_end, int32_t* row_to_route,
                       int32_t* route_to_row, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (T < 0 || K < 1 || E < 1 || E > 12288 || !dtype_ok(dtype)) return MOE_ERR_INVALID_ARG;
  if ((long long)T * K >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
  if (expert_input && (!hidden || H < 1)) return MOE_ERR_INVALID_ARG;
  if (!seg_end || (T > 0 && (!topk_ids || !row_to_route || !route_to_row)))
    return MOE_ERR_INVALID_ARG;
  const int M = T * K;
  if (!ws_ok(ws, ws_bytes, PermuteWs(M, E).total)) return MOE_ERR_WORKSPACE;
  const size_t esz = esize(dtype);
  Span outs[] = {{expert_input, expert_input ? (size_t)M * H * esz : 0},
                 {seg_end, (size_t)E * 4},
                 {row_to_route, (size_t)M * 4},
                 {route_to_row, (size_t)M * 4},
                 {ws, PermuteWs(M, E).total}};
  Span ins[] = {{hidden, expert_input ? (size_t)T * H * esz : 0}, {topk_ids, (size_t)M * 4}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  return cuda_status(launch_permute(hidden, (int)esz, topk_ids, T, H, E, K, expert_input, seg_end,
                                    row_to_route, route_to_row, ws, stream));
}

namespace {
// permute-align scratch: the permute's, then the tight maps and padded starts
struct AlignWs {
  size_t seg_end, r2r, route_to_row, pstart, total;
  AlignWs(int M, int E) {
    const size_t base = PermuteWs(M, E).total;
    seg_end = base;
    r2r = align256(seg_end + (size_t)E * 4);
    route_to_row = align256(r2r + (size_t)M * 4);
    pstart = align256(route_to_row + (size_t)M * 4);
    total = align256(pstart + (size_t)E * 4);
  }
};
}  // namespace

size_t moe_permute_align_workspace_size(int T, int K, int E) {
  if (T < 0 || K < 1 || E < 1) return 0;
  return AlignWs(T * K, E).total;
}

moe_status moe_permute_align(const int32_t* topk_ids, int T, int K, int E, int block_size,
                             int32_t* sorted_token_ids, int32_t* expert_ids,
                             int32_t* num_tokens_post_pad, void* ws, size_t ws_bytes,
                             cudaStream_t stream) {
  if (T < 0 || K < 1 || E < 1 || E > 12288 || block_size < 1 || block_size > (1 << 20))
    return MOE_ERR_INVALID_ARG;
  const long long L = (long long)T * K + (long long)(E + 1) * (block_size - 1);
  if (L >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
  if (!sorted_token_ids || !expert_ids || !num_tokens_post_pad || (T > 0 && !topk_ids))
    return MOE_ERR_INVALID_ARG;
  const int M = T * K;
  AlignWs A(M, E);
  if (!ws_ok(ws, ws_bytes, A.total)) return MOE_ERR_WORKSPACE;
  const size_t nb = (size_t)((L + block_size - 1) / block_size);
  Span outs[] = {{sorted_token_ids, (size_t)L * 4}, {expert_ids, nb * 4},
                 {num_tokens_post_pad, 4}, {ws, A.total}};
  Span ins[] = {{topk_ids, (size_t)M * 4}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  char* base = static_cast<char*>(ws);
  return cuda_status(launch_permute_align(
      topk_ids, T, K, E, block_size, sorted_token_ids, expert_ids, num_tokens_post_pad,
      reinterpret_cast<int32_t*>(base + A.seg_end), reinterpret_cast<int32_t*>(base + A.r2r),
      reinterpret_cast<int32_t*>(base + A.route_to_row),
      reinterpret_cast<int32_t*>(base + A.pstart), ws, stream));
}

moe_status moe_permute_gather(const void* hidden, moe_dtype dtype, const int32_t* seg_end,
                              const int32_t* row_to_route, int T, int H, int E, int K,
                              void* expert_input, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (T < 0 || H < 1 || K < 1 || E < 1 || !dtype_ok(dtype)) return MOE_ERR_INVALID_ARG;
  if ((long long)T * K >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
  if (!seg_end || (T > 0 && (!hidden || !row_to_route || !expert_input)))
    return MOE_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, MOE_STATUS_BYTES)) return MOE_ERR_WORKSPACE;
  const int M = T * K;
  const size_t esz = esize(dtype);
  Span outs[] = {{expert_input, (size_t)M * H * esz}};
  Span ins[] = {{hidden, (size_t)T * H * esz}, {seg_end, (size_t)E * 4},
                {row_to_route, (size_t)M * 4}, {ws, MOE_STATUS_BYTES}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  if (M == 0) return MOE_OK;
  return cuda_status(launch_permute_gather(hidden, (int)esz, T, H, E, K, seg_end, row_to_route,
                                           expert_input, ws, stream));
}

moe_status moe_grouped_gemm_fp8_masked(const void* a, const float* a_scale, const void* b,
                                       const float* b_scale, const int32_t* layout_metadata,
                                       int E, int max_m, int N, int K, void* out, void* ws,
                                       size_t ws_bytes, cudaStream_t stream) {
  if (E < 1 || E > kMaxExperts || max_m < 0 || N < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (K % 128 || N % 128) return MOE_ERR_INVALID_ARG;  // scale blocks of 128
  if ((long long)E * max_m >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
  if (!layout_metadata || (max_m > 0 && (!a || !a_scale || !b || !b_scale || !out)))
    return MOE_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, MOE_STATUS_BYTES)) return MOE_ERR_WORKSPACE;
  if (max_m > 0 && (!aligned16(a) || !aligned16(b) || ((uintptr_t)a_scale & 3) ||
                    ((uintptr_t)b_scale & 3) || ((uintptr_t)out & 1)))
    return MOE_ERR_UNSUPPORTED;
  const size_t nkb = (size_t)K / 128, rows = (size_t)E * max_m;
  Span outs[] = {{out, rows * N * 2}};
  Span ins[] = {{a, rows * K}, {a_scale, rows * nkb * 4}, {b, (size_t)E * N * K},
                {b_scale, (size_t)E * (N / 128) * nkb * 4}, {layout_metadata, (size_t)E * 4},
                {ws, MOE_STATUS_BYTES}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  if (max_m == 0) return MOE_OK;
  return cuda_status(launch_gemm_fp8(a, a_scale, b, b_scale, layout_metadata, E, max_m, N, K, out,
                                     static_cast<int*>(ws), stream));
}

size_t moe_grouped_gemm_workspace_size(int layout, int rows, int E) {
  if (rows < 0 || E < 1) return 0;
  if (layout == MOE_LAYOUT_PER_ROW) return MOE_STATUS_BYTES + align256((size_t)E * 4);
  return MOE_STATUS_BYTES;
}

moe_status moe_grouped_gemm(const void* a, const void* w, const void* bias, int layout,
                            const int32_t* layout_metadata, int rows, int N, int K, int E,
                            moe_dtype dtype, const moe_act_params* act, void* out, void* ws,
                            size_t ws_bytes, cudaStream_t stream) {
  if (rows < 0 || N < 1 || K < 1 || E < 1 || E > kMaxExperts || !dtype_ok(dtype))
    return MOE_ERR_INVALID_ARG;
  if (layout < MOE_LAYOUT_PSUM || layout > MOE_LAYOUT_MASKED) return MOE_ERR_INVALID_ARG;
  if (act && !act_ok(act)) return MOE_ERR_INVALID_ARG;
  const bool masked = layout == MOE_LAYOUT_MASKED;
  const long long M = masked ? (long long)E * rows : rows;
  if (M >= (1LL << 30)) return MOE_ERR_INVALID_ARG;
  if (!w || !layout_metadata || (M > 0 && (!a || !out))) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_grouped_gemm_workspace_size(layout, rows, E);
  if (!ws_ok(ws, ws_bytes, need)) return MOE_ERR_WORKSPACE;
  const size_t esz = esize(dtype);
  const size_t N1 = act && gated_kind(act->kind) ? 2 * (size_t)N : (size_t)N;
  const size_t meta_n = layout == MOE_LAYOUT_PER_ROW ? (size_t)M : (size_t)E;
  Span outs[] = {{out, (size_t)M * N * esz}, {ws, need}};
  Span ins[] = {{a, (size_t)M * K * esz}, {w, (size_t)E * N1 * K * esz},
                {bias, bias ? (size_t)E * N1 * esz : 0}, {layout_metadata, meta_n * 4}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  if (M == 0) return MOE_OK;
  int* status = static_cast<int*>(ws);
  const int32_t* seg = layout_metadata;
  if (layout == MOE_LAYOUT_PER_ROW) {
    int32_t* seg_end = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + MOE_STATUS_BYTES);
    if (launch_ids_to_seg_end(layout_metadata, (int)M, E, seg_end, stream) != cudaSuccess)
      return MOE_ERR_CUDA;
    seg = seg_end;
  }
  return cuda_status(grouped_gemm(a, w, bias, seg, (int)M, N, K, E, dtype, act, out, status,
                                  stream, masked ? rows : 0));
}

moe_status moe_grouped_gemm_act(const void* a, const void* w_gate_up, const void* b_gate_up,
                                const int32_t* seg_end, int M, int F, int Hk, int E,
                                moe_dtype dtype, const moe_act_params* act, void* out, void* ws,
                                size_t ws_bytes, cudaStream_t stream) {
  if (M < 0 || F < 1 || Hk < 1 || E < 1 || E > kMaxExperts || !dtype_ok(dtype) || !act_ok(act))
    return MOE_ERR_INVALID_ARG;
  if (!seg_end || !w_gate_up || (M > 0 && (!a || !out))) return MOE_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, MOE_STATUS_BYTES)) return MOE_ERR_WORKSPACE;
  const size_t esz = esize(dtype);
  const size_t N1 = gated_kind(act->kind) ? 2 * (size_t)F : (size_t)F;
  Span outs[] = {{out, (size_t)M * F * esz}};
  Span ins[] = {{a, (size_t)M * Hk * esz}, {w_gate_up, (size_t)E * N1 * Hk * esz},
                {b_gate_up, b_gate_up ? (size_t)E * N1 * esz : 0}, {seg_end, (size_t)E * 4},
                {ws, MOE_STATUS_BYTES}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  if (M == 0) return MOE_OK;
  return cuda_status(grouped_gemm(a, w_gate_up, b_gate_up, seg_end, M, F, Hk, E, dtype, act, out,
                                  static_cast<int*>(ws), stream));
}

moe_status moe_grouped_gemm_act_split(const void* a, const void* w_gate, const void* w_up,
                                      const void* b_gate, const void* b_up,
                                      const int32_t* seg_end, int M, int F, int Hk, int E,
                                      moe_dtype dtype, const moe_act_params* act, void* out,
                                      void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_act_params st{};
  if (M < 0 || F < 1 || Hk < 1 || E < 1 || E > kMaxExperts || !dtype_ok(dtype) ||
      !split_act(act, &st))
    return MOE_ERR_INVALID_ARG;
  if (!seg_end || !w_gate || !w_up || (M > 0 && (!a || !out)) || (!b_gate != !b_up))
    return MOE_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, MOE_STATUS_BYTES)) return MOE_ERR_WORKSPACE;
  const size_t esz = esize(dtype);
  const size_t wn = (size_t)E * F * Hk * esz, bn = b_gate ? (size_t)E * F * esz : 0;
  Span outs[] = {{out, (size_t)M * F * esz}};
  Span ins[] = {{a, (size_t)M * Hk * esz}, {w_gate, wn}, {w_up, wn}, {b_gate, bn}, {b_up, bn},
                {seg_end, (size_t)E * 4}, {ws, MOE_STATUS_BYTES}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  if (M == 0) return MOE_OK;
  const SplitUp split{w_up, b_up};
  return cuda_status(grouped_gemm(a, w_gate, b_gate, seg_end, M, F, Hk, E, dtype, &st, out,
                                  static_cast<int*>(ws), stream, 0, &split));
}

moe_status moe_grouped_gemm_act_gathered(const void* hidden, int T, const int32_t* row_to_route,
                                         int top_k, const void* w_gate_up,
                                         const void* b_gate_up, const int32_t* seg_end, int M,
                                         int F, int H, int E, moe_dtype dtype,
                                         const moe_act_params* act, void* out, void* ws,
                                         size_t ws_bytes, cudaStream_t stream) {
  if (T < 0 || top_k < 1 || M < 0 || F < 1 || H < 1 || E < 1 || E > kMaxExperts ||
      !dtype_ok(dtype) || !act_ok(act))
    return MOE_ERR_INVALID_ARG;
  if ((long long)T * top_k >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
  if (!seg_end || !w_gate_up || (M > 0 && (!hidden || !row_to_route || !out)))
    return MOE_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, MOE_STATUS_BYTES)) return MOE_ERR_WORKSPACE;
  const size_t N1 = gated_kind(act->kind) ? 2 * (size_t)F : (size_t)F;
  Span outs[] = {{out, (size_t)M * F * 2}};
  Span ins[] = {{hidden, (size_t)T * H * 2}, {row_to_route, (size_t)M * 4},
                {w_gate_up, (size_t)E * N1 * H * 2}, {b_gate_up, b_gate_up ? (size_t)E * N1 * 2 : 0},
                {seg_end, (size_t)E * 4}, {ws, MOE_STATUS_BYTES}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  if (dtype == MOE_F32 || !tc_ok(hidden, w_gate_up, out, F, H, M))
    return MOE_ERR_UNSUPPORTED;
  if (M == 0) return MOE_OK;
  return cuda_status(launch_gemm_tc(hidden, w_gate_up, b_gate_up, seg_end, M, F, H, E, act, out,
                                    static_cast<int*>(ws), stream, row_to_route, top_k, T, 0,
                                    nullptr, dtype == MOE_F16));
}

moe_status moe_grouped_gemm_down(const void* a, const void* w_down, const void* b_down,
                                 const int32_t* seg_end, int M, int H, int F, int E,
                                 moe_dtype dtype, void* out, void* ws, size_t ws_bytes,
                                 cudaStream_t stream) {
  if (M < 0 || H < 1 || F < 1 || E < 1 || E > kMaxExperts || !dtype_ok(dtype))
    return MOE_ERR_INVALID_ARG;
  if (!seg_end || !w_down || (M > 0 && (!a || !out))) return MOE_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, MOE_STATUS_BYTES)) return MOE_ERR_WORKSPACE;
  const size_t esz = esize(dtype);
  Span outs[] = {{out, (size_t)M * H * esz}};
  Span ins[] = {{a, (size_t)M * F * esz}, {w_down, (size_t)E * H * F * esz},
                {b_down, b_down ? (size_t)E * H * esz : 0}, {seg_end, (size_t)E * 4},
                {ws, MOE_STATUS_BYTES}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  if (M == 0) return MOE_OK;
  return cuda_status(grouped_gemm(a, w_down, b_down, seg_end, M, H, F, E, dtype, nullptr, out,
                                  static_cast<int*>(ws), stream));
}

moe_status moe_combine(const void* expert_out, const float* topk_weights,
                       const int32_t* route_to_row, int T, int K, int H, moe_dtype dtype,
                       float scale, void* out, cudaStream_t stream) {
  if (T < 0 || K < 1 || H < 1 || !dtype_ok(dtype) || !std::isfinite(scale))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!expert_out || !topk_weights || !route_to_row || !out)) return MOE_ERR_INVALID_ARG;
  const size_t esz = esize(dtype), M = (size_t)T * K;
  Span outs[] = {{out, (size_t)T * H * esz}};
  Span ins[] = {{expert_out, M * H * esz}, {topk_weights, M * 4}, {route_to_row, M * 4}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  return cuda_status(
      launch_combine(expert_out, topk_weights, route_to_row, T, K, H, dtype, scale, out, stream));
}

moe_status swiglu(const void* gate, const void* up, int64_t R, int I, moe_dtype dtype,
                  int swiglu_fusion, float limit, float alpha, float beta, void* out,
                  cudaStream_t stream) {
  if (R < 0 || I < 1 || !dtype_ok(dtype)) return MOE_ERR_INVALID_ARG;
  if (!up && swiglu_fusion != 1 && swiglu_fusion != 2) return MOE_ERR_INVALID_ARG;
  if (R > 0 && (!gate || !out)) return MOE_ERR_INVALID_ARG;
  const size_t esz = esize(dtype);
  const size_t n = (size_t)R * I * esz;
  Span outs[] = {{out, n}};
  Span ins[] = {{gate, up ? n : 2 * n}, {up, up ? n : 0}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  return cuda_status(
      launch_swiglu(gate, up, R, I, dtype, swiglu_fusion, limit, alpha, beta, out, stream));
}

size_t moe_workspace_size(int T, int H, int F, int E, int K, moe_dtype dtype) {
  if (T < 0 || H < 1 || F < 1 || E < 1 || K < 1 || !dtype_ok(dtype)) return 0;
  return ForwardWs(T, H, F, E, K, (int)esize(dtype)).total;
}

moe_status moe_indexed_mlp(const void* hidden, const void* w_gate_up, const void* w_down,
                           const float* topk_weights, const int32_t* topk_ids, int T, int H,
                           int F, int E, int K, float scale, void* out, void* ws,
                           size_t ws_bytes, cudaStream_t stream) {
  if (T < 0 || H < 1 || F < 1 || E < 1 || E > 12288 || K < 1 || !std::isfinite(scale))
    return MOE_ERR_INVALID_ARG;
  if (H % 128 != 0 || F % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if (!w_gate_up || !w_down || (T > 0 && (!hidden || !topk_weights || !topk_ids || !out)))
    return MOE_ERR_INVALID_ARG;
  // rows are streamed with 16-byte bulk copies and vector loads
  if (!aligned16(w_gate_up) || !aligned16(w_down) || (T > 0 && !aligned16(hidden)))
    return MOE_ERR_UNSUPPORTED;
  ForwardWs L(T, H, F, E, K, 2);
  if (!ws_ok(ws, ws_bytes, L.total)) return MOE_ERR_WORKSPACE;
  const size_t M = (size_t)T * K;
  Span outs[] = {{out, (size_t)T * H * 2}, {ws, L.total}};
  Span ins[] = {{hidden, (size_t)T * H * 2}, {w_gate_up, (size_t)E * 2 * F * H * 2},
                {w_down, (size_t)E * H * F * 2}, {topk_weights, M * 4}, {topk_ids, M * 4}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  if (T == 0) return MOE_OK;
  return cuda_status(launch_indexed(hidden, w_gate_up, w_down, topk_weights, topk_ids, T, H, F, E,
                                    K, scale, out, ws, L, stream));
}

namespace {

// What the entry points built on the forward change in it: the stream waits
// on hidden_ready after routing (the first step that reads the activations,
// whose copy runs on a side stream meanwhile); the combine writes its result
// to out_direct (page-locked host memory the device addresses) when set (the
// indexed path keeps writing `out`); token_scale [T] multiplies each token's
// combined sum (the indexed path is then not taken); split.w_up, when set, is
// the up projection [E, F, H] of a gate_up GEMM whose w_gate_up / b_gate_up
// then hold only the gate projection (SwiGLU fusion 0; split.b_up its bias).
struct HostHooks {
  SplitUp split{nullptr, nullptr};
  cudaEvent_t hidden_ready = nullptr;
  void* out_direct = nullptr;
  const float* token_scale = nullptr;
  bool waited = false;
  bool wrote_direct = false;
};

moe_status ffn_forward(const void* hidden, const void* logits, const void* w_gate_up,
                       const void* w_down, const float* correction_bias,
                       const int32_t* expert_ids, const void* b_gate_up, const void* b_down,
                       int T, int H, int F, int E, moe_dtype dtype, const moe_route_params* p,
                       const moe_act_params* act, void* out, float* topk_weights_out,
                       int32_t* topk_ids_out, void* router_probs, float* weight_scale,
                       void* ws, size_t ws_bytes, cudaStream_t stream, HostHooks* hooks) {
  const SplitUp* split = hooks && hooks->split.w_up ? &hooks->split : nullptr;
  moe_act_params split_st{};
  if (split) {
    if (!split_act(act, &split_st) || (!b_gate_up != !split->b_up)) return MOE_ERR_INVALID_ARG;
    act = &split_st;
  }
  if (!dtype_ok(dtype) || !act_ok(act) || H < 1 || F < 1) return MOE_ERR_INVALID_ARG;
  float dummy_w = 0.f;
  int32_t dummy_i = 0;
  moe_status st = check_route(logits, correction_bias, T, E, p, &dummy_w, &dummy_i, router_probs,
                              weight_scale);
  if (st != MOE_OK) return st;
  if (!w_gate_up || !w_down || (T > 0 && (!hidden || !out))) return MOE_ERR_INVALID_ARG;
  const int K = p->top_k;
  const size_t esz = esize(dtype), M = (size_t)T * K;
  if (M >= (1ULL << 31)) return MOE_ERR_INVALID_ARG;
  ForwardWs L(T, H, F, E, K, (int)esz);
  if (!ws_ok(ws, ws_bytes, L.total)) return MOE_ERR_WORKSPACE;
  // rows of w_gate_up (and of the up tensor, when split)
  const size_t N1 = gated_kind(act->kind) && !split ? 2 * (size_t)F : (size_t)F;
  const size_t n_up = split ? N1 : 0;
  const size_t lc = (size_t)p->local_expert_count;
  Span outs[] = {{out, (size_t)T * H * esz},        {topk_weights_out, M * 4},
                 {topk_ids_out, M * 4},             {router_probs, T * lc * rsz(p)},
                 {weight_scale, (size_t)T * 4},     {ws, L.total}};
  Span ins[] = {{hidden, (size_t)T * H * esz},
                {logits, (size_t)T * E * rsz(p)},
                {w_gate_up, (size_t)E * N1 * H * esz},
                {w_down, (size_t)E * H * F * esz},
                {correction_bias, correction_bias ? (size_t)E * 4 : 0},
                {expert_ids, expert_ids ? M * 4 : 0},
                {b_gate_up, b_gate_up ? (size_t)E * N1 * esz : 0},
                {b_down, b_down ? (size_t)E * H * esz : 0},
                {split ? split->w_up : nullptr, (size_t)E * n_up * H * esz},
                {split ? split->b_up : nullptr, split && split->b_up ? (size_t)E * n_up * esz : 0}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  if (T == 0) return MOE_OK;

  char* base = static_cast<char*>(ws);
  float* tw = topk_weights_out ? topk_weights_out : reinterpret_cast<float*>(base + L.topk_w);
  int32_t* ti = topk_ids_out ? topk_ids_out : reinterpret_cast<int32_t*>(base + L.topk_ids);
  int32_t* seg_end = reinterpret_cast<int32_t*>(base + L.seg_end);
  int32_t* r2r = reinterpret_cast<int32_t*>(base + L.row_to_route);
  int32_t* route_to_row = reinterpret_cast<int32_t*>(base + L.route_to_row);
  void* xin = base + L.expert_input;
  void* a1 = base + L.act;
  void* y = base + L.y;
  int* status = reinterpret_cast<int*>(base);
  const bool indexed =
      !(hooks && hooks->token_scale) && !split &&
      indexed_rule(T, H, F, E, K, dtype, act, b_gate_up, b_down, hidden, w_gate_up, w_down);
  // On the tcgen05 path the gate_up GEMM reads its rows straight from the
  // token-ordered hidden states through row_to_route, so the permute only
  // builds the index maps and the permuted copy of the activations is never
  // written or read back.
  const bool fused_gather = !indexed && dtype != MOE_F32 &&
                            tc_ok(hidden, w_gate_up, a1, F, H, (int)M) &&
                            (!split || aligned16(split->w_up));
  // Routing and the index maps take one launch; the staged path then copies
  // the permuted activations in a launch of its own.
  const bool fused_maps = route_permute_ok(E);
  StageTimer t_route(fused_maps ? "route_permute" : "route", stream);
  cudaError_t err =
      fused_maps ? launch_route_permute(logits, correction_bias, expert_ids, T, E, *p, tw, ti,
                                        router_probs, weight_scale, seg_end, r2r, route_to_row,
                                        ws, stream)
                 : launch_route(logits, correction_bias, expert_ids, T, E, *p, tw, ti,
                                router_probs, weight_scale, stream);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  t_route.done();
  if (hooks && hooks->hidden_ready) {
    if (cudaStreamWaitEvent(stream, hooks->hidden_ready, 0) != cudaSuccess) return MOE_ERR_CUDA;
    hooks->waited = true;
  }

  // routed_scaling_factor is folded into tw by the router: the combine scale is 1
  if (indexed) {
    StageTimer t_idx("indexed_mlp", stream);
    err = launch_indexed(hidden, w_gate_up, w_down, tw, ti, T, H, F, E, K, 1.0f, out, ws, L,
                         stream, fused_maps);
    t_idx.done();
    return cuda_status(err);
  }

  if (!fused_maps || !fused_gather) {
    StageTimer t_perm("permute", stream);
    if (!fused_maps)
      err = launch_permute(hidden, (int)esz, ti, T, H, E, K, fused_gather ? nullptr : xin,
                           seg_end, r2r, route_to_row, ws, stream);
    else
      err = launch_permute_gather(hidden, (int)esz, T, H, E, K, seg_end, r2r, xin, ws, stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    t_perm.done();
  }
  StageTimer t_gu("gate_up", stream);
  if (fused_gather)
    err = launch_gemm_tc(hidden, w_gate_up, b_gate_up, seg_end, (int)M, F, H, E, act, a1, status,
                         stream, r2r, K, T, 0, split, dtype == MOE_F16);
  else
    err = grouped_gemm(xin, w_gate_up, b_gate_up, seg_end, (int)M, F, H, E, dtype, act, a1,
                       status, stream, 0, split);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  t_gu.done();
  StageTimer t_down("down", stream);
  err = grouped_gemm(a1, w_down, b_down, seg_end, (int)M, H, F, E, dtype, nullptr, y, status,
                     stream);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  t_down.done();
  void* dst = out;
  if (hooks && hooks->out_direct) {
    dst = hooks->out_direct;
    hooks->wrote_direct = true;
  }
  StageTimer t_comb("combine", stream);
  err = launch_combine(y, tw, route_to_row, T, K, H, dtype, 1.0f, dst, stream,
                       hooks ? hooks->token_scale : nullptr);
  t_comb.done();
  return cuda_status(err);
}

// The device address of page-locked host memory (nullptr for anything else,
// e.g. pageable memory the runtime does not know).
void* mapped_host(const void* p) {
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return pa.type == cudaMemoryTypeHost ? pa.devicePointer : nullptr;
}

// One non-blocking side stream per device for the activation copy of
// moe_ffn_forward_host, created on first use and kept until the process
// exits.  Calls share it; each call's copy is ordered on it and joined back
// to the caller's stream through an event of its own.
constexpr int kMaxSideDevices = 64;
std::mutex g_side_mu;
cudaStream_t g_side[kMaxSideDevices] = {};

cudaError_t side_stream(cudaStream_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxSideDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_side_mu);
  if (!g_side[dev]) {
    e = cudaStreamCreateWithFlags(&g_side[dev], cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
  }
  *out = g_side[dev];
  return cudaSuccess;
}

}  // namespace

moe_status moe_ffn_forward_local(const void* hidden, const void* router_probs,
                                 const float* weight_scale, const void* w_gate_up,
                                 const void* w_down, const void* b_gate_up, const void* b_down,
                                 int T, int H, int F, int lc, int K, moe_dtype dtype,
                                 moe_dtype probs_dtype, const moe_act_params* act, void* out,
                                 void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (lc < 1 || K < 1 || (T > 0 && !weight_scale)) return MOE_ERR_INVALID_ARG;
  moe_route_params p{};
  p.dtype = probs_dtype;
  p.top_k = std::min(K, lc);
  p.scoring = MOE_SCORING_SOFTMAX;
  p.renormalize = 0;
  p.num_expert_group = 1;
  p.topk_group = 1;
  p.routed_scaling_factor = 1.0f;
  p.route_scale = 1.0f;
  if (T > 0) {
    Span outs[] = {{out, (size_t)T * H * esize(dtype)}};
    Span ins[] = {{weight_scale, (size_t)T * 4}};
    if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  }
  HostHooks hk;
  hk.token_scale = weight_scale;
  return ffn_forward(hidden, router_probs, w_gate_up, w_down, nullptr, nullptr, b_gate_up, b_down,
                     T, H, F, lc, dtype, &p, act, out, nullptr, nullptr, nullptr, nullptr, ws,
                     ws_bytes, stream, &hk);
}

moe_status moe_ffn_forward(const void* hidden, const void* logits, const void* w_gate_up,
                           const void* w_down, const float* correction_bias,
                           const int32_t* expert_ids, const void* b_gate_up, const void* b_down,
                           int T, int H, int F, int E, moe_dtype dtype, const moe_route_params* p,
                           const moe_act_params* act, void* out, float* topk_weights_out,
                           int32_t* topk_ids_out, void* router_probs, float* weight_scale,
                           void* ws, size_t ws_bytes, cudaStream_t stream) {
  return ffn_forward(hidden, logits, w_gate_up, w_down, correction_bias, expert_ids, b_gate_up,
                     b_down, T, H, F, E, dtype, p, act, out, topk_weights_out, topk_ids_out,
                     router_probs, weight_scale, ws, ws_bytes, stream, nullptr);
}

moe_status moe_ffn_forward_split(const void* hidden, const void* logits, const void* w_gate,
                                 const void* w_up, const void* w_down,
                                 const float* correction_bias, const int32_t* expert_ids,
                                 const void* b_gate, const void* b_up, const void* b_down, int T,
                                 int H, int F, int E, moe_dtype dtype, const moe_route_params* p,
                                 const moe_act_params* act, void* out, float* topk_weights_out,
                                 int32_t* topk_ids_out, void* router_probs, float* weight_scale,
                                 void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!w_up) return MOE_ERR_INVALID_ARG;
  HostHooks hk;
  hk.split = SplitUp{w_up, b_up};
  return ffn_forward(hidden, logits, w_gate, w_down, correction_bias, expert_ids, b_gate, b_down,
                     T, H, F, E, dtype, p, act, out, topk_weights_out, topk_ids_out,
                     router_probs, weight_scale, ws, ws_bytes, stream, &hk);
}

// ---- shared expert [TileOPs, SharedExpertMLPFwdOp]: the grouped GEMMs over one
// segment of T rows (no routing, no permutation): gate_up with silu_and_mul
// fused (gate rows then up rows, the stacked layout), then down.
namespace {
struct SharedWs {
  size_t seg_end, act, total;
  SharedWs(int T, int S, size_t esz) {
    seg_end = MOE_STATUS_BYTES;
    act = seg_end + 256;
    total = act + align256((size_t)T * S * esz);
  }
};

moe_status shared_checked(const void* hidden, const void* w_gate_up, const void* w_down, int T,
                          int H, int S, moe_dtype dtype, void* out, void* ws, cudaStream_t stream) {
  if (T == 0) return MOE_OK;
  const size_t esz = esize(dtype);
  SharedWs L(T, S, esz);
  char* base = static_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(base);
  int32_t* seg_end = reinterpret_cast<int32_t*>(base + L.seg_end);
  void* a1 = base + L.act;
  moe_act_params act{};
  act.kind = MOE_ACT_SILU_AND_MUL;
  act.swiglu_fusion = 2;
  if (launch_fill_i32(seg_end, T, 1, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (grouped_gemm(hidden, w_gate_up, nullptr, seg_end, T, S, H, 1, dtype, &act, a1, status,
                   stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cuda_status(
      grouped_gemm(a1, w_down, nullptr, seg_end, T, H, S, 1, dtype, nullptr, out, status, stream));
}
}  // namespace

size_t moe_shared_expert_workspace_size(int T, int H, int S, moe_dtype dtype) {
  if (T < 0 || H < 1 || S < 1 || !dtype_ok(dtype)) return 0;
  return SharedWs(T, S, esize(dtype)).total;
}

moe_status moe_shared_expert_mlp(const void* hidden, const void* w_gate_up, const void* w_down,
                                 int T, int H, int S, moe_dtype dtype, void* out, void* ws,
                                 size_t ws_bytes, cudaStream_t stream) {
  if (T < 0 || H < 1 || S < 1 || !dtype_ok(dtype)) return MOE_ERR_INVALID_ARG;
  if ((long long)T >= (1LL << 30)) return MOE_ERR_INVALID_ARG;
  if (!w_gate_up || !w_down || (T > 0 && (!hidden || !out))) return MOE_ERR_INVALID_ARG;
  const size_t esz = esize(dtype);
  SharedWs L(T, S, esz);
  if (!ws_ok(ws, ws_bytes, L.total)) return MOE_ERR_WORKSPACE;
  Span outs[] = {{out, (size_t)T * H * esz}, {ws, L.total}};
  Span ins[] = {{hidden, (size_t)T * H * esz},
                {w_gate_up, (size_t)2 * S * H * esz},
                {w_down, (size_t)H * S * esz}};
  if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  return shared_checked(hidden, w_gate_up, w_down, T, H, S, dtype, out, ws, stream);
}

size_t moe_workspace_size_shared(int T, int H, int F, int S, int E, int K, moe_dtype dtype) {
  const size_t a = moe_workspace_size(T, H, F, E, K, dtype);
  const size_t b = moe_shared_expert_workspace_size(T, H, S, dtype);
  return a == 0 || b == 0 ? 0 : std::max(a, b);
}

moe_status moe_ffn_forward_shared(const void* hidden, const void* logits, const void* w_gate_up,
                                  const void* w_down, const float* correction_bias,
                                  const void* shared_w_gate_up, const void* shared_w_down, int T,
                                  int H, int F, int S, int E, moe_dtype dtype,
                                  const moe_route_params* p, const moe_act_params* act,
                                  void* routed_out, void* shared_out, void* ws, size_t ws_bytes,
                                  cudaStream_t stream) {
  const bool has_shared = shared_w_gate_up != nullptr;
  if (has_shared != (shared_w_down != nullptr) || (has_shared && !shared_out))
    return MOE_ERR_INVALID_ARG;
  if (has_shared && (S < 1 || (long long)T >= (1LL << 30))) return MOE_ERR_INVALID_ARG;
  if (!p) return MOE_ERR_INVALID_ARG;
  const size_t need = has_shared ? moe_workspace_size_shared(T, H, F, S, E, p->top_k, dtype)
                                 : moe_workspace_size(T, H, F, E, p->top_k, dtype);
  if (need == 0) return MOE_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, need)) return MOE_ERR_WORKSPACE;
  if (has_shared) {
    const size_t esz = esize(dtype);
    Span outs[] = {{shared_out, (size_t)T * H * esz}, {routed_out, (size_t)T * H * esz},
                   {ws, need}};
    Span ins[] = {{hidden, (size_t)T * H * esz},
                  {shared_w_gate_up, (size_t)2 * S * H * esz},
                  {shared_w_down, (size_t)H * S * esz}};
    if (any_overlap(outs, ins)) return MOE_ERR_OVERLAP;
  }
  // the routed half (its own checks; rsf folded into its weights, so it
  // scales the routed output only), then the shared expert on the same
  // workspace (the launches are ordered on the stream)
  moe_status st = moe_ffn_forward(hidden, logits, w_gate_up, w_down, correction_bias, nullptr,
                                  nullptr, nullptr, T, H, F, E, dtype, p, act, routed_out, nullptr,
                                  nullptr, nullptr, nullptr, ws, ws_bytes, stream);
  if (st != MOE_OK || !has_shared) return st;
  return shared_checked(hidden, shared_w_gate_up, shared_w_down, T, H, S, dtype, shared_out, ws,
                        stream);
}

size_t moe_workspace_size_host(int T, int H, int F, int E, int K, moe_dtype dtype) {
  size_t base = moe_workspace_size(T, H, F, E, K, dtype);
  if (base == 0) return 0;
  const size_t esz = esize(dtype);
  return base + align256((size_t)T * H * esz) * 2 + align256((size_t)T * E * 4);
}

moe_status moe_ffn_forward_host(const void* hidden_host, const void* logits_host,
                                const void* w_gate_up, const void* w_down,
                                const float* correction_bias, const int32_t* expert_ids,
                                const void* b_gate_up, const void* b_down, int T, int H, int F,
                                int E, moe_dtype dtype, const moe_route_params* p,
                                const moe_act_params* act, void* out_host, void* router_probs,
                                float* weight_scale, void* ws, size_t ws_bytes,
                                cudaStream_t stream) {
  if (!p || !dtype_ok(dtype) || T < 0 || H < 1 || F < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!hidden_host || !logits_host || !out_host)) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_workspace_size_host(T, H, F, E, p->top_k, dtype);
  if (need == 0) return MOE_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, need)) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  const size_t esz = esize(dtype);
  const size_t fwd = moe_workspace_size(T, H, F, E, p->top_k, dtype);
  const size_t act_bytes = (size_t)T * H * esz;
  char* base = static_cast<char*>(ws);
  void* d_hidden = base + fwd;
  void* d_out = base + fwd + align256(act_bytes);
  float* d_logits = reinterpret_cast<float*>(base + fwd + 2 * align256(act_bytes));
  cudaStream_t side = nullptr;
  if (side_stream(&side) != cudaSuccess) return MOE_ERR_CUDA;
  // The activation copy runs on the side stream while the logits copy and the
  // routing run on `stream`; the forward waits for it after routing.
  cudaEvent_t fork = nullptr, ready = nullptr;
  if (cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaEventCreateWithFlags(&ready, cudaEventDisableTiming) != cudaSuccess) {
    cudaEventDestroy(fork);
    return MOE_ERR_CUDA;
  }
  moe_status st = MOE_OK;
  bool copied = false;
  // Page-locked activations are read by a copy kernel (one CTA per SM, so it
  // runs beside the routing launch), which outruns a copy engine over the
  // host link; anything else takes cudaMemcpyAsync.
  const void* h_dev = mapped_host(hidden_host);
  auto copy_in = [&]() {
    if (h_dev && act_bytes % 16 == 0 && (uintptr_t)h_dev % 16 == 0)
      return launch_copy16(h_dev, d_hidden, act_bytes, side);
    return cudaMemcpyAsync(d_hidden, hidden_host, act_bytes, cudaMemcpyHostToDevice, side);
  };
  if (cudaEventRecord(fork, stream) != cudaSuccess || cudaStreamWaitEvent(side, fork, 0) != cudaSuccess ||
      copy_in() != cudaSuccess || cudaEventRecord(ready, side) != cudaSuccess) {
    st = MOE_ERR_CUDA;
  } else {
    copied = true;
    if (cudaMemcpyAsync(d_logits, logits_host, (size_t)T * E * rsz(p), cudaMemcpyHostToDevice,
                        stream) != cudaSuccess)
      st = MOE_ERR_CUDA;
  }
  // The result is written in place when out_host is page-locked memory the
  // device can address (no staging copy; its writes overlap the combine's
  // reads); otherwise it is staged in `ws` and copied back.
  HostHooks hk;
  hk.hidden_ready = ready;
  if (st == MOE_OK) {
    hk.out_direct = mapped_host(out_host);
    st = ffn_forward(d_hidden, d_logits, w_gate_up, w_down, correction_bias, expert_ids,
                     b_gate_up, b_down, T, H, F, E, dtype, p, act, d_out, nullptr, nullptr,
                     router_probs, weight_scale, ws, fwd, stream, &hk);
  }
  // Whatever happened, nothing later on `stream` runs before the side copy.
  if (copied && !hk.waited && cudaStreamWaitEvent(stream, ready, 0) != cudaSuccess)
    st = MOE_ERR_CUDA;
  cudaEventDestroy(fork);  // released once the recorded work completes
  cudaEventDestroy(ready);
  if (st != MOE_OK) return st;
  if (hk.wrote_direct) return MOE_OK;
  return cuda_status(cudaMemcpyAsync(out_host, d_out, act_bytes, cudaMemcpyDeviceToHost, stream));
}

moe_status moe_clear_status(void* ws, cudaStream_t stream) {
  if (!ws) return MOE_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, MOE_STATUS_BYTES, stream));
}

moe_status moe_sync_status(void* ws, cudaStream_t stream) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  // after a timeout the launch that gave up may have left its grid-barrier
  // or tile counters set: the whole status area is cleared with the word
  const size_t clear = (word & kDevTimeout) ? MOE_STATUS_BYTES : sizeof(int);
  if (cudaMemset(ws, 0, clear) != cudaSuccess) return MOE_ERR_CUDA;
  if (word & kDevTimeout) return MOE_ERR_TIMEOUT;
  if (word & kDevBadIndex) return MOE_ERR_DEVICE;
  return MOE_OK;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_OVERLAP: return "an output overlaps an input";
    case MOE_ERR_UNSUPPORTED: return "unsupported dtype / activation / alignment";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "a bounded in-kernel wait ran out";
    case MOE_ERR_DEVICE: return "a kernel met an out-of-range id or index";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
  }
  return "unknown status";
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int moe_set_gemm_simt(int enable) {
  int old = g_force_simt;
  g_force_simt = enable ? 1 : 0;
  return old;
}

int moe_profile_report(char* buf, size_t buf_bytes) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    recs.swap(g_prof);
  }
  std::vector<std::string> order;
  std::map<std::string, std::pair<int, double>> agg;
  for (const ProfRec& r : recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      auto it = agg.find(r.name);
      if (it == agg.end()) {
        order.push_back(r.name);
        agg[r.name] = {1, (double)ms};
      } else {
        it->second.first += 1;
        it->second.second += ms;
      }
    }
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  std::string text;
  char line[160];
  for (const std::string& n : order) {
    const auto& v = agg[n];
    snprintf(line, sizeof line, "%s %d %.3f\n", n.c_str(), v.first, 1e3 * v.second);
    text += line;
  }
  if (buf && buf_bytes > 0) {
    const size_t n = std::min(buf_bytes - 1, text.size());
    memcpy(buf, text.data(), n);
    buf[n] = 0;
  }
  return (int)text.size();
}

int moe_test_force_wait_timeout(int enable, long long limit_ns) {
  return set_wait_timeout_test(enable, limit_ns);
}

}  // extern "C"
