// Router kernel: one warp per token (route_dev.cuh).
#include "route_dev.cuh"

namespace moe {
namespace {

using rt::RouteArgs;

template <int NPL>
__global__ void __launch_bounds__(256) route_kernel(const void* __restrict__ logits,
                                                    const float* __restrict__ bias,
                                                    const int32_t* __restrict__ ids_in, int T,
                                                    int E, RouteArgs a,
                                                    float* __restrict__ w_out,
                                                    int32_t* __restrict__ id_out,
                                                    void* __restrict__ probs,
                                                    float* __restrict__ wscale) {
  pdl_wait();  // everything below reads results of earlier launches
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  rt::route_token<NPL>(t, logits, bias, ids_in, E, a, w_out, id_out, probs, wscale);
}

template <int NPL>
cudaError_t launch_npl(const void* logits, const float* bias, const int32_t* ids_in, int T, int E,
                       const RouteArgs& a, float* w, int32_t* ids, void* probs, float* wscale,
                       cudaStream_t s) {
  const int warps = 8;
  dim3 grid((T + warps - 1) / warps);
  launch_pdl(route_kernel<NPL>, grid, warps * 32, 0, s, logits, bias, ids_in, T, E, a, w, ids,
      probs, wscale);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const void* logits, const float* bias, const int32_t* ids_in, int T,
                         int E, const moe_route_params& p, float* w, int32_t* ids, void* probs,
                         float* wscale, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const RouteArgs a = rt::route_args(p, probs, wscale);
  const int npl = (E + 31) / 32;
  if (npl <= 1) return launch_npl<1>(logits, bias, ids_in, T, E, a, w, ids, probs, wscale, s);
  if (npl <= 2) return launch_npl<2>(logits, bias, ids_in, T, E, a, w, ids, probs, wscale, s);
  if (npl <= 4) return launch_npl<4>(logits, bias, ids_in, T, E, a, w, ids, probs, wscale, s);
  if (npl <= 8) return launch_npl<8>(logits, bias, ids_in, T, E, a, w, ids, probs, wscale, s);
  if (npl <= 12) return launch_npl<12>(logits, bias, ids_in, T, E, a, w, ids, probs, wscale, s);
  if (npl <= 16) return launch_npl<16>(logits, bias, ids_in, T, E, a, w, ids, probs, wscale, s);
  return launch_npl<32>(logits, bias, ids_in, T, E, a, w, ids, probs, wscale, s);
}

}  // namespace moe
