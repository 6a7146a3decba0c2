// Standalone clamped SwiGLU: ONNX Runtime PR #32126 "[CUDA] Add MoERouter and
// SwiGLU contrib operators", section SwiGLU (float arithmetic for every T;
// limit <= 0 disables both clamps; `up` optional, then gate carries both
// halves), with the row layouts of ONNX Runtime PR #25619 "Update MoE and qMoE
// spec", section "Fusion Behavior".  Elementwise and HBM-bound: one thread per
// output element, grid-stride.
#include "common.cuh"

namespace moe {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) swiglu_kernel(const T* __restrict__ gate,
                                                     const T* __restrict__ up, int64_t R, int I,
                                                     int fusion, float limit, float alpha,
                                                     float beta, T* __restrict__ out) {
  pdl_wait();  // everything below reads results of earlier launches
  const int64_t n = R * (int64_t)I;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = idx / I;
    const int i = (int)(idx - r * I);
    float g, l;
    if (up) {
      g = Elem<T>::to_f(gate[idx]);
      l = Elem<T>::to_f(up[idx]);
    } else if (fusion == 1) {  // interleaved g, l, g, l, ...
      g = Elem<T>::to_f(gate[r * 2 * I + 2 * i]);
      l = Elem<T>::to_f(gate[r * 2 * I + 2 * i + 1]);
    } else {  // concatenated [g | l]
      g = Elem<T>::to_f(gate[r * 2 * I + i]);
      l = Elem<T>::to_f(gate[r * 2 * I + I + i]);
    }
    out[idx] = Elem<T>::from_f(swiglu_f(g, l, limit, alpha, beta));
  }
}

}  // namespace

cudaError_t launch_swiglu(const void* gate, const void* up, int64_t R, int I, moe_dtype dt,
                          int fusion, float limit, float alpha, float beta, void* out,
                          cudaStream_t s) {
  const int64_t n = R * (int64_t)I;
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)num_sms() * 16;
  if (blocks > cap) blocks = cap;
  if (dt == MOE_BF16) {
    using B = __nv_bfloat16;
    launch_pdl(swiglu_kernel<B>, (unsigned)blocks, 256, 0, s, static_cast<const B*>(gate),
        static_cast<const B*>(up), R, I, fusion, limit, alpha, beta, static_cast<B*>(out));
  } else if (dt == MOE_F16) {
    using B = __half;
    launch_pdl(swiglu_kernel<B>, (unsigned)blocks, 256, 0, s, static_cast<const B*>(gate),
        static_cast<const B*>(up), R, I, fusion, limit, alpha, beta, static_cast<B*>(out));
  } else {
    launch_pdl(swiglu_kernel<float>, (unsigned)blocks, 256, 0, s, static_cast<const float*>(gate),
        static_cast<const float*>(up), R, I, fusion, limit, alpha, beta, static_cast<float*>(out));
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
