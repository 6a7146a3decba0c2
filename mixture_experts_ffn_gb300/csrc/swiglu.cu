// Standalone clamped SwiGLU: ONNX Runtime PR #32126 "[CUDA] Add MoERouter and
// SwiGLU contrib operators", section SwiGLU (float arithmetic for every T;
// limit <= 0 disables both clamps; `up` optional, then gate carries both
// halves), with the row layouts of ONNX Runtime PR #25619 "Update MoE and qMoE
// spec", section "Fusion Behavior".  Elementwise and HBM-bound: with 16-byte
// aligned rows a thread handles 16 bytes of output (8 half-width or 4 fp32
// elements) from 16-byte loads, one row split per item; otherwise one thread
// per element.  Grid-stride over at most one resident round of CTAs.
#include <algorithm>
#include <type_traits>

#include "common.cuh"

namespace moe {
namespace {

// V consecutive elements of a row from 16 bytes at p (V * sizeof(T) == 16)
template <typename T, int V>
__device__ __forceinline__ void load_vec(const T* __restrict__ p, float (&v)[V]) {
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
  if constexpr (std::is_same<T, float>::value) {
    v[0] = __uint_as_float(q.x);
    v[1] = __uint_as_float(q.y);
    v[2] = __uint_as_float(q.z);
    v[3] = __uint_as_float(q.w);
  } else {
    constexpr bool H16 = std::is_same<T, __half>::value;
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = lo16<H16>(u[i]);
      v[2 * i + 1] = hi16<H16>(u[i]);
    }
  }
}
template <typename T, int V>
__device__ __forceinline__ void store_vec(T* __restrict__ p, const float (&v)[V]) {
  uint4 q;
  if constexpr (std::is_same<T, float>::value) {
    q = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                   __float_as_uint(v[3]));
  } else {
    constexpr bool H16 = std::is_same<T, __half>::value;
    q = make_uint4(pack2<H16>(v[0], v[1]), pack2<H16>(v[2], v[3]), pack2<H16>(v[4], v[5]),
                   pack2<H16>(v[6], v[7]));
  }
  *reinterpret_cast<uint4*>(p) = q;
}

// Item = V consecutive output elements of one row; needs I % V == 0 and every
// row start 16-byte aligned.
template <typename T, int V>
__global__ void __launch_bounds__(256) swiglu_vec_kernel(const T* __restrict__ gate,
                                                         const T* __restrict__ up, int64_t R,
                                                         int I, int fusion, float limit,
                                                         float alpha, float beta,
                                                         T* __restrict__ out) {
  pdl_wait();  // everything below reads results of earlier launches
  const int nv = I / V;
  const int64_t items = R * (int64_t)nv;
  for (int64_t it = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; it < items;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = it / nv;
    const int c = (int)(it - r * nv) * V;
    float g[V], l[V], o[V];
    if (up) {
      load_vec<T, V>(gate + r * I + c, g);
      load_vec<T, V>(up + r * I + c, l);
    } else if (fusion == 1) {  // interleaved g, l, g, l, ...: 2V elements
      float a[V], b[V];
      load_vec<T, V>(gate + r * 2 * I + 2 * c, a);
      load_vec<T, V>(gate + r * 2 * I + 2 * c + V, b);
#pragma unroll
      for (int i = 0; i < V / 2; ++i) {
        g[i] = a[2 * i];
        l[i] = a[2 * i + 1];
        g[V / 2 + i] = b[2 * i];
        l[V / 2 + i] = b[2 * i + 1];
      }
    } else {  // concatenated [g | l]
      load_vec<T, V>(gate + r * 2 * I + c, g);
      load_vec<T, V>(gate + r * 2 * I + I + c, l);
    }
#pragma unroll
    for (int i = 0; i < V; ++i) o[i] = swiglu_f(g[i], l[i], limit, alpha, beta);
    store_vec<T, V>(out + r * I + c, o);
  }
}

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
  // 16-byte items when every row start and the item offsets are 16-byte aligned
  const int V = dt == MOE_F32 ? 4 : 8;
  const auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (I % V == 0 && a16(gate) && a16(out) && (!up || a16(up))) {
    const int64_t items = R * (int64_t)(I / V);
    auto go = [&](auto tag) {
      using B = decltype(tag);
      constexpr int VB = sizeof(B) == 4 ? 4 : 8;
      const void* k = (const void*)swiglu_vec_kernel<B, VB>;
      const int64_t blocks = std::min<int64_t>((items + 255) / 256,
                                               (int64_t)num_sms() * resident_ctas(k, 256));
      launch_pdl(swiglu_vec_kernel<B, VB>, (unsigned)std::max<int64_t>(blocks, 1), 256, 0, s,
                 static_cast<const B*>(gate), static_cast<const B*>(up), R, I, fusion, limit,
                 alpha, beta, static_cast<B*>(out));
    };
    if (dt == MOE_BF16) go(__nv_bfloat16{});
    else if (dt == MOE_F16) go(__half{});
    else go(float{});
    count_launch();
    return cudaGetLastError();
  }
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
