// SIMT grouped GEMM over the expert-segmented ("contiguous · physical_psum")
// row layout, fp32 FMA accumulation, optional gated activation fused into the
// epilogue (TileOPs "MoE Operators", MoEGroupedGemmFwdOp).  This is the path
// for fp32 operands (kept in exact fp32, where the tensor cores would round
// to tf32) and for bf16 shapes the TMA path cannot address.
//
// Tile 64 rows x 64 output columns x 16 k, 256 threads, 4x4 outputs a thread.
// Persistent CTAs walk the per-expert tile list built in shared memory.
#include "common.cuh"

namespace moe {
namespace {

enum Mode { kPlain = 0, kStacked = 1, kInterleaved = 2 };

constexpr int SBM = 64, SBN = 64, SBK = 16;

template <typename T, int MODE>
__global__ void __launch_bounds__(256) gemm_simt_kernel(
    const T* __restrict__ a, const T* __restrict__ w, const T* __restrict__ bias,
    const int32_t* __restrict__ seg_end, int M, int Nout, int N1, int K, int E, int act_kind,
    float limit, float alpha, float beta, T* __restrict__ out, int seg_stride,
    const T* __restrict__ w_up, const T* __restrict__ bias_up) {
  __shared__ float As[SBK][SBM + 4];
  __shared__ float Bg[SBK][SBN + 4];
  __shared__ float Bu[MODE == kPlain ? 1 : SBK][SBN + 4];
  __shared__ int prefix[kMaxExperts + 1];
  __shared__ int scan_tmp[33];
  pdl_wait();  // everything below reads results of earlier launches

  const int n_tiles = (Nout + SBN - 1) / SBN;
  const int total = build_tile_prefix(seg_end, E, M, SBM, n_tiles, prefix, scan_tmp, seg_stride);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;

  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    const SegTile st = decode_tile(tile, prefix, seg_end, E, M, SBM, n_tiles, seg_stride);
    const int n0 = st.n_idx * SBN;
    const T* we = w + (size_t)st.e * N1 * K;
    // stacked up rows: Nout.. of the same expert, or 0.. of the up tensor
    const T* wu = w_up ? w_up + (size_t)st.e * N1 * K : we;
    const int up0 = w_up ? 0 : Nout;
    float accg[4][4], accu[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) accg[i][j] = accu[i][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += SBK) {
      // A: 64 rows x 16 k
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        int idx = tid + q * 256;
        int r = idx >> 4, kk = idx & 15;
        int m = st.m0 + r, k = k0 + kk;
        As[kk][r] = (m < st.m_end && k < K) ? Elem<T>::to_f(a[(size_t)m * K + k]) : 0.f;
      }
      // B: 64 output columns x 16 k (gate rows, and up rows when gated)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        int idx = tid + q * 256;
        int c = idx >> 4, kk = idx & 15;
        int j = n0 + c, k = k0 + kk;
        bool ok = j < Nout && k < K;
        int rg, ru;
        if (MODE == kStacked) { rg = j; ru = up0 + j; }
        else if (MODE == kInterleaved) { rg = 2 * j; ru = 2 * j + 1; }
        else { rg = j; ru = 0; }
        Bg[kk][c] = ok ? Elem<T>::to_f(we[(size_t)rg * K + k]) : 0.f;
        if (MODE != kPlain) Bu[kk][c] = ok ? Elem<T>::to_f(wu[(size_t)ru * K + k]) : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < SBK; ++kk) {
        float av[4], bg[4], bu[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          bg[j] = Bg[kk][tx * 4 + j];
          if (MODE != kPlain) bu[j] = Bu[kk][tx * 4 + j];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            accg[i][j] = fmaf(av[i], bg[j], accg[i][j]);
            if (MODE != kPlain) accu[i][j] = fmaf(av[i], bu[j], accu[i][j]);
          }
      }
      __syncthreads();
    }
    // epilogue: bias in fp32, activation, one cast
    const T* be = bias ? bias + (size_t)st.e * N1 : nullptr;
    const T* bue = bias_up ? bias_up + (size_t)st.e * N1 : be;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int m = st.m0 + ty * 4 + i;
      if (m >= st.m_end) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        int c = n0 + tx * 4 + j;
        if (c >= Nout) continue;
        float v;
        if (MODE == kPlain) {
          v = act_plain(act_kind, accg[i][j] + (be ? Elem<T>::to_f(be[c]) : 0.f));
        } else {
          int rg = MODE == kStacked ? c : 2 * c;
          int ru = MODE == kStacked ? up0 + c : 2 * c + 1;
          float g = accg[i][j] + (be ? Elem<T>::to_f(be[rg]) : 0.f);
          float u = accu[i][j] + (bue ? Elem<T>::to_f(bue[ru]) : 0.f);
          v = act_kind == MOE_ACT_SILU_AND_MUL   ? silu_mul(g, u)
              : act_kind == MOE_ACT_GELU_AND_MUL ? gelu_f(g) * u
                                                 : swiglu_f(g, u, limit, alpha, beta);
        }
        out[(size_t)m * Nout + c] = Elem<T>::from_f(v);
      }
    }
  }
}

template <typename T>
cudaError_t launch_t(const void* a, const void* w, const void* bias, const int32_t* seg_end, int M,
                     int Nout, int K, int E, const moe_act_params* act, void* out, cudaStream_t s,
                     int seg_stride, const SplitUp* split) {
  int mode = kPlain, kind = MOE_ACT_IDENTITY, N1 = Nout;
  float limit = 0.f, alpha = 1.f, beta = 0.f;
  if (act) kind = act->kind;
  if (act && act_is_gated(act->kind)) {
    mode = (kind == MOE_ACT_SWIGLU && act->swiglu_fusion == 1) ? kInterleaved : kStacked;
    N1 = 2 * Nout;
    limit = act->limit;
    alpha = act->alpha;
    beta = act->beta;
  }
  if (split && mode != kStacked) return cudaErrorInvalidValue;
  if (split) N1 = Nout;  // two [E, Nout, K] tensors
  const T* WU = split ? static_cast<const T*>(split->w_up) : nullptr;
  const T* BU = split ? static_cast<const T*>(split->b_up) : nullptr;
  // enough CTAs to cover the worst-case tile count, capped at a few waves
  long long max_tiles = (long long)((M + SBM - 1) / SBM + E) * ((Nout + SBN - 1) / SBN);
  long long grid = std::min<long long>(max_tiles, (long long)num_sms() * 4);
  if (grid < 1) grid = 1;
  const T* A = static_cast<const T*>(a);
  const T* W = static_cast<const T*>(w);
  const T* B = static_cast<const T*>(bias);
  T* O = static_cast<T*>(out);
  if (mode == kPlain)
    launch_pdl(gemm_simt_kernel<T, kPlain>, (unsigned)grid, 256, 0, s, A, W, B, seg_end, M, Nout,
        N1, K, E, kind, limit, alpha, beta, O, seg_stride, WU, BU);
  else if (mode == kStacked)
    launch_pdl(gemm_simt_kernel<T, kStacked>, (unsigned)grid, 256, 0, s, A, W, B, seg_end, M, Nout,
        N1, K, E, kind, limit, alpha, beta, O, seg_stride, WU, BU);
  else
    launch_pdl(gemm_simt_kernel<T, kInterleaved>, (unsigned)grid, 256, 0, s, A, W, B, seg_end, M,
        Nout, N1, K, E, kind, limit, alpha, beta, O, seg_stride, WU, BU);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_simt(const void* a, const void* w, const void* bias,
                             const int32_t* seg_end, int M, int N, int K, int E, moe_dtype dt,
                             const moe_act_params* act, void* out, int* status, cudaStream_t s,
                             int seg_stride, const SplitUp* split) {
  (void)status;
  if (M == 0 || N == 0) return cudaSuccess;
  if (dt == MOE_BF16)
    return launch_t<__nv_bfloat16>(a, w, bias, seg_end, M, N, K, E, act, out, s, seg_stride, split);
  if (dt == MOE_F16)
    return launch_t<__half>(a, w, bias, seg_end, M, N, K, E, act, out, s, seg_stride, split);
  return launch_t<float>(a, w, bias, seg_end, M, N, K, E, act, out, s, seg_stride, split);
}

}  // namespace moe
