// Routing of one token by one warp, shared by the router kernel and the fused
// route + permute kernel: scores in registers, group pruning and top-k by warp
// arg-max rounds.  Implements the routing of TileOPs "MoE Operators"
// (FusedTopKFwdOp, FusedMoEFwdOp) and the MoERouter log-domain outputs of
// ONNX Runtime PR #32126 "[CUDA] Add MoERouter and SwiGLU contrib operators".
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe {
namespace rt {


struct RouteArgs {
  int K, scoring, renorm, G, TG, ls, lc;
  float rsf, route_scale;
  int dt;  // moe_dtype of the logits and router_probs (the MoERouter type T)
};

// r[i] of a register array by a warp-uniform or per-lane index, without local memory
template <int NPL>
__device__ __forceinline__ float pick(const float (&r)[NPL], int i) {
  float v = 0.f;
#pragma unroll
  for (int j = 0; j < NPL; ++j) v = (j == i) ? r[j] : v;
  return v;
}

// Order-preserving unsigned key of a score: a < b  <=>  key(a) < key(b), with
// -0 and +0 equal (as the float comparison has them), every key of a real
// score >= 2, and NaN at 1 (below every score, as comparisons never pick it).
__device__ __forceinline__ unsigned order_key(float v) {
  if (v != v) return 1u;
  const unsigned b = __float_as_uint(v + 0.0f);  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The score of an order key of a real (non-NaN) score.
__device__ __forceinline__ float key_value(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// (value, index) arg-max across the warp; ties go to the lower index
__device__ __forceinline__ void warp_argmax(float& v, int& idx) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    if (ov > v || (ov == v && oi < idx)) {
      v = ov;
      idx = oi;
    }
  }
}

// Logits of token t in the calling lane's registers: z[i] = logit of expert
// lane + 32 i (-inf past E).
template <int NPL>
__device__ __forceinline__ void load_logits(int t, const void* __restrict__ logits, int E, int dt,
                                            float (&z)[NPL]) {
  const int lane = threadIdx.x & 31;
  // scores are float32 whatever the logits' type (16-bit logits widen exactly)
  if (dt == MOE_F32) {
    const float* row = static_cast<const float*>(logits) + (size_t)t * E;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      z[i] = e < E ? __ldg(row + e) : -INFINITY;
    }
  } else {
    const unsigned short* row = static_cast<const unsigned short*>(logits) + (size_t)t * E;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      const unsigned short u = e < E ? __ldg(row + e) : 0;
      z[i] = e >= E            ? -INFINITY
             : dt == MOE_F16 ? __half2float(__ushort_as_half(u))
                             : __uint_as_float((uint32_t)u << 16);
    }
  }
}

// Route token t (the calling warp; all 32 lanes) from its logits z (as
// load_logits leaves them).  Writes topk weights and ids of t, and its
// MoERouter row when a.lc > 0.
template <int NPL>
__device__ __forceinline__ void route_loaded(int t, const float (&z)[NPL],
                                             const float* __restrict__ bias,
                                             const int32_t* __restrict__ ids_in, int E,
                                             const RouteArgs& a, float* __restrict__ w_out,
                                             int32_t* __restrict__ id_out,
                                             void* __restrict__ probs,
                                             float* __restrict__ wscale) {
  const int lane = threadIdx.x & 31;
  const int K = a.K;

  // ---- scores s (float32), experts e = lane + 32 i
  float s[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) s[i] = z[i];
  if (a.scoring == MOE_SCORING_SOFTMAX) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < NPL; ++i) m = fmaxf(m, s[i]);
    m = warp_max(m);
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      int e = lane + 32 * i;
      s[i] = e < E ? expf(s[i] - m) : 0.f;
      sum += s[i];
    }
    sum = warp_sum(sum);
#pragma unroll
    for (int i = 0; i < NPL; ++i) s[i] = s[i] / sum;
  } else if (a.scoring == MOE_SCORING_SQRT_SOFTPLUS) {
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      int e = lane + 32 * i;
      // softplus(z) = max(z, 0) + log1p(exp(-|z|)), without overflow
      const float z = s[i];
      s[i] = e < E ? sqrtf(fmaxf(z, 0.f) + log1pf(expf(-fabsf(z)))) : 0.f;
    }
  } else {
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      int e = lane + 32 * i;
      s[i] = e < E ? 1.0f / (1.0f + expf(-s[i])) : 0.f;
    }
  }

  uint32_t sel = 0;  // bit i: expert lane + 32 i selected (selection path)
  float total = 0.f; // sum of the chosen scores (with multiplicity)
  const bool hash = ids_in != nullptr;
  if (hash) {
    // fixed ids: selection skipped, bias ignored
    for (int k = 0; k < K; ++k) {
      int id = __ldg(ids_in + (size_t)t * K + k);
      bool ok = id >= 0 && id < E;
      int idc = ok ? id : 0;
      float sc = __shfl_sync(0xffffffffu, pick(s, idc >> 5), idc & 31);
      total += ok ? sc : 0.f;
    }
  } else {
    // ---- selection scores u = s + bias
    float u[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      int e = lane + 32 * i;
      const float v = bias && e < E ? s[i] + __ldg(bias + e) : s[i];
      // a NaN score ranks below every number (it is never preferred to a
      // finite score, for its group or for the top-K)
      u[i] = e < E && !isnan(v) ? v : -INFINITY;
    }
    // ---- group restriction
    if (a.G > 1) {
      const int S = E / a.G;
      float my_gs = -INFINITY;  // lane g holds group g's score
      if (S % 32 == 0 && S / 32 <= NPL) {
        // A group is m = S / 32 whole registers of every lane (experts
        // lane + 32 i, i in [g m, (g + 1) m)): per lane its two best of them,
        // then the warp's best (max of the order keys) and its second best (the
        // max again with the lowest lane holding the best giving its own
        // second instead) -- the same two values, duplicates counted, as the
        // shuffle reduction below.
        const int m = S / 32;
#pragma unroll
        for (int g = 0; g < NPL; ++g) {
          if (g >= a.G) break;
          float l1 = -INFINITY, l2 = -INFINITY;
          if (m == 1) {  // one register a group (32 experts): its only value
            l1 = u[g];
          } else {
#pragma unroll
            for (int j = 0; j < NPL; ++j) {
              if (j >= g * m && j < (g + 1) * m) {
                const float v = u[j];
                if (v > l1) { l2 = l1; l1 = v; } else if (v > l2) { l2 = v; }
              }
            }
          }
          const unsigned k1 = __reduce_max_sync(0xffffffffu, order_key(l1));
          const unsigned first =
              __reduce_min_sync(0xffffffffu, order_key(l1) == k1 ? (unsigned)lane : 32u);
          const unsigned k2 = __reduce_max_sync(
              0xffffffffu, order_key((unsigned)lane == first ? l2 : l1));
          const float b1 = key_value(k1), b2 = key_value(k2);
          const float gs = bias ? b1 + b2 : b1;
          if (lane == g) my_gs = gs;
        }
      } else
      for (int g = 0; g < a.G; ++g) {
        float b1 = -INFINITY, b2 = -INFINITY;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
          int e = lane + 32 * i;
          if (e >= g * S && e < (g + 1) * S) {
            float v = u[i];
            if (v > b1) { b2 = b1; b1 = v; } else if (v > b2) { b2 = v; }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          float o1 = __shfl_xor_sync(0xffffffffu, b1, o);
          float o2 = __shfl_xor_sync(0xffffffffu, b2, o);
          float n1 = fmaxf(b1, o1);
          float n2 = fmaxf(fminf(b1, o1), fmaxf(b2, o2));
          b1 = n1;
          b2 = n2;
        }
        float gs = bias ? b1 + b2 : b1;
        if (lane == g) my_gs = gs;
      }
      uint32_t keep = 0;
      float cand = lane < a.G ? my_gs : -INFINITY;
      for (int r = 0; r < a.TG; ++r) {
        float v = cand;
        int idx = lane < a.G ? lane : 0x7fffffff;
        if (lane >= a.G) v = -INFINITY;
        // already kept groups are out of the running
        if ((keep >> lane) & 1u) { v = -INFINITY; idx = 0x7fffffff; }
        warp_argmax(v, idx);
        if (idx < a.G) keep |= 1u << idx;  // (always true: TG <= G groups to keep)
      }
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        int e = lane + 32 * i;
        if (e < E && !((keep >> (e / S)) & 1u)) u[i] = -INFINITY;
      }
    }
    // ---- top-K, ties to the lower expert index
    for (int r = 0; r < K; ++r) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        int e = lane + 32 * i;
        // ascending e inside a lane: strict '>' keeps the lower index on ties
        if (e < E && !((sel >> i) & 1u) && (be == 0x7fffffff || u[i] > bv)) {
          bv = u[i];
          be = e;
        }
      }
      // warp arg-max with the hardware warp reductions: the largest score
      // (order-preserving 32-bit key), then the lowest expert index holding it
      const unsigned key = be == 0x7fffffff ? 0u : order_key(bv);
      const unsigned kmax = __reduce_max_sync(0xffffffffu, key);
      const unsigned cand = (key == kmax && be != 0x7fffffff) ? (unsigned)be : 0x7fffffffu;
      be = (int)__reduce_min_sync(0xffffffffu, cand);
      if (be != 0x7fffffff && (be & 31) == lane) sel |= 1u << (be >> 5);
    }
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) part += ((sel >> i) & 1u) ? s[i] : 0.f;
    total = warp_sum(part);
  }

  // ---- topk ids / weights
  if (hash) {
    for (int k = 0; k < K; ++k) {
      int id = __ldg(ids_in + (size_t)t * K + k);
      bool ok = id >= 0 && id < E;
      int idc = ok ? id : 0;
      float sc = __shfl_sync(0xffffffffu, pick(s, idc >> 5), idc & 31);
      sc = ok ? sc : 0.f;
      if (lane == 0) {
        float w = a.renorm ? sc / total : sc;
        w_out[(size_t)t * K + k] = w * a.rsf;
        id_out[(size_t)t * K + k] = id;
      }
    }
  } else {
    int base = 0;
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      bool me = (sel >> i) & 1u;
      uint32_t m = __ballot_sync(0xffffffffu, me);
      if (me) {
        int pos = base + __popc(m & lt);
        float w = a.renorm ? s[i] / total : s[i];
        w_out[(size_t)t * K + pos] = w * a.rsf;
        id_out[(size_t)t * K + pos] = lane + 32 * i;
      }
      base += __popc(m);
    }
  }

  // ---- MoERouter outputs over the local slice [ls, ls + lc)
  if (a.lc > 0) {
    float acc[NPL];  // w^ mass per owned expert
#pragma unroll
    for (int i = 0; i < NPL; ++i) acc[i] = 0.f;
    if (hash) {
      for (int k = 0; k < K; ++k) {
        int id = __ldg(ids_in + (size_t)t * K + k);
        if (id < 0 || id >= E) continue;
        float sc = __shfl_sync(0xffffffffu, pick(s, id >> 5), id & 31);
        if ((id & 31) == lane) {
#pragma unroll
          for (int i = 0; i < NPL; ++i)
            if (i == (id >> 5)) acc[i] += sc / total;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < NPL; ++i) acc[i] = ((sel >> i) & 1u) ? s[i] / total : 0.f;
    }
    float local = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      int e = lane + 32 * i;
      if (e >= a.ls && e < a.ls + a.lc && e < E) {
        float v = acc[i];
        // the sentinel for an expert not chosen: -1e30, or -1e4 in float16,
        // where -1e30 would overflow to -inf
        const size_t o = (size_t)t * a.lc + (e - a.ls);
        if (a.dt == MOE_F32)
          static_cast<float*>(probs)[o] = v > 0.f ? logf(v) : -1e30f;
        else if (a.dt == MOE_F16)
          static_cast<__half*>(probs)[o] = __float2half_rn(v > 0.f ? logf(v) : -1e4f);
        else
          static_cast<__nv_bfloat16*>(probs)[o] = __float2bfloat16_rn(v > 0.f ? logf(v) : -1e30f);
        local += v;
      }
    }
    local = warp_sum(local);
    if (lane == 0) wscale[t] = a.route_scale * local;
  }
}

// Route token t (the calling warp): load_logits then route_loaded.
template <int NPL>
__device__ __forceinline__ void route_token(int t, const void* __restrict__ logits,
                                            const float* __restrict__ bias,
                                            const int32_t* __restrict__ ids_in, int E,
                                            const RouteArgs& a, float* __restrict__ w_out,
                                            int32_t* __restrict__ id_out,
                                            void* __restrict__ probs,
                                            float* __restrict__ wscale) {
  float z[NPL];
  load_logits<NPL>(t, logits, E, a.dt, z);
  route_loaded<NPL>(t, z, bias, ids_in, E, a, w_out, id_out, probs, wscale);
}

// RouteArgs from the C-ABI parameters (the MoERouter outputs are skipped when
// either of their buffers is absent).
inline RouteArgs route_args(const moe_route_params& p, const void* probs, const float* wscale) {
  RouteArgs a;
  a.K = p.top_k;
  a.scoring = p.scoring;
  a.renorm = p.renormalize != 0;
  a.G = p.num_expert_group;
  a.TG = p.topk_group;
  a.ls = p.local_expert_start;
  a.lc = (probs && wscale) ? p.local_expert_count : 0;
  a.rsf = p.routed_scaling_factor;
  a.route_scale = p.route_scale;
  a.dt = p.dtype;
  return a;
}

}  // namespace rt
}  // namespace moe
