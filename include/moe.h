/*
 * moe.h -- C ABI of libmoe.so, a GB300 (sm_103a) routed Mixture-of-Experts FFN
 * forward.
 *
 * The layer computes, per token t with hidden row h[t] and router logits z[t]:
 *
 *   ids, w = route(z[t])                                   (moe_route)
 *   out[t] = sum_k w[k] * (down_k(act(gate_up_k(h[t]) + b1_k)) + b2_k)
 *
 * staged as route -> permute into an expert-contiguous layout
 * (moe_permute) -> grouped gate_up GEMM with the gated activation fused into its
 * epilogue (moe_grouped_gemm_act) -> grouped down GEMM (moe_grouped_gemm_down)
 * -> unpermute and weighted combine (moe_combine); or, when the routes are few,
 * the indexed per-route path (moe_indexed_mlp).  moe_ffn_forward runs the whole
 * layer, fusing stages where it can (moe_route_permute,
 * moe_grouped_gemm_act_gathered).  Sources are cited per function as (page title, section):
 *   [TileOPs]    TileOPs "MoE Operators" (one section per op),
 *   [MoERouter]  ONNX Runtime PR #32126 "[CUDA] Add MoERouter and SwiGLU
 *                contrib operators",
 *   [ORT-spec]   ONNX Runtime PR #25619 "Update MoE and qMoE spec",
 *   [ORT-MoE]    onnx-light-cpu "MoE (CPU)".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is caller-owned DEVICE memory (cudaMalloc'd or any
 *    device-accessible allocation).  The library never allocates; scratch space
 *    comes from the caller's workspace `ws` of `ws_bytes` bytes (see
 *    moe_workspace_size) and must be 256-byte aligned.
 *  - Tensors are dense, row-major, with the shapes given in brackets.
 *    Element types: MOE_F32 (float) or MOE_BF16 (bfloat16) for activations,
 *    weights, biases and outputs; logits, correction bias, routing weights and
 *    MoERouter outputs are always float32; ids and index maps int32.
 *  - Every call is asynchronous on `stream` (0 = legacy default stream) and
 *    returns a moe_status.  Argument checks happen on the host before anything
 *    is launched: an invalid call writes nothing.  Outputs that overlap an
 *    input return MOE_ERR_OVERLAP before any launch (disjoint views of one
 *    allocation are fine) [TileOPs, MoEPostPermuteFwdOp / MoEGroupedGemmFwdOp].
 *  - The CONTENTS of index tensors (ids, segment ends, index maps) are not
 *    checked on the host, since checking would synchronise [TileOPs,
 *    MoEGroupedGemmFwdOp].  Kernels that meet an out-of-range id or index skip
 *    that item and latch a device error in the workspace status word;
 *    moe_sync_status reports it as MOE_ERR_DEVICE.
 *  - Every wait inside a kernel is bounded; a wait that runs out latches
 *    MOE_ERR_TIMEOUT in the status word instead of hanging.
 *  - A workspace serves one call at a time: calls that can run at the same
 *    time on the GPU (on different streams) need workspaces of their own,
 *    since the status word and the self-resetting counters at the start of
 *    a workspace are state the call's kernels update.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* a shape, enum or parameter is out of range          */
  MOE_ERR_OVERLAP = 2,     /* an output overlaps an input                          */
  MOE_ERR_UNSUPPORTED = 3, /* a dtype / activation / alignment combination not built */
  MOE_ERR_CUDA = 4,        /* a CUDA launch or runtime call failed                 */
  MOE_ERR_TIMEOUT = 5,     /* a bounded in-kernel wait ran out (status word)       */
  MOE_ERR_DEVICE = 6,      /* a kernel met an out-of-range id / index (status word) */
  MOE_ERR_WORKSPACE = 7    /* ws is NULL, misaligned or smaller than required      */
} moe_status;

/* Element types [ORT-MoE and MoERouter, tensor type T: float, float16,
 * bfloat16].  Arithmetic is float32 for every type; results are rounded to
 * the operand type (round to nearest even) at the points the bf16 path
 * rounds.  MOE_F16 takes the same paths as MOE_BF16 (tcgen05 GEMMs with
 * kind::f16 float16 operands) except the indexed decode kernel, which is
 * bf16 only. */
typedef enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1, MOE_F16 = 2 } moe_dtype;

/* Router scores of the logits z [MoERouter scoring; TileOPs FusedTopKFwdOp]:
 * softmax over the experts; sigmoid(z); sqrt(log(1 + exp(z))) (the name
 * "sqrt_softplus" read literally). */
typedef enum moe_scoring {
  MOE_SCORING_SOFTMAX = 0,
  MOE_SCORING_SIGMOID = 1,
  MOE_SCORING_SQRT_SOFTPLUS = 2
} moe_scoring;

typedef enum moe_act_kind {
  /* silu(gate) * up over a STACKED w_gate_up: F gate rows, then F up rows
     [TileOPs, MoEGroupedGemmFwdOp]. */
  MOE_ACT_SILU_AND_MUL = 0,
  /* clamped SwiGLU G*sigmoid(alpha*G)*(L+beta), G = min(gate, limit),
     L = clamp(up, -limit, limit), limit <= 0 disables both clamps; rows
     interleaved (swiglu_fusion 1: row 2j gate j, row 2j+1 up j -- gpt-oss
     "swigluoai" with limit 7, alpha 1.702, beta 1) or concatenated
     (swiglu_fusion 2: gate rows then up rows) [MoERouter, SwiGLU;
     ORT-spec, "SwiGLU Activation Function" and "Fusion Behavior"]. */
  MOE_ACT_SWIGLU = 1,
  /* non-gated identity: w_gate_up is [E, F, H] and act(p) = p
     [ORT-MoE, activation_type "identity"]. */
  MOE_ACT_IDENTITY = 2,
  /* gelu(gate) * up over a STACKED w_gate_up, gelu(x) = x * Phi(x) (the
     exact, erf form) [TileOPs, MoEGroupedGemmFwdOp "gelu_and_mul"]. */
  MOE_ACT_GELU_AND_MUL = 3,
  /* non-gated: w_gate_up is [E, F, H] and act(p) = max(p, 0), gelu(p) or
     p * sigmoid(p) [ORT-MoE, activation_type relu / gelu / silu]. */
  MOE_ACT_RELU = 4,
  MOE_ACT_GELU = 5,
  MOE_ACT_SILU = 6
} moe_act_kind;

/* Router configuration [TileOPs, FusedTopKFwdOp / FusedMoEFwdOp; MoERouter]. */
typedef struct moe_route_params {
  int32_t top_k;                 /* K, 1 <= K <= min(E, 64)                            */
  int32_t scoring;               /* moe_scoring                                        */
  int32_t renormalize;           /* nonzero: divide the K weights by their sum         */
  int32_t num_expert_group;      /* G >= 1, must divide E, G <= 32                     */
  int32_t topk_group;            /* TG, 1 <= TG <= G, TG * E / G >= K                   */
  float routed_scaling_factor;   /* rsf > 0, multiplies the weights once               */
  int32_t local_expert_start;    /* MoERouter slice [start, start + count) of [0, E)   */
  int32_t local_expert_count;    /* 0: no router_probs / weight_scale outputs          */
  float route_scale;             /* MoERouter weight_scale multiplier                  */
  int32_t dtype;                 /* moe_dtype of logits and router_probs (MoERouter's
                                    T; 0 = float32).  Scores are float32 whatever T;
                                    the router_probs sentinel is -1e30, or -1e4 in
                                    float16 (-1e30 overflows it)                      */
} moe_route_params;

/* Gated activation fused into the gate_up GEMM epilogue. */
typedef struct moe_act_params {
  int32_t kind;          /* moe_act_kind                                          */
  int32_t swiglu_fusion; /* MOE_ACT_SWIGLU only: 1 interleaved, 2 concatenated,
                            0 two tensors (the *_split entry points)             */
  float limit;           /* SwiGLU clamp; <= 0 disables both clamps                */
  float alpha;           /* SwiGLU sigmoid scale                                   */
  float beta;            /* SwiGLU linear offset                                   */
} moe_act_params;

/* ------------------------------------------------------------------------ */
/* Router.  [TileOPs, FusedTopKFwdOp and FusedMoEFwdOp; MoERouter, MoERouter]
 *
 * Per token t (one warp per token), in float32:
 *   s = softmax(z[t]) or sigmoid(z[t]);  u = s + correction_bias (selection only);
 *   G > 1: groups of E/G consecutive experts score the sum of their two best u
 *          (with a bias) or their best u (without); the TG best groups are kept,
 *          ties to the lower group index;
 *   the K largest u among kept experts, ties to the lower expert index -- or the
 *   given expert_ids[t] (hash routing: selection skipped, bias ignored);
 *   w_k = s[id_k], divided by sum_j s[id_j] when renormalize, times rsf once.
 * Selected ids are written in ASCENDING expert order; fixed expert_ids keep
 * their given order.
 * MoERouter outputs (when local_expert_count > 0): with w^_k = s[id_k] /
 * sum_j s[id_j] (always normalised, no rsf), router_probs[t, j] =
 * log(sum of w^_k over routes on expert local_expert_start + j) if chosen,
 * else -1e30 (-1e4 when p->dtype is MOE_F16: -1e30 overflows float16);
 * weight_scale[t] = route_scale * sum of w^ over local routes (0 when no
 * chosen expert is local).
 *
 *   logits          [T, E] p->dtype (f32, bf16 or f16; scores in f32)
 *   correction_bias [E] f32 or NULL; not with MOE_SCORING_SOFTMAX
 *   expert_ids      [T, K] i32 or NULL (hash routing)
 *   topk_weights    [T, K] f32 out;  topk_ids [T, K] i32 out
 *   router_probs    [T, local_expert_count] p->dtype out or NULL
 *   weight_scale    [T] f32 out or NULL (both or neither when count > 0)
 * E <= 1024.  T == 0 is a no-op. */
moe_status moe_route(const void* logits, const float* correction_bias,
                     const int32_t* expert_ids, int T, int E, const moe_route_params* p,
                     float* topk_weights, int32_t* topk_ids, void* router_probs,
                     float* weight_scale, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* moe_route followed by moe_permute without the gather (expert_input NULL),
 * in one launch (an addition; the forward uses it whenever E <= 512).
 * Outputs are bit-identical to the two calls: topk_weights,
 * topk_ids, router_probs, weight_scale as moe_route; seg_end, row_to_route,
 * route_to_row as moe_permute.  E <= 512 (MOE_ERR_UNSUPPORTED above; use the
 * two calls).  ws: >= moe_permute_workspace_size(T*K, E) bytes whose status
 * word was cleared (moe_clear_status); the call also uses bytes 16..27 of the
 * status area.  It runs one CTA per SM that meet at two bounded grid
 * barriers; the launch is cooperative, so the grid starts only when all of
 * its CTAs can be resident (concurrent calls on other streams are safe).  A
 * barrier that still waits after 2 s latches MOE_ERR_TIMEOUT. */
moe_status moe_route_permute(const void* logits, const float* correction_bias,
                             const int32_t* expert_ids, int T, int E, const moe_route_params* p,
                             float* topk_weights, int32_t* topk_ids, void* router_probs,
                             float* weight_scale, int32_t* seg_end, int32_t* row_to_route,
                             int32_t* route_to_row, void* ws, size_t ws_bytes,
                             cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Permute into the tight expert-contiguous layout ("contiguous ·
 * physical_psum": segment END rows) [TileOPs, MoEPrePermuteFwdOp and
 * MoEGroupedGemmFwdOp].
 *
 * Route r = t*K + k goes to expert topk_ids[r].  seg_end[e] = number of routes
 * on experts 0..e (inclusive prefix sum).  Rows of expert e hold its routes in
 * ascending r.  row_to_route[row] = r and route_to_row[r] = row.
 * expert_input[row, :] = hidden[row_to_route[row] / K, :]; pass NULL
 * expert_input (and hidden) to build the index maps only.
 *
 *   hidden       [T, H] dtype (or NULL)     topk_ids     [T, K] i32
 *   expert_input [T*K, H] dtype out or NULL seg_end      [E] i32 out
 *   row_to_route [T*K] i32 out              route_to_row [T*K] i32 out
 *   ws: >= moe_permute_workspace_size(T*K, E) bytes.
 * An id outside [0, E) latches MOE_ERR_DEVICE; that route is dropped. */
moe_status moe_permute(const void* hidden, moe_dtype dtype, const int32_t* topk_ids, int T,
                       int H, int E, int K, void* expert_input, int32_t* seg_end,
                       int32_t* row_to_route, int32_t* route_to_row, void* ws,
                       size_t ws_bytes, cudaStream_t stream);

/* Padded permute-align layout [TileOPs "MoE Operators", MoEPermuteAlignFwdOp]:
 * with numel = T*K routes and count[e] on expert e, num_tokens_post_pad[0] =
 * sum over e of count[e] rounded up to block_size; sorted_token_ids holds one
 * range per expert, in expert order, of that rounded-up length: its first
 * count[e] slots are the routes on e in ascending route index (the order the
 * pages leave open, fixed here), the rest numel; every entry past
 * num_tokens_post_pad is numel.  expert_ids names the owner of each
 * block_size block of the ranges and is -1 past them.  An id outside [0, E)
 * drops its route and latches MOE_ERR_DEVICE, as in moe_permute.
 *
 *   topk_ids [T, K] i32;  sorted_token_ids [T*K + (E+1)*(block_size-1)] i32 out;
 *   expert_ids [ceil(that / block_size)] i32 out;  num_tokens_post_pad [1] i32 out;
 *   ws >= moe_permute_align_workspace_size(T, K, E).  E <= 12288. */
moe_status moe_permute_align(const int32_t* topk_ids, int T, int K, int E, int block_size,
                             int32_t* sorted_token_ids, int32_t* expert_ids,
                             int32_t* num_tokens_post_pad, void* ws, size_t ws_bytes,
                             cudaStream_t stream);
size_t moe_permute_align_workspace_size(int T, int K, int E);

/* The gather step of moe_permute on its own (an addition), from index maps
 * already built (moe_route_permute, or moe_permute without the gather):
 * expert_input[row, :] = hidden[row_to_route[row] / K, :] for every row below
 * seg_end[E-1].  Bit-identical to moe_permute's expert_input.
 *
 *   hidden [T, H] dtype;  seg_end [E] i32;  row_to_route [T*K] i32;
 *   expert_input [T*K, H] dtype out (rows past seg_end[E-1] not written);
 *   ws >= MOE_STATUS_BYTES bytes.
 * A map entry outside [0, T*K) latches MOE_ERR_DEVICE and its row is not
 * written. */
moe_status moe_permute_gather(const void* hidden, moe_dtype dtype, const int32_t* seg_end,
                              const int32_t* row_to_route, int T, int H, int E, int K,
                              void* expert_input, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* moe_permute for callers that cannot allocate device memory.  (The pages have
 * no counterpart: this is a property of the library, not of the method.)
 *
 * Some callers cannot call cudaMalloc where they run the layer: cudaMalloc and
 * cudaFree can synchronise the whole device, and serving runtimes with a fixed
 * memory budget (or their own allocator owning all device memory) forbid any
 * allocation after start-up.  This variant takes no workspace: its scratch is
 * a fixed 1 MiB array in device memory owned by the library, which every GPU
 * that loads the library holds until the process exits.  The caller still
 * passes every input and output; arguments, layout and results are those of
 * moe_permute.
 *
 *  - Limit: the permute scratch (256 + ceil(T*K/1024)*E*4 + E*4 bytes, rounded
 *    up to 256-byte sections) must fit in 1 MiB -- e.g. T*K up to 131072 routes
 *    with E up to 1024 experts; larger sizes return MOE_ERR_WORKSPACE and launch
 *    nothing.
 *  - The first call on each device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Every call on a device shares the one array and it keeps the last call's
 *    contents (each call clears what must start at zero): calls that can
 *    overlap on the GPU -- on different streams, or from different threads --
 *    race and must be serialised by the caller.
 *  - Out-of-range ids are dropped as in moe_permute, but the device status bit
 *    they latch lives in the library's array and is not reported. */
moe_status moe_permute_noalloc(const void* hidden, moe_dtype dtype, const int32_t* topk_ids,
                               int T, int H, int E, int K, void* expert_input, int32_t* seg_end,
                               int32_t* row_to_route, int32_t* route_to_row, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Grouped gate_up GEMM with the gated activation fused into its epilogue
 * [TileOPs, MoEGroupedGemmFwdOp ("activation"), MoEExpertMLPFwdOp].
 *
 * For each expert e and each row m in [seg_end[e-1], seg_end[e]):
 *   p = a[m, :] . w_gate_up[e, n, :] (+ b_gate_up[e, n])   for every n, in fp32
 *   out[m, j] = act(p)_j, cast to dtype                     (j < F)
 * The [M, 2F] product is never written.  bf16 runs on the tcgen05 tensor
 * cores (TMA-fed, TMEM accumulators) when Hk % 8 == 0, F % 8 == 0 and a,
 * w_gate_up, out are 16-byte aligned (16-byte TMA strides); f32, and bf16
 * shapes outside those limits, run a SIMT kernel in exact fp32 FMA.
 *
 *   a          [M, Hk] dtype               w_gate_up [E, N1, Hk] dtype
 *              (N1 = 2F for the gated kinds, F for the non-gated ones)
 *   b_gate_up  [E, N1] dtype or NULL (in w_gate_up's row order)
 *   seg_end    [E] i32, non-decreasing, seg_end[E-1] <= M
 *   out        [M, F] dtype
 *   ws: >= MOE_STATUS_BYTES bytes (holds the status word).
 * E <= 1024.  Rows past seg_end[E-1] are not written. */
moe_status moe_grouped_gemm_act(const void* a, const void* w_gate_up, const void* b_gate_up,
                                const int32_t* seg_end, int M, int F, int Hk, int E,
                                moe_dtype dtype, const moe_act_params* act, void* out, void* ws,
                                size_t ws_bytes, cudaStream_t stream);

/* The same GEMM with the gate and up projections in two tensors [ORT-spec,
 * "Fusion Behavior", swiglu_fusion 0: FC1 gives g, FC3 gives l, two GEMMs
 * computed independently]:
 *   g = a[m, :] . w_gate[e, j, :] (+ b_gate[e, j]),
 *   l = a[m, :] . w_up[e, j, :] (+ b_up[e, j]),   out[m, j] = act(g, l).
 * Both projections feed one accumulator tile, so neither is written out.
 * act->kind: MOE_ACT_SILU_AND_MUL, MOE_ACT_GELU_AND_MUL, or MOE_ACT_SWIGLU
 * with swiglu_fusion 0 (MOE_ERR_INVALID_ARG otherwise).
 *   w_gate, w_up [E, F, Hk] dtype;  b_gate, b_up [E, F] dtype, both or neither;
 *   a, seg_end, out, ws and the tensor-core rule as moe_grouped_gemm_act
 *   (w_up 16-byte aligned as well). */
moe_status moe_grouped_gemm_act_split(const void* a, const void* w_gate, const void* w_up,
                                      const void* b_gate, const void* b_up,
                                      const int32_t* seg_end, int M, int F, int Hk, int E,
                                      moe_dtype dtype, const moe_act_params* act, void* out,
                                      void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* moe_grouped_gemm_act over gathered rows (an addition; the pages' grouped
 * GEMM takes the permuted copy of the activations).  Row m of the operand is
 * hidden[row_to_route[m] / top_k], read straight from the token-ordered hidden
 * states, so the [M, H] permuted copy (moe_permute's expert_input) is neither
 * written nor read: moe_permute with expert_input == NULL builds the maps.
 * The result equals moe_grouped_gemm_act on that copy, bit for bit.
 *
 *   hidden        [T, H] bf16, 16-byte aligned, H % 8 == 0
 *   row_to_route  [M] i32 from moe_permute (route index t*top_k + k of row m)
 *   w_gate_up, b_gate_up, seg_end, act, out, ws: as moe_grouped_gemm_act with
 *   Hk = H (F % 8 == 0; w_gate_up and out 16-byte aligned)
 * Only rows below seg_end[E-1] are read; an entry of row_to_route outside
 * [0, T*top_k) gives a zero row.  bf16 on the tcgen05 path only: other dtypes,
 * shapes or alignments return MOE_ERR_UNSUPPORTED (use moe_permute with an
 * expert_input buffer and moe_grouped_gemm_act instead). */
moe_status moe_grouped_gemm_act_gathered(const void* hidden, int T, const int32_t* row_to_route,
                                         int top_k, const void* w_gate_up,
                                         const void* b_gate_up, const int32_t* seg_end, int M,
                                         int F, int H, int E, moe_dtype dtype,
                                         const moe_act_params* act, void* out, void* ws,
                                         size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Plain grouped down GEMM [TileOPs, MoEGroupedGemmFwdOp (no activation),
 * MoEExpertMLPFwdOp]: out[m, :] = a[m, :] . w_down[e]^T (+ b_down[e]) in fp32,
 * cast to dtype, for the rows m of expert e.
 *
 *   a [M, F] dtype;  w_down [E, H, F] dtype;  b_down [E, H] dtype or NULL;
 *   seg_end [E] i32;  out [M, H] dtype;  ws >= MOE_STATUS_BYTES bytes.
 * Kernel choice as for moe_grouped_gemm_act (tcgen05 for bf16 with H % 8 == 0,
 * F % 8 == 0 and 16-byte aligned a, w_down, out). */
moe_status moe_grouped_gemm_down(const void* a, const void* w_down, const void* b_down,
                                 const int32_t* seg_end, int M, int H, int F, int E,
                                 moe_dtype dtype, void* out, void* ws, size_t ws_bytes,
                                 cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Unpermute + weighted combine [TileOPs, MoEPostPermuteFwdOp and
 * FusedMoEExpertsFwdOp]:
 *   out[t, :] = scale * sum_{k = 0..K-1} topk_weights[t, k] *
 *               expert_out[route_to_row[t*K + k], :]
 * accumulated in fp32 in fixed k order (deterministic, no atomics) and cast
 * once to dtype.
 *
 *   expert_out [M, H] dtype (M = T*K);  topk_weights [T, K] f32;
 *   route_to_row [T*K] i32;  out [T, H] dtype.
 * An index outside [0, T*K) contributes nothing (nothing is latched: this
 * entry point has no workspace). */
moe_status moe_combine(const void* expert_out, const float* topk_weights,
                       const int32_t* route_to_row, int T, int K, int H, moe_dtype dtype,
                       float scale, void* out, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Standalone SwiGLU [MoERouter, section SwiGLU; ORT-spec "SwiGLU Activation
 * Function", "Fusion Behavior"]:
 *   G = min(g, limit), L = max(min(l, limit), -limit)   (limit <= 0: no clamp)
 *   out = G * sigmoid(alpha * G) * (L + beta), arithmetic in float32.
 * With `up` given, g = gate[r, i] and l = up[r, i] ([R, I] each).  With up ==
 * NULL, gate is one [R, 2I] projection: swiglu_fusion 2 = [g | l] (gate
 * first, then up), 1 = interleaved (g, l, g, l, ...).
 *   out [R, I] dtype. */
moe_status swiglu(const void* gate, const void* up, int64_t R, int I, moe_dtype dtype,
                  int swiglu_fusion, float limit, float alpha, float beta, void* out,
                  cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Indexed small-route expert MLP [TileOPs, IndexedExpertMLPFwdOp]: the same
 * result as permute + the two grouped GEMMs (silu_and_mul, no bias) +
 * combine, dispatched per route.  Routes sharing an expert are grouped and
 * each distinct expert's weights are streamed from HBM once, for all of its
 * routes, with 128-bit loads.  bf16 only; H % 128 == 0, F % 256 == 0,
 * hidden / w_gate_up / w_down 16-byte aligned (MOE_ERR_UNSUPPORTED otherwise).
 *
 *   hidden [T, H] bf16;  w_gate_up [E, 2F, H] bf16 (stacked);  w_down [E, H, F];
 *   topk_weights [T, K] f32;  topk_ids [T, K] i32;  out [T, H] bf16;
 *   ws >= moe_workspace_size(T, H, F, E, K, MOE_BF16). */
moe_status moe_indexed_mlp(const void* hidden, const void* w_gate_up, const void* w_down,
                           const float* topk_weights, const int32_t* topk_ids, int T, int H,
                           int F, int E, int K, float scale, void* out, void* ws,
                           size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* The whole routed MoE FFN forward [TileOPs, FusedMoEFwdOp and
 * FusedMoEExpertsFwdOp].  Routes with moe_route (rsf folded into the weights,
 * so it applies once), then runs the indexed path when T*K <= 2E, the
 * activation is silu_and_mul, there is no bias, dtype is bf16, H % 128 == 0,
 * F % 256 == 0 and hidden and the weights are 16-byte aligned [TileOPs,
 * FusedMoEExpertsFwdOp dispatch rule]; otherwise
 * the staged pipeline permute -> gate_up+act -> down -> combine.
 * Routing and the index maps take one launch when E <= 512
 * (moe_route_permute).  When the gate_up GEMM runs on the tensor cores (bf16,
 * H % 8 == 0, F % 8 == 0, 16-byte aligned hidden, weights and workspace
 * sections), the permuted copy of the activations is never materialised: the
 * gate_up GEMM reads its rows through row_to_route
 * (moe_grouped_gemm_act_gathered), so the layer is four launches; otherwise
 * the permuted copy takes a launch of its own after the maps.  The results
 * are the same as the staged calls'.  Every launch is made with programmatic dependent launch, so each
 * overlaps the tail of the previous one.
 *
 *   hidden [T, H] dtype;  logits [T, E] p->dtype;  w_gate_up [E, N1, H];
 *   w_down [E, H, F];  correction_bias [E] f32 | NULL;  expert_ids [T, K] | NULL;
 *   b_gate_up [E, N1] | NULL;  b_down [E, H] | NULL;  out [T, H] dtype;
 *   topk_weights_out [T, K] f32 | NULL, topk_ids_out [T, K] i32 | NULL
 *   (optional copies of the routing);  router_probs / weight_scale as in
 *   moe_route (NULL unless p->local_expert_count > 0);
 *   ws >= moe_workspace_size(T, H, F, E, K, dtype). */
moe_status moe_ffn_forward(const void* hidden, const void* logits, const void* w_gate_up,
                           const void* w_down, const float* correction_bias,
                           const int32_t* expert_ids, const void* b_gate_up, const void* b_down,
                           int T, int H, int F, int E, moe_dtype dtype,
                           const moe_route_params* p, const moe_act_params* act, void* out,
                           float* topk_weights_out, int32_t* topk_ids_out, void* router_probs,
                           float* weight_scale, void* ws, size_t ws_bytes, cudaStream_t stream);

/* moe_ffn_forward with the gate and up projections of the experts in two
 * tensors (SwiGLU fusion 0 [ORT-spec, "Fusion Behavior"]; act as
 * moe_grouped_gemm_act_split): w_gate, w_up [E, F, H]; b_gate, b_up [E, F] |
 * NULL, both or neither.  Always the staged pipeline (the indexed path reads
 * stacked weights); the gate_up GEMM reads both tensors into one accumulator
 * tile.  Everything else, ws included, as moe_ffn_forward. */
moe_status moe_ffn_forward_split(const void* hidden, const void* logits, const void* w_gate,
                                 const void* w_up, const void* w_down,
                                 const float* correction_bias, const int32_t* expert_ids,
                                 const void* b_gate, const void* b_up, const void* b_down, int T,
                                 int H, int F, int E, moe_dtype dtype, const moe_route_params* p,
                                 const moe_act_params* act, void* out, float* topk_weights_out,
                                 int32_t* topk_ids_out, void* router_probs, float* weight_scale,
                                 void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* The layer of one expert-parallel rank, fed by the MoERouter outputs of its
 * slice of lc experts [ONNX Runtime PR #32126 "[CUDA] Add MoERouter and
 * SwiGLU contrib operators", MoERouter: the expert op's own softmax over the
 * local row of router_probs returns w_e / W_local, and weight_scale
 * multiplies that factor back out before the ranks' outputs are summed].
 * Routes each token by the softmax (in fp32) of its router_probs row and its top
 * min(K, lc) experts (ties to the lower index, no renormalisation), runs the
 * expert MLPs of this rank's experts as moe_ffn_forward does (the tensor-core
 * or staged path; not the indexed one), and multiplies each token's combined
 * sum by weight_scale[t] before the single cast.  Summed over the ranks the
 * outputs give the routed layer with normalised weights times route_scale; a
 * token with no expert on this rank has weight_scale 0 and contributes 0.
 *
 *   hidden [T, H] dtype;  router_probs [T, lc] probs_dtype (as the router
 *   wrote it: f32, bf16, or f16 with its -1e4 sentinel);  weight_scale [T] f32;
 *   w_gate_up [lc, N1, H], w_down [lc, H, F] (this rank's experts);
 *   b_gate_up [lc, N1] | NULL, b_down [lc, H] | NULL;  out [T, H] dtype;
 *   ws >= moe_workspace_size(T, H, F, lc, min(K, lc), dtype). */
moe_status moe_ffn_forward_local(const void* hidden, const void* router_probs,
                                 const float* weight_scale, const void* w_gate_up,
                                 const void* w_down, const void* b_gate_up, const void* b_down,
                                 int T, int H, int F, int lc, int K, moe_dtype dtype,
                                 moe_dtype probs_dtype, const moe_act_params* act, void* out,
                                 void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* moe_ffn_forward for a caller whose activations live in HOST memory:
 * hidden_host [T, H] dtype and logits_host [T, E] f32 are brought to device
 * staging space inside `ws`, the layer runs as in moe_ffn_forward, and the
 * result lands in out_host [T, H].  The activations come in on a side stream
 * of the library's (one per device, created on first use, joined back to
 * `stream` through events) while the logits are copied and the tokens routed
 * on `stream`; page-locked activations are read by a copy kernel, others by
 * cudaMemcpyAsync.  A page-locked out_host is written in place by the combine
 * (its writes overlap the combine's reads); otherwise the result is staged in
 * `ws` and copied back (always so on the indexed decode path).  All of it is
 * asynchronous on `stream`: out_host is valid after the stream is
 * synchronised.  Pageable buffers work, but their copies synchronise.
 * Weights, biases and expert_ids stay device pointers.  topk_weights and
 * topk_ids are not returned; the MoERouter outputs of the local slice, when
 * p->local_expert_count > 0, go to the DEVICE buffers router_probs
 * [T, local_expert_count] and weight_scale [T] as in moe_ffn_forward (both
 * required then, ignored otherwise).
 * ws >= moe_workspace_size_host(T, H, F, E, K, dtype). */
moe_status moe_ffn_forward_host(const void* hidden_host, const void* logits_host,
                                const void* w_gate_up, const void* w_down,
                                const float* correction_bias, const int32_t* expert_ids,
                                const void* b_gate_up, const void* b_down, int T, int H, int F,
                                int E, moe_dtype dtype, const moe_route_params* p,
                                const moe_act_params* act, void* out_host, void* router_probs,
                                float* weight_scale, void* ws, size_t ws_bytes,
                                cudaStream_t stream);

/* Workspace bytes of moe_ffn_forward_host: moe_workspace_size plus device
 * staging for hidden, logits and out. */
size_t moe_workspace_size_host(int T, int H, int F, int E, int K, moe_dtype dtype);

/* ------------------------------------------------------------------------ */
/* The grouped GEMM over any of its row layouts [TileOPs "MoE Operators",
 * MoEGroupedGemmFwdOp, layout table]:
 *   MOE_LAYOUT_PSUM     a [rows, K]; layout_metadata [E] segment END rows
 *                       (as moe_grouped_gemm_act / _down); out [rows, N]
 *   MOE_LAYOUT_PER_ROW  a [rows, K]; layout_metadata [rows] the expert of
 *                       every row, rows grouped by expert in ascending order
 *                       (not checked, as on the pages); out [rows, N]
 *   MOE_LAYOUT_MASKED   a [E, rows, K] (rows = max_m); layout_metadata [E]
 *                       valid rows of each expert, read as
 *                       min(max(m, 0), max_m); out [E, max_m, N], rows past
 *                       the count not written
 * w [E, N1, K] with N1 = 2N for a gated act (gate rows then up rows, or
 * interleaved for SwiGLU fusion 1), N otherwise; act NULL for the plain
 * product; bias [E, N1] | NULL, added before the activation and the cast.
 * ws >= moe_grouped_gemm_workspace_size(layout, rows, E). */
typedef enum moe_layout {
  MOE_LAYOUT_PSUM = 0,
  MOE_LAYOUT_PER_ROW = 1,
  MOE_LAYOUT_MASKED = 2
} moe_layout;
moe_status moe_grouped_gemm(const void* a, const void* w, const void* bias, int layout,
                            const int32_t* layout_metadata, int rows, int N, int K, int E,
                            moe_dtype dtype, const moe_act_params* act, void* out, void* ws,
                            size_t ws_bytes, cudaStream_t stream);
size_t moe_grouped_gemm_workspace_size(int layout, int rows, int E);

/* ------------------------------------------------------------------------ */
/* Block-scaled FP8 grouped GEMM over a masked slab [TileOPs, "MoE Operators",
 * MoEGroupedGemmFP8FwdOp]: out[g, :m_g] = a[g, :m_g] @ b[g]^T.
 *
 * a [E, max_m, K] and b [E, N, K] hold float8_e4m3fn codes (one byte each);
 * a_scale [E, max_m, K/128] f32 holds one scale per row and 128 columns of a,
 * b_scale [E, N/128, K/128] f32 one per 128 x 128 block of b; K and N are
 * multiples of 128.  Each 128-wide K block is contracted from the raw FP8
 * values, then multiplied by its two scales and added to an fp32
 * accumulator; out [E, max_m, N] is bf16.  m_g = layout_metadata[g] is read
 * as min(max(m_g, 0), max_m) on the device (counts are not checked on the
 * host); rows at or past m_g are not written (their contents are
 * undefined), and nothing outside out is.  a and b 16-byte aligned, the
 * scales 4-byte aligned (MOE_ERR_UNSUPPORTED otherwise); ws >=
 * MOE_STATUS_BYTES bytes.  E <= 1024. */
moe_status moe_grouped_gemm_fp8_masked(const void* a, const float* a_scale, const void* b,
                                       const float* b_scale, const int32_t* layout_metadata,
                                       int E, int max_m, int N, int K, void* out, void* ws,
                                       size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Shared expert [TileOPs, SharedExpertMLPFwdOp]: the dense gated MLP applied
 * to every token,
 *     out = down(silu(hidden @ gate^T) * (hidden @ up^T)),
 * both products accumulated in fp32, the gated activation rounded to the
 * operand dtype before the down projection.  Run as the grouped GEMMs over a
 * single segment of T rows (bf16 on the tensor cores when H % 8 == 0 and
 * S % 8 == 0 with 16-byte aligned buffers; the exact-fp32 SIMT GEMM
 * otherwise).
 *
 *   hidden [T, H] dtype;  w_gate_up [2S, H] dtype (the S gate rows, then the
 *   S up rows);  w_down [H, S] dtype;  out [T, H] dtype;
 *   ws >= moe_shared_expert_workspace_size(T, H, S, dtype) (its status word
 *   as in every call). */
moe_status moe_shared_expert_mlp(const void* hidden, const void* w_gate_up, const void* w_down,
                                 int T, int H, int S, moe_dtype dtype, void* out, void* ws,
                                 size_t ws_bytes, cudaStream_t stream);
size_t moe_shared_expert_workspace_size(int T, int H, int S, moe_dtype dtype);

/* Shared + routed MoE FFN [TileOPs, FusedMoESharedExpertFwdOp] with
 * tp_size 1: routed_out as moe_ffn_forward (no expert_ids, no biases, no
 * MoERouter outputs: p->local_expert_count must be 0, MOE_ERR_INVALID_ARG
 * otherwise; routed_scaling_factor scales the routed output only, once) and
 * shared_out
 * as moe_shared_expert_mlp, returned apart.  shared_w_gate_up and
 * shared_w_down are passed together (then shared_out is written) or both
 * NULL (shared_out untouched, S ignored).  The two halves run one after the
 * other on `stream` and share `ws`:
 * ws >= moe_workspace_size_shared(T, H, F, S, E, K, dtype). */
moe_status moe_ffn_forward_shared(const void* hidden, const void* logits, const void* w_gate_up,
                                  const void* w_down, const float* correction_bias,
                                  const void* shared_w_gate_up, const void* shared_w_down, int T,
                                  int H, int F, int S, int E, moe_dtype dtype,
                                  const moe_route_params* p, const moe_act_params* act,
                                  void* routed_out, void* shared_out, void* ws, size_t ws_bytes,
                                  cudaStream_t stream);
size_t moe_workspace_size_shared(int T, int H, int F, int S, int E, int K, moe_dtype dtype);

/* ------------------------------------------------------------------------ */
/* Sizes and status.  (The workspace query plays the role of the peak-memory
 * query of [ORT-MoE].) */

/* Bytes at the start of every workspace that hold the device status word
 * (and the grid-barrier counters of the fused route + permute launch and the
 * tile counters of the SM-pair grouped GEMM, which reset themselves after
 * every successful launch).  Clear them with moe_clear_status before a
 * workspace's first use and after an error. */
#define MOE_STATUS_BYTES 256

/* Workspace bytes moe_ffn_forward / moe_indexed_mlp need for these extents. */
size_t moe_workspace_size(int T, int H, int F, int E, int K, moe_dtype dtype);

/* Workspace bytes moe_permute needs for M = T*K routes over E experts. */
size_t moe_permute_workspace_size(int M, int E);

/* Zero the status word of `ws` (asynchronously, on `stream`). */
moe_status moe_clear_status(void* ws, cudaStream_t stream);

/* Synchronise `stream`, then read and clear the status word of `ws`:
 * MOE_OK, MOE_ERR_DEVICE (bad id / index met) or MOE_ERR_TIMEOUT.  On a
 * timeout the whole status area (MOE_STATUS_BYTES, with the counters a launch
 * that gave up may have left set) is cleared, so the workspace is ready for
 * the next call. */
moe_status moe_sync_status(void* ws, cudaStream_t stream);

/* Static text for a status code. */
const char* moe_status_string(moe_status s);

/* Number of this library's kernel launches issued since load (all entry
 * points, all streams); lets a caller count device work per call. */
uint64_t moe_launch_count(void);

/* Verification switch: nonzero routes every grouped GEMM (bf16 included) to
 * the exact-fp32 SIMT kernel instead of the tcgen05 kernel; returns the
 * previous setting.  Process-wide; not meant to change while calls are in
 * flight. */
int moe_set_gemm_simt(int enable);

/* Stage profile (a tracing aid; no counterpart on the pages): with
 * MOE_PROFILE=1 in the environment when the library loads, every forward
 * brackets its stages (route_permute or route, permute, gate_up, down,
 * combine, or indexed_mlp) with CUDA events on the caller's stream.  This call
 * waits for the recorded events, writes one line per stage, "name count
 * total_us", into buf (NUL-terminated, truncated to buf_bytes - 1), drops the
 * records and returns the length of the full text.  Without MOE_PROFILE
 * nothing is recorded and the text is empty.  The events sit between the
 * launches, so a profiled forward runs its launches without overlap. */
int moe_profile_report(char* buf, size_t buf_bytes);

/* Test hook, off by default (no counterpart on the pages; it exists so that
 * a test can make a bounded device wait run out without faulting or hanging
 * anything).  With enable != 0, both grid barriers of the fused route +
 * index-map launch (moe_route_permute, and the first launch of the forward
 * when E <= 512) wait for one arrival more than the grid provides and give up
 * after limit_ns instead of 2 s: every CTA then latches MOE_ERR_TIMEOUT in the
 * workspace status word and returns, leaving the index maps unwritten and the
 * barrier counters as they stand (moe_clear_status resets both the status
 * word and the counters).  enable = 0 restores the normal barriers and the
 * 2 s limit.  Process-wide, read when a call is issued; returns the previous
 * enable state. */
int moe_test_force_wait_timeout(int enable, long long limit_ns);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
