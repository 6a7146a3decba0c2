"""Thin Python binding over libmoe.so (argument marshalling only).

Every function here has the name of the C entry point it calls, takes CUDA
tensors, allocates missing outputs and workspaces with torch, and calls the C
ABI on the current torch stream.  All arithmetic runs in the library's CUDA
kernels; there is no Python or CPU fallback, and every call raises if the
library is missing or the device is not a CUDA device.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_OVERLAP, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, \
    MOE_ERR_TIMEOUT, MOE_ERR_DEVICE, MOE_ERR_WORKSPACE = range(8)
MOE_F32, MOE_BF16, MOE_F16 = 0, 1, 2
MOE_SCORING_SOFTMAX, MOE_SCORING_SIGMOID, MOE_SCORING_SQRT_SOFTPLUS = 0, 1, 2
MOE_ACT_SILU_AND_MUL, MOE_ACT_SWIGLU, MOE_ACT_IDENTITY, MOE_ACT_GELU_AND_MUL = 0, 1, 2, 3
MOE_ACT_RELU, MOE_ACT_GELU, MOE_ACT_SILU = 4, 5, 6
MOE_STATUS_BYTES = 256
MOE_LAYOUT_PSUM, MOE_LAYOUT_PER_ROW, MOE_LAYOUT_MASKED = 0, 1, 2

# C entry points and their argument types (mirrors include/moe.h)
_vp, _i, _i64, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, \
    ctypes.c_size_t


class RouteParams(ctypes.Structure):
    _fields_ = [("top_k", ctypes.c_int32), ("scoring", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("num_expert_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float),
                ("local_expert_start", ctypes.c_int32), ("local_expert_count", ctypes.c_int32),
                ("route_scale", ctypes.c_float), ("dtype", ctypes.c_int32)]


class ActParams(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("swiglu_fusion", ctypes.c_int32),
                ("limit", ctypes.c_float), ("alpha", ctypes.c_float), ("beta", ctypes.c_float)]


_SIGNATURES = {
    "moe_route": [_vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp],
    "moe_permute": [_vp, _i, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _sz, _vp],
    "moe_route_permute": [_vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                          _sz, _vp],
    "moe_permute_gather": [_vp, _i, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _sz, _vp],
    "moe_permute_align": [_vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp],
    "moe_grouped_gemm": [_vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _sz, _vp],
    "moe_grouped_gemm_workspace_size": [_i, _i, _i],
    "moe_permute_align_workspace_size": [_i, _i, _i],
    "moe_grouped_gemm_act": [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _sz, _vp],
    "moe_grouped_gemm_act_split": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp,
                                   _vp, _sz, _vp],
    "moe_ffn_forward_split": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i,
                              _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp],
    "moe_grouped_gemm_act_gathered": [_vp, _i, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp,
                                      _vp, _vp, _sz, _vp],
    "moe_grouped_gemm_down": [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _sz, _vp],
    "moe_combine": [_vp, _vp, _vp, _i, _i, _i, _i, _f, _vp, _vp],
    "swiglu": [_vp, _vp, _i64, _i, _i, _i, _f, _f, _f, _vp, _vp],
    "moe_indexed_mlp": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp],
    "moe_ffn_forward": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp,
                        _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp],
    "moe_ffn_forward_host": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp,
                             _vp, _vp, _vp, _vp, _vp, _sz, _vp],
    "moe_shared_expert_mlp": [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _sz, _vp],
    "moe_ffn_forward_local": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                              _vp, _vp, _vp, _sz, _vp],
    "moe_grouped_gemm_fp8_masked": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _sz, _vp],
    "moe_shared_expert_workspace_size": [_i, _i, _i, _i],
    "moe_ffn_forward_shared": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp,
                               _vp, _vp, _vp, _vp, _sz, _vp],
    "moe_workspace_size_shared": [_i, _i, _i, _i, _i, _i, _i],
    "moe_workspace_size": [_i, _i, _i, _i, _i, _i],
    "moe_workspace_size_host": [_i, _i, _i, _i, _i, _i],
    "moe_permute_workspace_size": [_i, _i],
    "moe_clear_status": [_vp, _vp],
    "moe_sync_status": [_vp, _vp],
    "moe_status_string": [_i],
    "moe_launch_count": [],
    "moe_set_gemm_simt": [_i],
    "moe_test_force_wait_timeout": [_i, ctypes.c_longlong],
    "moe_profile_report": [ctypes.c_char_p, _sz],
}
_RESTYPES = {"moe_workspace_size": _sz, "moe_permute_workspace_size": _sz,
             "moe_workspace_size_host": _sz, "moe_shared_expert_workspace_size": _sz,
             "moe_workspace_size_shared": _sz, "moe_permute_align_workspace_size": _sz,
             "moe_grouped_gemm_workspace_size": _sz,
             "moe_status_string": ctypes.c_char_p, "moe_launch_count": ctypes.c_uint64}

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmoe.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m mixture_experts_ffn_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, args in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = _RESTYPES.get(name, ctypes.c_int)
        _lib = lib
    return _lib


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = load_library().moe_status_string(status).decode()
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoEError(fn, status)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    if t.dtype == torch.float32:
        return MOE_F32
    if t.dtype == torch.float16:
        return MOE_F16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("libmoe takes CUDA tensors only")
            if not t.is_contiguous():
                raise ValueError("libmoe takes contiguous tensors only")


def _ws(nbytes: int, device) -> torch.Tensor:
    """A fresh workspace with a cleared status word (torch's caching allocator
    returns 512-byte aligned blocks)."""
    ws = torch.empty(max(nbytes, MOE_STATUS_BYTES), dtype=torch.uint8, device=device)
    ws[:MOE_STATUS_BYTES].zero_()
    return ws


def route_params(top_k, scoring="softmax", renormalize=True, num_expert_group=1, topk_group=1,
                 routed_scaling_factor=1.0, local_expert_start=0, local_expert_count=0,
                 route_scale=1.0) -> RouteParams:
    sc = {"softmax": MOE_SCORING_SOFTMAX, "sigmoid": MOE_SCORING_SIGMOID,
          "sqrt_softplus": MOE_SCORING_SQRT_SOFTPLUS}.get(scoring, scoring)
    return RouteParams(top_k, sc, int(bool(renormalize)), num_expert_group, topk_group,
                       routed_scaling_factor, local_expert_start, local_expert_count, route_scale,
                       MOE_F32)


def _rp(p: RouteParams, logits) -> RouteParams:
    """A copy of p whose MoERouter type T (logits and router_probs) is the
    logits tensor's dtype."""
    q = RouteParams.from_buffer_copy(p)
    q.dtype = _dt(logits)
    return q


def act_params(kind=MOE_ACT_SILU_AND_MUL, swiglu_fusion=2, limit=0.0, alpha=1.0,
               beta=0.0) -> ActParams:
    return ActParams(kind, swiglu_fusion, limit, alpha, beta)


# ----------------------------------------------------------------- entry points
def moe_workspace_size(T, H, F, E, K, dtype=MOE_BF16) -> int:
    return load_library().moe_workspace_size(T, H, F, E, K, dtype)


def moe_permute_workspace_size(M, E) -> int:
    return load_library().moe_permute_workspace_size(M, E)


def moe_route(logits, p: RouteParams, correction_bias=None, expert_ids=None, topk_weights=None,
              topk_ids=None, router_probs=None, weight_scale=None):
    """Router; returns (topk_weights, topk_ids, router_probs, weight_scale)."""
    lib = load_library()
    _cuda(logits, correction_bias, expert_ids)
    T, E = logits.shape
    dev = logits.device
    if topk_weights is None:
        topk_weights = torch.empty((T, p.top_k), dtype=torch.float32, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty((T, p.top_k), dtype=torch.int32, device=dev)
    if p.local_expert_count > 0:
        if router_probs is None:
            router_probs = torch.empty((T, p.local_expert_count), dtype=logits.dtype, device=dev)
        if weight_scale is None:
            weight_scale = torch.empty((T,), dtype=torch.float32, device=dev)
    _check("moe_route", lib.moe_route(_p(logits), _p(correction_bias), _p(expert_ids), T, E,
                                      ctypes.byref(_rp(p, logits)), _p(topk_weights), _p(topk_ids),
                                      _p(router_probs), _p(weight_scale), _stream()))
    return topk_weights, topk_ids, router_probs, weight_scale


def moe_permute(topk_ids, E: int, hidden=None, ws=None, with_gather=True):
    """Returns dict(expert_input, seg_end, row_to_route, route_to_row, ws)."""
    lib = load_library()
    _cuda(topk_ids, hidden)
    T, K = topk_ids.shape
    M = T * K
    dev = topk_ids.device
    H = hidden.shape[1] if hidden is not None else 0
    dt = _dt(hidden) if hidden is not None else MOE_BF16
    xin = None
    if with_gather and hidden is not None:
        xin = torch.empty((M, H), dtype=hidden.dtype, device=dev)
    seg_end = torch.empty((E,), dtype=torch.int32, device=dev)
    r2r = torch.empty((M,), dtype=torch.int32, device=dev)
    route_to_row = torch.empty((M,), dtype=torch.int32, device=dev)
    need = lib.moe_permute_workspace_size(M, E)
    if ws is None:
        ws = _ws(need, dev)
    _check("moe_permute", lib.moe_permute(_p(hidden if xin is not None else None), dt,
                                          _p(topk_ids), T, H, E, K, _p(xin), _p(seg_end), _p(r2r),
                                          _p(route_to_row), _p(ws), ws.numel(), _stream()))
    return {"expert_input": xin, "seg_end": seg_end, "row_to_route": r2r,
            "route_to_row": route_to_row, "ws": ws}


def moe_grouped_gemm(a, w, layout: int, layout_metadata, N: int, act=None, bias=None, out=None,
                     ws=None):
    """The grouped GEMM over a row layout (MOE_LAYOUT_PSUM / PER_ROW: a [M, K],
    out [M, N]; MASKED: a [E, max_m, K], out [E, max_m, N]); w [E, N1, K]."""
    lib = load_library()
    _cuda(a, w, bias, layout_metadata)
    E, _, K = w.shape
    masked = layout == MOE_LAYOUT_MASKED
    rows = a.shape[1] if masked else a.shape[0]
    if out is None:
        shape = (E, rows, N) if masked else (rows, N)
        out = torch.empty(shape, dtype=a.dtype, device=a.device)
    if ws is None:
        ws = _ws(lib.moe_grouped_gemm_workspace_size(layout, rows, E), a.device)
    _check("moe_grouped_gemm",
           lib.moe_grouped_gemm(_p(a), _p(w), _p(bias), layout, _p(layout_metadata), rows, N, K, E,
                                _dt(a), None if act is None else ctypes.byref(act), _p(out),
                                _p(ws), ws.numel(), _stream()))
    return out


def moe_permute_align(topk_ids, E: int, block_size: int = 64, ws=None):
    """Padded layout: returns (sorted_token_ids, expert_ids, num_tokens_post_pad)."""
    lib = load_library()
    _cuda(topk_ids)
    T, K = topk_ids.shape
    dev = topk_ids.device
    L = T * K + (E + 1) * (block_size - 1)
    sorted_ids = torch.empty((L,), dtype=torch.int32, device=dev)
    expert_ids = torch.empty(((L + block_size - 1) // block_size,), dtype=torch.int32, device=dev)
    npp = torch.empty((1,), dtype=torch.int32, device=dev)
    if ws is None:
        ws = _ws(lib.moe_permute_align_workspace_size(T, K, E), dev)
    _check("moe_permute_align",
           lib.moe_permute_align(_p(topk_ids), T, K, E, block_size, _p(sorted_ids),
                                 _p(expert_ids), _p(npp), _p(ws), ws.numel(), _stream()))
    return sorted_ids, expert_ids, npp


def moe_permute_gather(hidden, seg_end, row_to_route, K: int, out=None, ws=None):
    """The permuted copy of the activations from index maps already built:
    out[row] = hidden[row_to_route[row] // K] for the rows below seg_end[-1]."""
    lib = load_library()
    _cuda(hidden, seg_end, row_to_route)
    T, H = hidden.shape
    E = seg_end.numel()
    if out is None:
        out = torch.empty((T * K, H), dtype=hidden.dtype, device=hidden.device)
    if ws is None:
        ws = _ws(MOE_STATUS_BYTES, hidden.device)
    _check("moe_permute_gather",
           lib.moe_permute_gather(_p(hidden), _dt(hidden), _p(seg_end), _p(row_to_route), T, H, E,
                                  K, _p(out), _p(ws), ws.numel(), _stream()))
    return out


def moe_route_permute(logits, p: RouteParams, correction_bias=None, expert_ids=None, ws=None):
    """moe_route then the index maps of moe_permute, in one launch; returns
    (topk_weights, topk_ids, router_probs, weight_scale, maps) with maps =
    dict(seg_end, row_to_route, route_to_row, ws)."""
    lib = load_library()
    _cuda(logits, correction_bias, expert_ids)
    T, E = logits.shape
    K = p.top_k
    dev = logits.device
    tw = torch.empty((T, K), dtype=torch.float32, device=dev)
    ti = torch.empty((T, K), dtype=torch.int32, device=dev)
    probs = wsc = None
    if p.local_expert_count > 0:
        probs = torch.empty((T, p.local_expert_count), dtype=logits.dtype, device=dev)
        wsc = torch.empty((T,), dtype=torch.float32, device=dev)
    seg_end = torch.empty((E,), dtype=torch.int32, device=dev)
    r2r = torch.empty((T * K,), dtype=torch.int32, device=dev)
    route_to_row = torch.empty((T * K,), dtype=torch.int32, device=dev)
    if ws is None:
        ws = _ws(lib.moe_permute_workspace_size(T * K, E), dev)
    _check("moe_route_permute",
           lib.moe_route_permute(_p(logits), _p(correction_bias), _p(expert_ids), T, E,
                                 ctypes.byref(_rp(p, logits)), _p(tw), _p(ti), _p(probs), _p(wsc),
                                 _p(seg_end),
                                 _p(r2r), _p(route_to_row), _p(ws), ws.numel(), _stream()))
    return tw, ti, probs, wsc, {"seg_end": seg_end, "row_to_route": r2r,
                                "route_to_row": route_to_row, "ws": ws}


def moe_grouped_gemm_act(a, w_gate_up, seg_end, F: int, act: ActParams, b_gate_up=None, out=None,
                         ws=None):
    lib = load_library()
    _cuda(a, w_gate_up, seg_end, b_gate_up)
    M, Hk = a.shape
    E = w_gate_up.shape[0]
    if out is None:
        out = torch.empty((M, F), dtype=a.dtype, device=a.device)
    if ws is None:
        ws = _ws(MOE_STATUS_BYTES, a.device)
    _check("moe_grouped_gemm_act",
           lib.moe_grouped_gemm_act(_p(a), _p(w_gate_up), _p(b_gate_up), _p(seg_end), M, F, Hk, E,
                                    _dt(a), ctypes.byref(act), _p(out), _p(ws), ws.numel(),
                                    _stream()))
    return out


def moe_grouped_gemm_act_split(a, w_gate, w_up, seg_end, act: ActParams, b_gate=None, b_up=None,
                               out=None, ws=None):
    """moe_grouped_gemm_act with the gate and up projections in two tensors
    w_gate, w_up [E, F, Hk] (SwiGLU fusion 0); returns out [M, F]."""
    lib = load_library()
    _cuda(a, w_gate, w_up, seg_end, b_gate, b_up)
    M, Hk = a.shape
    E, F, _ = w_gate.shape
    if out is None:
        out = torch.empty((M, F), dtype=a.dtype, device=a.device)
    if ws is None:
        ws = _ws(MOE_STATUS_BYTES, a.device)
    _check("moe_grouped_gemm_act_split",
           lib.moe_grouped_gemm_act_split(_p(a), _p(w_gate), _p(w_up), _p(b_gate), _p(b_up),
                                          _p(seg_end), M, F, Hk, E, _dt(a), ctypes.byref(act),
                                          _p(out), _p(ws), ws.numel(), _stream()))
    return out


def moe_grouped_gemm_act_gathered(hidden, row_to_route, top_k: int, w_gate_up, seg_end, F: int,
                                  act: ActParams, b_gate_up=None, out=None, ws=None):
    """moe_grouped_gemm_act with row m of the operand read as
    hidden[row_to_route[m] // top_k] (no permuted copy of the activations)."""
    lib = load_library()
    _cuda(hidden, row_to_route, w_gate_up, seg_end, b_gate_up)
    T, H = hidden.shape
    M = row_to_route.numel()
    E = w_gate_up.shape[0]
    if out is None:
        out = torch.empty((M, F), dtype=hidden.dtype, device=hidden.device)
    if ws is None:
        ws = _ws(MOE_STATUS_BYTES, hidden.device)
    _check("moe_grouped_gemm_act_gathered",
           lib.moe_grouped_gemm_act_gathered(_p(hidden), T, _p(row_to_route), top_k,
                                             _p(w_gate_up), _p(b_gate_up), _p(seg_end), M, F, H,
                                             E, _dt(hidden), ctypes.byref(act), _p(out), _p(ws),
                                             ws.numel(), _stream()))
    return out


def moe_grouped_gemm_down(a, w_down, seg_end, b_down=None, out=None, ws=None):
    lib = load_library()
    _cuda(a, w_down, seg_end, b_down)
    M, F = a.shape
    E, H, _ = w_down.shape
    if out is None:
        out = torch.empty((M, H), dtype=a.dtype, device=a.device)
    if ws is None:
        ws = _ws(MOE_STATUS_BYTES, a.device)
    _check("moe_grouped_gemm_down",
           lib.moe_grouped_gemm_down(_p(a), _p(w_down), _p(b_down), _p(seg_end), M, H, F, E,
                                     _dt(a), _p(out), _p(ws), ws.numel(), _stream()))
    return out


def moe_combine(expert_out, topk_weights, route_to_row, scale=1.0, out=None):
    lib = load_library()
    _cuda(expert_out, topk_weights, route_to_row)
    T, K = topk_weights.shape
    H = expert_out.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=expert_out.dtype, device=expert_out.device)
    _check("moe_combine", lib.moe_combine(_p(expert_out), _p(topk_weights), _p(route_to_row), T, K,
                                          H, _dt(expert_out), scale, _p(out), _stream()))
    return out


def swiglu(gate, up=None, swiglu_fusion=2, limit=0.0, alpha=1.0, beta=0.0, out=None):
    """The standalone SwiGLU op.  gate [R, 2I] (up None) or gate, up [R, I]."""
    lib = load_library()
    _cuda(gate, up)
    R = gate.shape[0]
    I = gate.shape[1] if up is not None else gate.shape[1] // 2
    if out is None:
        out = torch.empty((R, I), dtype=gate.dtype, device=gate.device)
    _check("swiglu", lib.swiglu(_p(gate), _p(up), R, I, _dt(gate), swiglu_fusion, limit, alpha,
                                beta, _p(out), _stream()))
    return out


def moe_indexed_mlp(hidden, w_gate_up, w_down, topk_weights, topk_ids, scale=1.0, out=None,
                    ws=None):
    lib = load_library()
    _cuda(hidden, w_gate_up, w_down, topk_weights, topk_ids)
    T, H = hidden.shape
    E, H2, F = w_down.shape
    K = topk_ids.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=hidden.dtype, device=hidden.device)
    if ws is None:
        ws = _ws(lib.moe_workspace_size(T, H, F, E, K, MOE_BF16), hidden.device)
    _check("moe_indexed_mlp",
           lib.moe_indexed_mlp(_p(hidden), _p(w_gate_up), _p(w_down), _p(topk_weights),
                               _p(topk_ids), T, H, F, E, K, scale, _p(out), _p(ws), ws.numel(),
                               _stream()))
    return out


def moe_ffn_forward(hidden, logits, w_gate_up, w_down, p: RouteParams, act: ActParams,
                    correction_bias=None, expert_ids=None, b_gate_up=None, b_down=None, out=None,
                    topk_weights_out=None, topk_ids_out=None, router_probs=None,
                    weight_scale=None, ws=None):
    """The whole routed MoE FFN forward; returns ``out`` [T, H]."""
    lib = load_library()
    _cuda(hidden, logits, w_gate_up, w_down, correction_bias, expert_ids, b_gate_up, b_down)
    T, H = hidden.shape
    E, _, F = w_down.shape
    if out is None:
        out = torch.empty_like(hidden)
    if ws is None:
        ws = _ws(lib.moe_workspace_size(T, H, F, E, p.top_k, _dt(hidden)), hidden.device)
    _check("moe_ffn_forward",
           lib.moe_ffn_forward(_p(hidden), _p(logits), _p(w_gate_up), _p(w_down),
                               _p(correction_bias), _p(expert_ids), _p(b_gate_up), _p(b_down), T,
                               H, F, E, _dt(hidden), ctypes.byref(_rp(p, logits)),
                               ctypes.byref(act), _p(out),
                               _p(topk_weights_out), _p(topk_ids_out), _p(router_probs),
                               _p(weight_scale), _p(ws), ws.numel(), _stream()))
    return out


def moe_ffn_forward_split(hidden, logits, w_gate, w_up, w_down, p: RouteParams, act: ActParams,
                          correction_bias=None, expert_ids=None, b_gate=None, b_up=None,
                          b_down=None, out=None, topk_weights_out=None, topk_ids_out=None,
                          router_probs=None, weight_scale=None, ws=None):
    """moe_ffn_forward with the gate and up projections in two tensors
    w_gate, w_up [E, F, H] (SwiGLU fusion 0); returns ``out`` [T, H]."""
    lib = load_library()
    _cuda(hidden, logits, w_gate, w_up, w_down, correction_bias, expert_ids, b_gate, b_up,
          b_down)
    T, H = hidden.shape
    E, _, F = w_down.shape
    if out is None:
        out = torch.empty_like(hidden)
    if ws is None:
        ws = _ws(lib.moe_workspace_size(T, H, F, E, p.top_k, _dt(hidden)), hidden.device)
    _check("moe_ffn_forward_split",
           lib.moe_ffn_forward_split(_p(hidden), _p(logits), _p(w_gate), _p(w_up), _p(w_down),
                                     _p(correction_bias), _p(expert_ids), _p(b_gate), _p(b_up),
                                     _p(b_down), T, H, F, E, _dt(hidden),
                                     ctypes.byref(_rp(p, logits)),
                                     ctypes.byref(act), _p(out), _p(topk_weights_out),
                                     _p(topk_ids_out), _p(router_probs), _p(weight_scale),
                                     _p(ws), ws.numel(), _stream()))
    return out


def moe_grouped_gemm_fp8_masked(a, a_scale, b, b_scale, layout_metadata, out=None, ws=None):
    """Block-scaled FP8 GEMM per expert over a masked slab: a [E, max_m, K] and
    b [E, N, K] float8_e4m3fn (or their uint8 codes), a_scale [E, max_m, K/128]
    and b_scale [E, N/128, K/128] float32, layout_metadata [E] int32 valid row
    counts; returns out [E, max_m, N] bf16 (rows past a count undefined)."""
    lib = load_library()
    _cuda(a, a_scale, b, b_scale, layout_metadata)
    E, max_m, K = a.shape
    N = b.shape[1]
    if out is None:
        out = torch.empty((E, max_m, N), dtype=torch.bfloat16, device=a.device)
    if ws is None:
        ws = _ws(MOE_STATUS_BYTES, a.device)
    _check("moe_grouped_gemm_fp8_masked",
           lib.moe_grouped_gemm_fp8_masked(_p(a), _p(a_scale), _p(b), _p(b_scale),
                                           _p(layout_metadata), E, max_m, N, K, _p(out), _p(ws),
                                           ws.numel(), _stream()))
    return out


def moe_shared_expert_workspace_size(T, H, S, dtype=MOE_BF16) -> int:
    return load_library().moe_shared_expert_workspace_size(T, H, S, dtype)


def moe_workspace_size_shared(T, H, F, S, E, K, dtype=MOE_BF16) -> int:
    return load_library().moe_workspace_size_shared(T, H, F, S, E, K, dtype)


def moe_shared_expert_mlp(hidden, w_gate_up, w_down, out=None, ws=None):
    """Shared expert: down(silu(hidden @ gate^T) * (hidden @ up^T)) for every
    token; w_gate_up [2S, H] (gate rows then up rows), w_down [H, S]."""
    lib = load_library()
    _cuda(hidden, w_gate_up, w_down)
    T, H = hidden.shape
    S = w_down.shape[1]
    if out is None:
        out = torch.empty_like(hidden)
    if ws is None:
        ws = _ws(lib.moe_shared_expert_workspace_size(T, H, S, _dt(hidden)), hidden.device)
    _check("moe_shared_expert_mlp",
           lib.moe_shared_expert_mlp(_p(hidden), _p(w_gate_up), _p(w_down), T, H, S, _dt(hidden),
                                     _p(out), _p(ws), ws.numel(), _stream()))
    return out


def moe_ffn_forward_shared(hidden, logits, w_gate_up, w_down, p: RouteParams, act: ActParams,
                           correction_bias=None, shared_w_gate_up=None, shared_w_down=None,
                           routed_out=None, shared_out=None, ws=None):
    """Shared + routed MoE FFN; returns (shared_out or None, routed_out)."""
    lib = load_library()
    _cuda(hidden, logits, w_gate_up, w_down, correction_bias, shared_w_gate_up, shared_w_down)
    T, H = hidden.shape
    E, _, F = w_down.shape
    S = shared_w_down.shape[1] if shared_w_down is not None else 0
    if routed_out is None:
        routed_out = torch.empty_like(hidden)
    if shared_w_gate_up is not None and shared_out is None:
        shared_out = torch.empty_like(hidden)
    if ws is None:
        need = (lib.moe_workspace_size_shared(T, H, F, S, E, p.top_k, _dt(hidden)) if S else
                lib.moe_workspace_size(T, H, F, E, p.top_k, _dt(hidden)))
        ws = _ws(need, hidden.device)
    _check("moe_ffn_forward_shared",
           lib.moe_ffn_forward_shared(_p(hidden), _p(logits), _p(w_gate_up), _p(w_down),
                                      _p(correction_bias), _p(shared_w_gate_up),
                                      _p(shared_w_down), T, H, F, S, E, _dt(hidden),
                                      ctypes.byref(_rp(p, logits)), ctypes.byref(act),
                                      _p(routed_out),
                                      _p(shared_out if shared_w_gate_up is not None else None),
                                      _p(ws), ws.numel(), _stream()))
    return (shared_out if shared_w_gate_up is not None else None), routed_out


def moe_ffn_forward_local(hidden, router_probs, weight_scale, w_gate_up, w_down, K: int,
                          act: ActParams, b_gate_up=None, b_down=None, out=None, ws=None):
    """The expert-parallel rank's layer from its MoERouter outputs
    (router_probs [T, lc], weight_scale [T]) and its lc experts' weights."""
    lib = load_library()
    _cuda(hidden, router_probs, weight_scale, w_gate_up, w_down, b_gate_up, b_down)
    T, H = hidden.shape
    lc, _, F = w_down.shape
    if out is None:
        out = torch.empty_like(hidden)
    if ws is None:
        ws = _ws(lib.moe_workspace_size(T, H, F, lc, min(K, lc), _dt(hidden)), hidden.device)
    _check("moe_ffn_forward_local",
           lib.moe_ffn_forward_local(_p(hidden), _p(router_probs), _p(weight_scale),
                                     _p(w_gate_up), _p(w_down), _p(b_gate_up), _p(b_down), T, H,
                                     F, lc, K, _dt(hidden), _dt(router_probs), ctypes.byref(act),
                                     _p(out), _p(ws),
                                     ws.numel(), _stream()))
    return out


def moe_workspace_size_host(T, H, F, E, K, dtype=MOE_BF16) -> int:
    return load_library().moe_workspace_size_host(T, H, F, E, K, dtype)


def moe_ffn_forward_host(hidden_host, logits_host, w_gate_up, w_down, p: RouteParams,
                         act: ActParams, out_host, ws, correction_bias=None, expert_ids=None,
                         b_gate_up=None, b_down=None, router_probs=None, weight_scale=None):
    """moe_ffn_forward with hidden / logits / out in host memory (pinned for
    asynchronous copies); asynchronous on the current stream.  router_probs /
    weight_scale (device tensors) receive the MoERouter slice outputs when
    ``p`` has a local slice."""
    lib = load_library()
    _cuda(w_gate_up, w_down, correction_bias, expert_ids, b_gate_up, b_down, ws, router_probs,
          weight_scale)
    for t in (hidden_host, logits_host, out_host):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("moe_ffn_forward_host takes contiguous host tensors")
    T, H = hidden_host.shape
    E, _, F = w_down.shape
    _check("moe_ffn_forward_host",
           lib.moe_ffn_forward_host(_p(hidden_host), _p(logits_host), _p(w_gate_up), _p(w_down),
                                    _p(correction_bias), _p(expert_ids), _p(b_gate_up),
                                    _p(b_down), T, H, F, E, _dt(hidden_host),
                                    ctypes.byref(_rp(p, logits_host)),
                                    ctypes.byref(act), _p(out_host), _p(router_probs),
                                    _p(weight_scale), _p(ws), ws.numel(), _stream()))
    return out_host


def moe_clear_status(ws):
    _check("moe_clear_status", load_library().moe_clear_status(_p(ws), _stream()))


def moe_sync_status(ws) -> int:
    """Synchronise the current stream and return (and clear) the status word."""
    return load_library().moe_sync_status(_p(ws), _stream())


def moe_launch_count() -> int:
    return load_library().moe_launch_count()


def moe_set_gemm_simt(enable: bool) -> bool:
    return bool(load_library().moe_set_gemm_simt(int(bool(enable))))


def moe_profile_report() -> dict:
    """Per-stage totals of the forwards recorded since the last report (with
    MOE_PROFILE=1 set before the library loads): {stage: (count, total_us)}."""
    lib = load_library()
    buf = ctypes.create_string_buffer(1 << 16)
    lib.moe_profile_report(buf, len(buf))
    out = {}
    for line in buf.value.decode().splitlines():
        name, count, us = line.split()
        out[name] = (int(count), float(us))
    return out


def moe_test_force_wait_timeout(enable: bool, limit_ns: int = 50_000_000) -> bool:
    """Test hook: make the fused route launch's grid barriers wait for an
    arrival that never comes and give up after ``limit_ns`` (see moe.h)."""
    return bool(load_library().moe_test_force_wait_timeout(int(bool(enable)), int(limit_ns)))


def config_params(cfg):
    """(RouteParams, ActParams) of a synthetic workload recipe (see synth.MoEConfig)."""
    p = route_params(cfg.K, cfg.scoring, cfg.renormalize, cfg.G, cfg.TG, cfg.rsf,
                     cfg.local_start, cfg.local_count, cfg.route_scale)
    a = act_params(cfg.act, cfg.swiglu_fusion, cfg.limit, cfg.alpha, cfg.beta)
    return p, a
