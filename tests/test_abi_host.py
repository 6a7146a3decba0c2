"""Host-only checks of the C ABI: the library loads, exports every function
include/moe.h declares, sizes workspaces, and rejects invalid calls before any
launch.  Calls here pass placeholder device addresses that are never
dereferenced, so they run only where no GPU is visible (on a GPU machine the
same rejections are covered by the GPU tests with real buffers)."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_ffn_gb300 import build, moe

    build.build()
    return moe.load_library()


def test_library_exports_every_declared_function(lib):
    names = _declared_functions()
    assert "moe_ffn_forward" in names and "swiglu" in names and len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_sizes(lib):
    from mixture_experts_ffn_gb300 import moe

    a = moe.moe_workspace_size(4096, 2048, 768, 128, 8, moe.MOE_BF16)
    M = 4096 * 8
    # the staged intermediates dominate: expert_input + y [M, H] and act [M, F]
    assert a >= M * (2048 * 2 * 2 + 768 * 2)
    assert a % 256 == 0
    assert moe.moe_workspace_size(-1, 1, 1, 1, 1, 1) == 0
    assert moe.moe_permute_workspace_size(M, 128) >= 256 + 32 * 128 * 4
    assert lib.moe_status_string(0) == b"ok"
    assert b"overlap" in lib.moe_status_string(2)
    assert moe.moe_launch_count() >= 0


nogpu = pytest.mark.skipif(torch.cuda.is_available(), reason="placeholder pointers: CPU only")

# placeholder device addresses, 4 KiB apart unless a test wants them to overlap
A = lambda i: ctypes.c_void_p(0x7F0000000000 + i * (1 << 30))  # noqa: E731


@nogpu
def test_route_rejects_bad_arguments(lib):
    from mixture_experts_ffn_gb300 import moe

    def call(p, T=8, E=16, bias=None, probs=None, wscale=None):
        return lib.moe_route(A(0), bias, None, T, E, ctypes.byref(p), A(1), A(2), probs, wscale,
                             None)

    ok = moe.route_params(4, "softmax")
    bad = [
        moe.route_params(0),                                   # K < 1
        moe.route_params(17),                                  # K > E
        moe.route_params(4, scoring=7),                        # unknown scoring
        moe.route_params(4, num_expert_group=3),               # G does not divide E
        moe.route_params(4, num_expert_group=4, topk_group=5), # TG > G
        moe.route_params(4, num_expert_group=8, topk_group=1), # TG * E / G < K
        moe.route_params(4, routed_scaling_factor=0.0),        # rsf <= 0
        moe.route_params(4, local_expert_start=10, local_expert_count=8),  # slice outside E
    ]
    for p in bad:
        assert call(p) == moe.MOE_ERR_INVALID_ARG
    # a correction bias needs sigmoid scoring
    assert call(ok, bias=A(3)) == moe.MOE_ERR_INVALID_ARG
    # MoERouter outputs: both or neither, and only with a local slice
    p = moe.route_params(4, local_expert_start=0, local_expert_count=8)
    assert call(p, probs=A(4)) == moe.MOE_ERR_INVALID_ARG
    assert call(ok, probs=A(4), wscale=A(5)) == moe.MOE_ERR_INVALID_ARG
    assert call(ok, E=2000) == moe.MOE_ERR_INVALID_ARG
    # T == 0 is a no-op and launches nothing
    assert call(ok, T=0) == moe.MOE_OK


@nogpu
def test_overlap_is_rejected_before_launch(lib):
    from mixture_experts_ffn_gb300 import moe

    p = moe.route_params(4)
    base = 0x7F0000000000
    logits = ctypes.c_void_p(base)
    # topk_weights placed inside the logits buffer [8, 16] f32 = 512 bytes
    r = lib.moe_route(logits, None, None, 8, 16, ctypes.byref(p), ctypes.c_void_p(base + 256),
                      A(2), None, None, None)
    assert r == moe.MOE_ERR_OVERLAP
    # outputs overlapping each other
    r = lib.moe_route(logits, None, None, 8, 16, ctypes.byref(p), A(1),
                      ctypes.c_void_p(A(1).value + 64), None, None, None)
    assert r == moe.MOE_ERR_OVERLAP
    # combine: out overlapping expert_out; disjoint views of one allocation are fine only
    # when they do not intersect -- here they do
    r = lib.moe_combine(A(0), A(1), A(2), 4, 2, 64, moe.MOE_BF16, 1.0, ctypes.c_void_p(base + 128),
                        None)
    assert r == moe.MOE_ERR_OVERLAP
    # swiglu: out inside gate
    r = lib.swiglu(A(0), None, 4, 8, moe.MOE_F32, 2, 7.0, 1.0, 0.0, ctypes.c_void_p(base + 16),
                   None)
    assert r == moe.MOE_ERR_OVERLAP


@nogpu
def test_stage_entry_points_reject_bad_arguments(lib):
    from mixture_experts_ffn_gb300 import moe

    act = moe.act_params(moe.MOE_ACT_SWIGLU, swiglu_fusion=3)  # fusion must be 1 or 2
    ws = A(9)
    assert lib.moe_grouped_gemm_act(A(0), A(1), None, A(2), 64, 32, 64, 4, moe.MOE_BF16,
                                    ctypes.byref(act), A(3), ws, 4096, None) == moe.MOE_ERR_INVALID_ARG
    act = moe.act_params(moe.MOE_ACT_SILU_AND_MUL)
    # workspace too small / misaligned
    assert lib.moe_grouped_gemm_act(A(0), A(1), None, A(2), 64, 32, 64, 4, moe.MOE_BF16,
                                    ctypes.byref(act), A(3), ws, 16, None) == moe.MOE_ERR_WORKSPACE
    assert lib.moe_grouped_gemm_act(A(0), A(1), None, A(2), 64, 32, 64, 4, moe.MOE_BF16,
                                    ctypes.byref(act), A(3), ctypes.c_void_p(A(9).value + 8), 4096,
                                    None) == moe.MOE_ERR_WORKSPACE
    # bad dtype
    assert lib.moe_grouped_gemm_down(A(0), A(1), None, A(2), 64, 32, 64, 4, 5, A(3), ws, 4096,
                                     None) == moe.MOE_ERR_INVALID_ARG
    # indexed path: tiled widths
    assert lib.moe_indexed_mlp(A(0), A(1), A(2), A(3), A(4), 4, 100, 256, 8, 2, 1.0, A(5), ws,
                               1 << 30, None) == moe.MOE_ERR_UNSUPPORTED
    # swiglu without up needs a fusion layout
    assert lib.swiglu(A(0), None, 4, 8, moe.MOE_F32, 0, 7.0, 1.0, 0.0, A(1), None) == \
        moe.MOE_ERR_INVALID_ARG
    # permute: workspace size
    need = lib.moe_permute_workspace_size(64, 8)
    assert lib.moe_permute(A(0), moe.MOE_BF16, A(1), 32, 64, 8, 2, A(2), A(3), A(4), A(5), ws,
                           need - 256, None) == moe.MOE_ERR_WORKSPACE
    # permute gather: missing hidden, small workspace, out inside hidden
    assert lib.moe_permute_gather(None, moe.MOE_BF16, A(1), A(2), 32, 64, 8, 2, A(3), ws, 4096,
                                  None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_permute_gather(A(0), moe.MOE_BF16, A(1), A(2), 32, 64, 8, 2, A(3), ws, 64,
                                  None) == moe.MOE_ERR_WORKSPACE
    assert lib.moe_permute_gather(A(0), moe.MOE_BF16, A(1), A(2), 32, 64, 8, 2,
                                  ctypes.c_void_p(A(0).value + 256), ws, 4096,
                                  None) == moe.MOE_ERR_OVERLAP
    # the forward checks the router parameters too
    p = moe.route_params(3, num_expert_group=2, topk_group=1)
    need = lib.moe_workspace_size(16, 64, 32, 4, 3, moe.MOE_BF16)
    assert lib.moe_ffn_forward(A(0), A(1), A(2), A(3), None, None, None, None, 16, 64, 32, 4,
                               moe.MOE_BF16, ctypes.byref(p), ctypes.byref(act), A(4), None, None,
                               None, None, ws, need, None) == moe.MOE_ERR_INVALID_ARG
