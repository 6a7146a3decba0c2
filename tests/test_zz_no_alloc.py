"""moe_permute_noalloc, the permute for callers that cannot allocate device
memory (it uses the library's own fixed scratch array instead of a caller
workspace), checked through the C ABI against moe_permute and the oracle on
two calls in a row, at its size limit, in every operand type, on the
large-expert-count scatter path, and for allocating nothing.  Kept in its own
file, collected last."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_ffn_gb300 import build, moe

    build.build()
    lib = moe.load_library()
    fn = lib.moe_permute_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, hidden, ids, E):
    T, K = ids.shape
    H = hidden.shape[1]
    M = T * K
    dev = hidden.device
    xin = torch.empty((M, H), dtype=hidden.dtype, device=dev)
    seg = torch.empty((E,), dtype=torch.int32, device=dev)
    r2r = torch.empty((M,), dtype=torch.int32, device=dev)
    route_to_row = torch.empty((M,), dtype=torch.int32, device=dev)
    from mixture_experts_ffn_gb300 import moe

    dt = moe._dt(hidden)
    st = lib.moe_permute_noalloc(_p(hidden), dt, _p(ids), T, H, E, K, _p(xin), _p(seg), _p(r2r),
                                 _p(route_to_row),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    return xin, seg, r2r, route_to_row


def _check_against_oracle(got, ids, hidden, E):
    """The permutation is integer work and the gather a copy: both bit-exact
    against the oracle's permute."""
    from oracle import moe_oracle as O

    K = ids.shape[1]
    want = O.permute(ids.cpu().numpy(), E)
    assert torch.equal(got[1].cpu(), torch.from_numpy(want["seg_end"]))
    assert torch.equal(got[2].cpu(), torch.from_numpy(want["row_to_route"]))
    assert torch.equal(got[3].cpu(), torch.from_numpy(want["route_to_row"]))
    rows = torch.from_numpy(want["row_to_route"]).long() // K
    assert torch.equal(got[0].cpu(), hidden.cpu()[rows])


@pytest.mark.parametrize("T,K,E,H,dtype", [
    (4096, 8, 128, 256, torch.bfloat16),
    (333, 3, 40, 72, torch.float32),
    (2048, 4, 64, 128, torch.float16),
    (4096, 8, 600, 64, torch.bfloat16),    # E > 384: the scatter step with > 48 KB of shared memory
    (16384, 8, 1024, 64, torch.bfloat16),  # 131072 routes over 1024 experts
])
def test_noalloc_matches_workspace_permute_twice(lib, T, K, E, H, dtype):
    from mixture_experts_ffn_gb300 import moe

    g = torch.Generator().manual_seed(T + E)
    for call in range(2):  # two calls in a row, different inputs, shared scratch
        ids = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)]).to(torch.int32)
        hidden = torch.randn((T, H), generator=g).to(dtype)
        ids, hidden = ids.cuda(), hidden.cuda()
        got = _noalloc(lib, hidden, ids, E)
        ref = moe.moe_permute(ids, E, hidden)
        torch.cuda.synchronize()
        # the permutation is integer work: bit-exact, as in the other permute tests
        assert torch.equal(got[0], ref["expert_input"]), call
        assert torch.equal(got[1], ref["seg_end"]), call
        assert torch.equal(got[2], ref["row_to_route"]), call
        assert torch.equal(got[3], ref["route_to_row"]), call
        _check_against_oracle(got, ids, hidden, E)


def test_noalloc_allocates_no_device_memory(lib):
    """After a first call (which looks up the scratch array's address and may
    load the kernels), a call changes neither the device's free memory nor
    torch's reserved memory."""
    T, K, E, H = 2048, 8, 256, 128
    g = torch.Generator().manual_seed(5)
    ids = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)]).to(torch.int32).cuda()
    hidden = torch.randn((T, H), generator=g).to(torch.bfloat16).cuda()
    M = T * K
    bufs = (torch.empty((M, H), dtype=torch.bfloat16, device="cuda"),
            torch.empty((E,), dtype=torch.int32, device="cuda"),
            torch.empty((M,), dtype=torch.int32, device="cuda"),
            torch.empty((M,), dtype=torch.int32, device="cuda"))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call():
        st = lib.moe_permute_noalloc(_p(hidden), 1, _p(ids), T, H, E, K, _p(bufs[0]), _p(bufs[1]),
                                     _p(bufs[2]), _p(bufs[3]), stream)
        assert st == 0, st
        torch.cuda.synchronize()

    call()
    free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
    call()
    call()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_reserved() == reserved0
    _check_against_oracle(bufs, ids, hidden, E)


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    from mixture_experts_ffn_gb300 import moe

    # T*K = 262144 routes over 1024 experts needs ~1.03 MiB of scratch: rejected
    # before anything is launched (buffers sized for the call all the same)
    T, K, E = 32768, 8, 1024
    ids = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    seg = torch.zeros(E, dtype=torch.int32, device="cuda")
    r2r = torch.full((T * K,), -7, dtype=torch.int32, device="cuda")
    route_to_row = torch.full((T * K,), -7, dtype=torch.int32, device="cuda")
    st = lib.moe_permute_noalloc(None, 1, _p(ids), T, 8, E, K, None, _p(seg), _p(r2r),
                                 _p(route_to_row),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == moe.MOE_ERR_WORKSPACE
    assert int((r2r != -7).sum()) == 0  # nothing was written
