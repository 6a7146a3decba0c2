"""Permute (bit-exact index maps and gathered rows) and the weighted combine
against the oracle; device-detected bad ids."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

from gpu_cases import np_
from tolerances import assert_rounded_once

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_ffn_gb300 import build, moe as m

    build.build()
    return m


def _ids(T, K, E, gen, mode="random"):
    if mode == "one":  # every route on one expert
        return torch.full((T, K), E // 2, dtype=torch.int32)
    if mode == "skewed":  # most routes on two experts, several empty experts
        x = torch.randint(0, 4, (T, K), generator=gen, dtype=torch.int32)
        return torch.where(x < 3, torch.tensor(E - 1, dtype=torch.int32), x * 2)
    rows = [torch.randperm(E, generator=gen)[:K] if K <= E else
            torch.randint(0, E, (K,), generator=gen) for _ in range(T)]
    return torch.stack(rows).to(torch.int32)


@pytest.mark.parametrize("T,K,E,H,mode,dtype", [
    (1, 1, 1, 64, "random", torch.bfloat16),
    (3, 2, 8, 72, "random", torch.float32),
    (1000, 8, 128, 256, "random", torch.bfloat16),
    (700, 4, 64, 40, "skewed", torch.bfloat16),
    (257, 6, 16, 128, "one", torch.float32),
    (4096, 8, 128, 2048, "random", torch.bfloat16),
    (8192, 8, 256, 64, "random", torch.bfloat16),
    (3000, 8, 2000, 16, "random", torch.bfloat16),     # E > 1024, one warp per chunk
    (5000, 8, 12288, 16, "random", torch.bfloat16),    # the largest E accepted
    (70000, 2, 384, 16, "skewed", torch.bfloat16),     # 137 chunks: scan over > 128 chunks
])
def test_permute_bit_exact(moe, T, K, E, H, mode, dtype):
    g = torch.Generator().manual_seed(T * 7 + E)
    ids = _ids(T, K, E, g, mode)
    hidden = torch.randn((T, H), generator=g).to(dtype)
    r = moe.moe_permute(ids.cuda(), E, hidden.cuda())
    torch.cuda.synchronize()
    ref = O.permute(ids.numpy(), E)
    np.testing.assert_array_equal(np_(r["seg_end"]), ref["seg_end"])
    np.testing.assert_array_equal(np_(r["row_to_route"]), ref["row_to_route"])
    np.testing.assert_array_equal(np_(r["route_to_row"]), ref["route_to_row"])
    xin = O.gather_rows(np_(hidden), ref["row_to_route"], K)
    np.testing.assert_array_equal(np_(r["expert_input"]), xin)
    assert moe.moe_sync_status(r["ws"]) == moe.MOE_OK


def test_permute_bad_ids_latch_device_error(moe):
    ids = torch.tensor([[0, 1], [5, 2], [-1, 3]], dtype=torch.int32, device="cuda")  # E = 4
    hidden = torch.randn((3, 16), device="cuda").to(torch.bfloat16)
    r = moe.moe_permute(ids, 4, hidden)
    assert moe.moe_sync_status(r["ws"]) == moe.MOE_ERR_DEVICE
    assert moe.moe_sync_status(r["ws"]) == moe.MOE_OK  # the read clears the word
    seg = np_(r["seg_end"])
    assert list(seg) == [1, 2, 3, 4]  # the two bad routes are dropped
    r2r = np_(r["route_to_row"])
    assert r2r[2] == -1 and r2r[4] == -1


@pytest.mark.parametrize("T,K,H,dtype,scale", [
    (1, 1, 8, "f32", 1.0),
    (64, 2, 128, "f32", 0.5),
    (333, 8, 2048, "bf16", 1.0),
    (50, 3, 7, "bf16", 2.5),     # H not a multiple of the vector width
    (2048, 4, 2880, "bf16", 1.0),
])
def test_combine(moe, T, K, H, dtype, scale):
    g = torch.Generator().manual_seed(T + H)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    M = T * K
    y = torch.randn((M, H), generator=g).to(tdt)
    w = torch.rand((T, K), generator=g)
    r2r = torch.randperm(M, generator=g).to(torch.int32)
    out = moe.moe_combine(y.cuda(), w.cuda(), r2r.cuda(), scale)
    torch.cuda.synchronize()
    exact = O.combine(np_(y), np_(w), np_(r2r), T, K, scale, None)
    assert_rounded_once(np_(out), exact, dtype, "combine")
    # deterministic: a second call is bitwise identical
    out2 = moe.moe_combine(y.cuda(), w.cuda(), r2r.cuda(), scale)
    assert torch.equal(out, out2)


@pytest.mark.parametrize("T,K,E,bs", [
    (4096, 8, 128, 64),      # Qwen3-style routes
    (37, 3, 5, 16),
    (1, 1, 1, 64),
    (2000, 4, 2000, 16),     # many empty experts
    (0, 2, 8, 16),           # no tokens
])
def test_permute_align(moe, T, K, E, bs):
    """MoEPermuteAlignFwdOp: equal to the oracle (ascending route index inside
    each range, the order this build fixes), entry for entry."""
    g = torch.Generator().manual_seed(T * 7 + E)
    ids = (torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)]).to(torch.int32)
           if T else torch.empty((0, K), dtype=torch.int32))
    sid, eid, npp = moe.moe_permute_align(ids.cuda(), E, bs)
    torch.cuda.synchronize()
    want = O.permute_align(ids.numpy(), E, bs)
    assert int(npp[0]) == int(want["num_tokens_post_pad"])
    np.testing.assert_array_equal(sid.cpu().numpy(), want["sorted_token_ids"])
    np.testing.assert_array_equal(eid.cpu().numpy(), want["expert_ids"])
