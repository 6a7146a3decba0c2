"""A bounded in-kernel wait made to run out on purpose, without faulting or
hanging the GPU: the test hook makes both grid barriers of the fused route +
index-map launch wait for one arrival more than the grid provides, with a
50 ms limit.  Every CTA then gives up, latches the timeout bit in the
workspace status word and returns.  The test checks that the host reads
MOE_ERR_TIMEOUT, that the context stays usable, and that once the status
area is cleared the same workspace gives results bit-identical to a clean
run."""
import pytest
import torch

from mixture_experts_ffn_gb300 import synth

from gpu_cases import make

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_ffn_gb300 import build, moe as m

    build.build()
    return m


def _route_permute(moe, cfg, inp, ws):
    p, _ = moe.config_params(cfg)
    return moe.moe_route_permute(inp["logits"], p, inp["correction_bias"], inp["expert_ids"],
                                 ws=ws)


@pytest.mark.parametrize("name", ["qwen3_bf16", "deepseek_v3_bf16"])
def test_grid_barrier_timeout_is_reported_and_recovered(moe, name):
    cfg = synth.CONFIGS[name].replace(T=512, H=256, F=128)
    inp, _ = make(cfg)
    ws = moe._ws(moe.load_library().moe_permute_workspace_size(cfg.T * cfg.K, cfg.E), "cuda")
    ref = _route_permute(moe, cfg, inp, ws)
    assert moe.moe_sync_status(ws) == moe.MOE_OK

    was_on = moe.moe_test_force_wait_timeout(True, 50_000_000)  # 50 ms
    try:
        assert not was_on
        _route_permute(moe, cfg, inp, ws)
        assert moe.moe_sync_status(ws) == moe.MOE_ERR_TIMEOUT
        # reporting the timeout cleared the whole status area, the barrier
        # counters the failed launch left set included
        assert int(ws[:moe.MOE_STATUS_BYTES].to(torch.int32).sum()) == 0
    finally:
        moe.moe_test_force_wait_timeout(False)
    # the context is still usable: plain work on the same stream runs
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 1023 * 1024 / 2

    # the barrier counters were left as the failed launch stood; the status
    # clear resets them, and the next launch is the clean one again
    moe.moe_clear_status(ws)
    got = _route_permute(moe, cfg, inp, ws)
    assert moe.moe_sync_status(ws) == moe.MOE_OK
    for a, b in zip(got[:2], ref[:2]):
        assert torch.equal(a, b)
    for k in ("seg_end", "row_to_route", "route_to_row"):
        assert torch.equal(got[4][k], ref[4][k]), k


def test_forward_after_a_timeout_matches_a_clean_forward(moe):
    """The whole forward reports the timeout of its first launch, and after
    the status clear the same workspace gives the clean forward's output bit
    for bit."""
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=300, H=256, F=128, E=32, local_count=0)
    inp, _ = make(cfg)
    p, a = moe.config_params(cfg)
    ws = moe._ws(moe.moe_workspace_size(cfg.T, cfg.H, cfg.F, cfg.E, cfg.K, moe.MOE_BF16), "cuda")

    def fwd():
        return moe.moe_ffn_forward(inp["hidden"], inp["logits"], inp["w_gate_up"],
                                   inp["w_down"], p, a, ws=ws)

    ref = fwd()
    assert moe.moe_sync_status(ws) == moe.MOE_OK
    moe.moe_test_force_wait_timeout(True, 50_000_000)
    try:
        fwd()
        assert moe.moe_sync_status(ws) == moe.MOE_ERR_TIMEOUT
    finally:
        moe.moe_test_force_wait_timeout(False)
    moe.moe_clear_status(ws)
    got = fwd()
    assert moe.moe_sync_status(ws) == moe.MOE_OK
    assert torch.equal(got, ref)


def test_forward_after_a_reported_timeout_needs_no_clear(moe):
    """moe_sync_status that reports a timeout leaves the workspace ready: the
    next forward on it, with no status clear in between, is the clean one."""
    # H = 2048 and 256 routes per expert: the gate_up runs on the SM-pair
    # kernel, whose tile counters share the status area
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=256, H=2048, F=256, E=8, local_count=0)
    inp, _ = make(cfg)
    p, a = moe.config_params(cfg)
    ws = moe._ws(moe.moe_workspace_size(cfg.T, cfg.H, cfg.F, cfg.E, cfg.K, moe.MOE_BF16), "cuda")

    def fwd():
        return moe.moe_ffn_forward(inp["hidden"], inp["logits"], inp["w_gate_up"],
                                   inp["w_down"], p, a, ws=ws)

    ref = fwd().clone()
    assert moe.moe_sync_status(ws) == moe.MOE_OK
    moe.moe_test_force_wait_timeout(True, 50_000_000)
    try:
        fwd()
        assert moe.moe_sync_status(ws) == moe.MOE_ERR_TIMEOUT
    finally:
        moe.moe_test_force_wait_timeout(False)
    got = fwd()
    assert moe.moe_sync_status(ws) == moe.MOE_OK
    assert torch.equal(got, ref)


def test_stage_profile_in_a_fresh_process():
    """MOE_PROFILE=1 (read when the library loads) records the forward's
    stages with CUDA events; moe_profile_report returns one entry per stage
    and empties the record."""
    import os
    import subprocess
    import sys

    code = r"""
import sys, torch
sys.path.insert(0, "tests")
from mixture_experts_ffn_gb300 import moe, synth
from gpu_cases import make
cfg = synth.CONFIGS["qwen3_bf16"].replace(T=300, H=256, F=128, E=32, local_count=0)
inp, _ = make(cfg)
p, a = moe.config_params(cfg)
for _ in range(3):
    moe.moe_ffn_forward(inp["hidden"], inp["logits"], inp["w_gate_up"], inp["w_down"], p, a)
torch.cuda.synchronize()
rep = moe.moe_profile_report()
assert set(rep) == {"route_permute", "gate_up", "down", "combine"}, rep
assert all(c == 3 and us > 0 for c, us in rep.values()), rep
assert moe.moe_profile_report() == {}
print("ok", rep)
"""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       env=dict(os.environ, MOE_PROFILE="1"), timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
