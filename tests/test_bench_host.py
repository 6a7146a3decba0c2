"""Host-side helpers of bench.py (no GPU): the input hashes of the JSON line
and the rule that a committed ncu traffic figure is used only while the
kernel's sources still hash to what the capture ran on."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mixture_experts_ffn_gb300 import synth  # noqa: E402


def test_input_hashes_follow_the_bytes():
    cfg = synth.CONFIGS["gpt_oss_bf16"].replace(T=8, H=64, F=32, E=4)
    inp = synth.make_inputs(cfg, "cpu")
    h1 = bench.inputs_sha256(inp)
    assert set(h1) == {"hidden", "logits", "b_gate_up", "b_down"}  # no bias, no fixed ids
    assert all(len(v) == 16 for v in h1.values())
    assert bench.inputs_sha256(synth.make_inputs(cfg, "cpu")) == h1  # same seeds, same bytes
    inp["hidden"] = inp["hidden"].clone()
    inp["hidden"][3, 5] += 1
    h2 = bench.inputs_sha256(inp)
    assert h2["hidden"] != h1["hidden"] and h2["logits"] == h1["logits"]


def test_traffic_figure_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// kernel v1\n")
    (tmp_path / "profiles").mkdir()
    prof = tmp_path / "profiles" / f"some_kernel_{bench.WORKLOAD}.md"
    prof.write_text("traffic_bytes_per_launch: 12345678\n"
                    f"source_sha256: {bench.sources_sha256([str(src)])}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("some_kernel", [str(src)]) == 12345678.0
    src.write_text("// kernel v2\n")  # the kernel changed since the capture
    assert bench.profile_traffic("some_kernel", [str(src)]) is None
    assert bench.profile_traffic("other_kernel", [str(src)]) is None  # no summary at all
