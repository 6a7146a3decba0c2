"""Benchmark of the routed MoE FFN forward on GB300.

One step = one full forward (route -> permute -> gate_up GEMM + fused
activation -> down GEMM -> combine) of the DeepSeek-V3-style workload (T=8192
tokens, H=7168, F=2048, E=256 experts, top-8, sigmoid scoring with a
selection-only correction bias, 8 expert groups of which 4 are kept,
renormalised, routed_scaling_factor 2.5, silu_and_mul), the largest of the
model-shaped workloads, on synthetic seeded inputs already resident in HBM.  The L2 is flushed before every timed step (a
512 MiB write, then a 512 MiB read so that the written lines are cleaned
inside the flush rather than written back inside the timed step) and each step
is bracketed by CUDA events on the launching stream.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain fp64 restatement of the
method) on the host cores, on a bounded token sample of the same workload
(the oracle's cost is one float64 conversion and product per distinct expert
hit, so the sample is a few tokens on the DeepSeek-V3-style workload).
Under torchrun with N > 1 each rank runs its own replica of the workload (the
layer has no cross-token exchange, so the path shards with no collective);
value = tokens of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "deepseek_v3_bf16"  # the default workload (bench line); --workload picks another
METRIC = "MoE FFN fwd tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(x: float) -> float:
    """x maximised over the ranks of the default process group (x itself when
    there is none): the slowest rank's time."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = (torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl"
           else torch.device("cpu"))
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, slowest_ms: float) -> float:
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    return world * units_per_rank / (slowest_ms / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


_SAMPLER = r"""
import ctypes, sys, time
uuid = sys.argv[1]
lib = ctypes.CDLL("libnvidia-ml.so.1")
assert lib.nvmlInit_v2() == 0
n = ctypes.c_uint()
lib.nvmlDeviceGetCount_v2(ctypes.byref(n))
h = None
for i in range(n.value):
    d = ctypes.c_void_p()
    lib.nvmlDeviceGetHandleByIndex_v2(i, ctypes.byref(d))
    buf = ctypes.create_string_buffer(96)
    lib.nvmlDeviceGetUUID(d, buf, 96)
    if h is None or (uuid and uuid in buf.value.decode()):
        h = d
mx = ctypes.c_uint()
lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
    lib.nvmlDeviceGetCurrentClocksThrottleReasons
print("max", mx.value, flush=True)
clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
while True:
    lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk))
    get_reasons(h, ctypes.byref(rs))
    print(f"{time.time():.6f} {clk.value} {rs.value}", flush=True)
    time.sleep(0.002)
"""


class ClockSampler:
    """SM clock and clock-event reasons of this GPU, sampled every ~2 ms by a
    separate process through NVML (read-only queries), so that short timed
    regions still get samples; ``mark()`` brackets the timed region."""

    BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
            0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index=0):
        import torch

        try:
            self.uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            self.uuid = ""
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen([sys.executable, "-c", _SAMPLER, self.uuid],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.01)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = out.splitlines()

    def summary(self):
        smax, sm, reasons = None, [], set()
        for l in self.lines:
            f = l.split()
            if len(f) == 2 and f[0] == "max":
                smax = float(f[1])
                continue
            if len(f) != 3:
                continue
            t, c, r = float(f[0]), float(f[1]), int(f[2])
            if self.t0 is not None and not (self.t0 <= t <= (self.t1 or t)):
                continue
            sm.append(c)
            for bit, name in self.BITS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvml"}


# the files each tcgen05 GEMM kernel is compiled from (the ncu summary under
# profiles/ records their hash, so a stale summary is never quoted)
GEMM_SOURCES = {
    k: [os.path.join(ROOT, "mixture_experts_ffn_gb300", "csrc", f) for f in files]
    for k, files in {
        "gemm_tc_kernel": ("gemm_tc.cu", "gemm_epilogue.cuh", "tc_ptx.cuh", "common.cuh"),
        "gemm_sw_kernel": ("gemm_sw.cu", "gemm_epilogue.cuh", "tc_ptx.cuh", "common.cuh"),
    }.items()}


def gemm_kernel(M, N, K, E, split=False):
    """The tcgen05 kernel the library picks for a bf16/f16 grouped GEMM of M
    rows over E experts, N output (or activation) columns and depth K: the
    SM-pair kernel with 256 weight rows per CTA for long K and segments
    averaging >= 128 rows, else the one-SM row-tile kernel (the rule of
    launch_gemm_tc, with no MOE_TC_KERNEL override)."""
    env = os.environ.get("MOE_TC_KERNEL", "")
    sw_ok = not split and N % 8 == 0 and K % 8 == 0
    if sw_ok and (env[:1] in ("s", "w") or (env[:1] != "1" and K >= 2048 and M >= 128 * E)):
        return "gemm_sw_kernel"
    return "gemm_tc_kernel"


def sources_sha256(paths):
    """SHA-256 over the concatenated bytes of a kernel's source files, in order."""
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def inputs_sha256(inp):
    """SHA-256 (first 16 hex digits) of the bytes of each input drawn on the
    host (activations, logits, correction bias, fixed ids, biases); the weight
    stacks are drawn on the device from their seeds and are not hashed."""
    import torch

    out = {}
    for k in ("hidden", "logits", "correction_bias", "expert_ids", "b_gate_up", "b_down"):
        t = inp.get(k)
        if t is None:
            continue
        b = t.detach().contiguous().view(-1).view(torch.uint8).cpu().numpy().tobytes()
        out[k] = hashlib.sha256(b).hexdigest()[:16]
    return out


def profile_traffic(kernel: str, srcs):
    """DRAM bytes per launch from the committed ncu summary of ``kernel``, when
    the summary was taken on the current source of the kernel."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{WORKLOAD}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not m or not h:
        return None
    return float(m.group(1)) if sources_sha256(srcs) == h.group(1) else None


# --------------------------------------------------------------------- reference
class HostExperts:
    """The oracle's view of a weight stack [E, rows, cols]: expert e as a
    float32 numpy array, copied from the stack (host or device) on demand."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, e):
        return self.t[int(e)].float().cpu().numpy()


def workload_config(args, cfg, world, **extra):
    """The `config` object of the JSON line, the same for both arms."""
    from mixture_experts_ffn_gb300 import synth

    c = {"workload": args.workload, "T": cfg.T, "H": cfg.H, "F": cfg.F, "E": cfg.E, "K": cfg.K,
         "scoring": cfg.scoring, "renormalize": cfg.renormalize, "groups": [cfg.G, cfg.TG],
         "rsf": cfg.rsf, "act": ["silu_and_mul", "swiglu", "identity", "gelu_and_mul", "relu", "gelu",
                                                     "silu"][cfg.act],
         "moerouter_slice": [cfg.local_start, cfg.local_count],
         "parallelism": f"replicas x{world}"}
    c.update(extra)
    return c


def run_reference(args, rank, world):
    """The CPU oracle, as it stands, on a bounded token sample per step."""
    if rank != 0:
        return
    import numpy as np
    import torch

    from mixture_experts_ffn_gb300 import synth
    from oracle import cases
    from oracle import moe_oracle as O

    cfg = synth.CONFIGS[args.workload]
    # the inputs are drawn where the GPU arm draws them (the weight stacks on
    # the GPU when there is one, so both arms see the same bytes, and a host
    # never holds the largest stacks whole); the oracle runs on the host cores
    # and fetches each expert it needs inside the timed call
    inp = synth.make_inputs(cfg, "cuda" if torch.cuda.is_available() else "cpu")
    n = {k: cases.to_np(v) for k, v in inp.items() if k not in ("w_gate_up", "w_down")}
    w1, w2 = HostExperts(inp["w_gate_up"]), HostExperts(inp["w_down"])
    sample = min(args.ref_tokens, cfg.T)
    per_step = []
    for step in range(args.warmup + args.steps):
        toks = synth.subset_tokens(cfg.T, sample)
        t0 = time.perf_counter()
        O.ffn_forward(n["hidden"], n["logits"], w1, w2, K=cfg.K, F=cfg.F, scoring=cfg.scoring,
                      renormalize=cfg.renormalize, G=cfg.G, TG=cfg.TG, rsf=cfg.rsf,
                      correction_bias=n["correction_bias"], expert_ids=n["expert_ids"],
                      act=cfg.act, fusion=cfg.swiglu_fusion, limit=cfg.limit, alpha=cfg.alpha,
                      beta=cfg.beta, b_gate_up=n["b_gate_up"], b_down=n["b_down"],
                      dtype=cfg.dtype, local_start=cfg.local_start,
                      local_count=cfg.local_count, route_scale=cfg.route_scale, tokens=toks)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            per_step.append(dt)
    cores = len(os.sched_getaffinity(0))
    sec = sum(per_step) / len(per_step)
    value = sample / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args, cfg, world, path="CPU oracle (numpy float64)",
                                  sample_tokens_per_step=sample),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample} tokens of the {cfg.T}-token workload per step "
                                   f"(all their routes and experts), numpy float64; each "
                                   f"distinct expert's weights fetched and converted inside "
                                   f"the timed call"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- ours
def stage_cost(cfg, D):
    """Algorithmic FLOPs and bytes per launch of each stage.  The bytes are the
    method's own traffic: the distinct experts' weights and biases, hidden,
    logits, the output and the routing weights and ids.  The staged
    pipeline's permuted copy, gated intermediate and per-route outputs Y are
    implementation overhead and are not counted (so the permute, and the
    combine's Y reads, count nothing but their share of those tensors)."""
    T, H, F, E, K = cfg.T, cfg.H, cfg.F, cfg.E, cfg.K
    M = T * K
    lc = cfg.local_count
    b = 4 if cfg.dtype == "f32" else 2
    bias1 = D * 2 * F * b if cfg.bias_std is not None else 0
    bias2 = D * H * b if cfg.bias_std is not None else 0
    route = T * E * 4 + M * 8 + T * lc * 4 + (T * 4 if lc else 0)
    return {
        "route": (0.0, route),
        "permute": (0.0, M * 4 + T * H * b),
        "permute_maps": (0.0, M * 4),
        "permute_gather": (0.0, T * H * b),
        "route_permute": (0.0, route),
        "gemm_act": (4.0 * M * H * F, D * 2 * F * H * b + bias1 + T * H * b),
        "gemm_act_gathered": (4.0 * M * H * F, D * 2 * F * H * b + bias1 + T * H * b),
        "gemm_down": (2.0 * M * F * H, D * H * F * b + bias2),
        "combine": (0.0, M * 4 + T * H * b),
        "indexed_mlp": (6.0 * M * H * F, D * 3 * F * H * b + T * H * b + M * 8 + T * H * b),
        "forward": (6.0 * M * H * F, D * 3 * F * H * b + bias1 + bias2 + T * H * b + route
                    + T * H * b),
    }


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    from mixture_experts_ffn_gb300 import build as mbuild
    from mixture_experts_ffn_gb300 import moe, synth

    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    if rank == 0 or not os.path.exists(mbuild.LIB):
        mbuild.build()
    if world > 1:
        dist.barrier()
    dev = torch.device("cuda", local)
    cfg = synth.CONFIGS[args.workload]
    if args.override:
        cfg = cfg.replace(**{k: type(getattr(cfg, k))(v) for k, v in
                             (kv.split("=") for kv in args.override.split(","))})
    inp = synth.make_inputs(cfg, dev)
    p, a = moe.config_params(cfg)
    indexed = (cfg.T * cfg.K <= 2 * cfg.E and cfg.act == synth.ACT_SILU_AND_MUL
               and cfg.bias_std is None and cfg.dtype == "bf16" and cfg.H % 128 == 0
               and cfg.F % 256 == 0)
    T, H, F, E, K = cfg.T, cfg.H, cfg.F, cfg.E, cfg.K
    # the forward reads the gate_up rows through the permutation on the
    # tensor-core path (bf16 or f16, 16-byte rows)
    gathered = not indexed and cfg.dtype != "f32" and H % 8 == 0 and F % 8 == 0
    tdt = synth.torch_dtype(cfg.dtype)
    mdt = {"bf16": moe.MOE_BF16, "f16": moe.MOE_F16, "f32": moe.MOE_F32}[cfg.dtype]
    out = torch.empty((T, H), dtype=tdt, device=dev)
    tw = torch.empty((T, K), dtype=torch.float32, device=dev)
    ti = torch.empty((T, K), dtype=torch.int32, device=dev)
    probs = torch.empty((T, cfg.local_count), dtype=torch.float32, device=dev) \
        if cfg.local_count else None
    wsc = torch.empty((T,), dtype=torch.float32, device=dev) if cfg.local_count else None
    ws = moe._ws(moe.moe_workspace_size(T, H, F, E, K, mdt), dev)
    flush_w = torch.zeros(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(128 << 20, dtype=torch.float32, device=dev)

    class L2Flush:
        """Write 512 MiB (evicts everything), then read another 512 MiB: the read
        forces the write-back of the dirty lines the write left, so the L2
        holds only clean lines of an unrelated buffer when a step starts."""

        def zero_(self):
            flush_w.zero_()
            torch.sum(flush_r)

    flush = L2Flush()
    stream = torch.cuda.current_stream()

    def forward():
        moe.moe_ffn_forward(inp["hidden"], inp["logits"], inp["w_gate_up"], inp["w_down"], p, a,
                            inp["correction_bias"], inp["expert_ids"], inp["b_gate_up"],
                            inp["b_down"], out=out, topk_weights_out=tw, topk_ids_out=ti,
                            router_probs=probs, weight_scale=wsc, ws=ws)

    def timed(fn, steps, warmup):
        for _ in range(warmup):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        n0 = moe.moe_launch_count()
        for s, e in ev:
            flush.zero_()
            s.record(stream)
            fn()
            e.record(stream)
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in ev], moe.moe_launch_count() - n0

    if args.stage:
        run_stage(args, moe, cfg, inp, p, a, ws, flush, timed)
        return

    # ---- the timed forward: W warm-up steps, then untimed steps for about a
    # second so the SM clock leaves its idle state, then exactly K timed steps
    for _ in range(args.warmup):
        flush.zero_()
        forward()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_soak = time.time()
        soak = 0
        while time.time() - t_soak < args.soak_s:
            for _ in range(16):
                forward()
            torch.cuda.synchronize()
            soak += 16
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        clk.mark(True)
        times, launches = timed(forward, args.steps, 0)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        clk.mark(False)
    status = moe.moe_sync_status(ws)
    ms = reduce_max(sum(times) / len(times))
    value = job_throughput(T, world, ms)

    # ---- per-stage breakdown (rank 0), same inputs, each stage timed alone
    breakdown = {}
    roofline = None
    e2e = None
    if rank == 0:
        D = int((torch.bincount(ti.flatten().long(), minlength=E) > 0).sum())
        costs = stage_cost(cfg, D)
        perm = moe.moe_permute(ti, E, inp["hidden"])
        act_out = torch.empty((T * K, F), dtype=tdt, device=dev)
        y = torch.empty((T * K, H), dtype=tdt, device=dev)
        stage_ws = moe._ws(256, dev)
        # the forward routes and builds the index maps in one launch (E <= 512);
        # the staged path then copies the permuted rows in a launch of its own
        fused_maps = E <= 512
        if fused_maps:
            stages = {"route_permute": lambda: moe.moe_route_permute(
                inp["logits"], p, inp["correction_bias"], inp["expert_ids"], ws=perm["ws"])}
        else:
            stages = {"route": lambda: moe.moe_route(inp["logits"], p, inp["correction_bias"],
                                                     inp["expert_ids"], topk_weights=tw,
                                                     topk_ids=ti, router_probs=probs,
                                                     weight_scale=wsc)}
        if indexed:
            stages["indexed_mlp"] = lambda: moe.moe_indexed_mlp(inp["hidden"], inp["w_gate_up"],
                                                                inp["w_down"], tw, ti, out=out,
                                                                ws=ws)
        elif gathered:
            if not fused_maps:
                stages["permute"] = lambda: moe.moe_permute(ti, E, inp["hidden"], ws=perm["ws"],
                                                            with_gather=False)
            stages.update({
                "gemm_act": lambda: moe.moe_grouped_gemm_act_gathered(
                    inp["hidden"], perm["row_to_route"], K, inp["w_gate_up"], perm["seg_end"], F,
                    a, inp["b_gate_up"], out=act_out, ws=stage_ws),
                "gemm_down": lambda: moe.moe_grouped_gemm_down(act_out, inp["w_down"],
                                                               perm["seg_end"], inp["b_down"],
                                                               out=y, ws=stage_ws),
                "combine": lambda: moe.moe_combine(y, tw, perm["route_to_row"], out=out),
            })
        else:
            if fused_maps:
                stages["permute_gather"] = lambda: moe.moe_permute_gather(
                    inp["hidden"], perm["seg_end"], perm["row_to_route"], K,
                    out=perm["expert_input"], ws=stage_ws)
            else:
                stages["permute"] = lambda: moe.moe_permute(ti, E, inp["hidden"], ws=perm["ws"])
            stages.update({
                "gemm_act": lambda: moe.moe_grouped_gemm_act(perm["expert_input"],
                                                             inp["w_gate_up"], perm["seg_end"], F,
                                                             a, inp["b_gate_up"], out=act_out,
                                                             ws=stage_ws),
                "gemm_down": lambda: moe.moe_grouped_gemm_down(act_out, inp["w_down"],
                                                               perm["seg_end"], inp["b_down"],
                                                               out=y, ws=stage_ws),
                "combine": lambda: moe.moe_combine(y, tw, perm["route_to_row"], out=out),
            })
        pk, pk_src = load_peaks()
        for name, fn in stages.items():
            st, nl = timed(fn, max(5, args.steps), 3)
            us = 1e3 * sum(st) / len(st)
            fl, by = costs[{"permute": "permute_maps", "gemm_act": "gemm_act_gathered"}
                           .get(name, name) if gathered else name]
            t_tc = fl / (pk["bf16_tflops"] * 1e12)
            t_hbm = by / (pk["hbm_gbs"] * 1e9)
            bound = "tensor" if t_tc > t_hbm else "hbm"
            breakdown[name] = {
                "us": round(us, 2), "launches": nl // max(5, args.steps),
                "tflops": round(fl / (us * 1e-6) / 1e12, 1),
                "gbs": round(by / (us * 1e-6) / 1e9, 1), "bound": bound,
                "frac": round(max(t_tc, t_hbm) / (us * 1e-6), 3),
            }
        if indexed:
            dom = "indexed_mlp"
            kname = "indexed_gate_up + indexed_down"
            traffic = None
        else:
            dom = max(("gemm_act", "gemm_down"), key=lambda k: breakdown[k]["us"])
            # bf16 / f16 with 16-byte rows runs a tcgen05 kernel, anything else the SIMT one
            tc = cfg.dtype != "f32" and H % 8 == 0 and F % 8 == 0
            gated = cfg.act in synth.GATED_ACTS
            kern = (gemm_kernel(T * K, F, H, E, split=gated and cfg.swiglu_fusion == 0)
                    if dom == "gemm_act" else gemm_kernel(T * K, H, F, E)) if tc else \
                "gemm_simt_kernel"
            kname = f"{kern} ({dom})"
            traffic = profile_traffic(kern, GEMM_SOURCES[kern]) if tc and (
                dom == "gemm_act" and args.workload == WORKLOAD) else None
        fl, by = costs["gemm_act_gathered" if gathered and dom == "gemm_act" else dom]
        b = breakdown[dom]
        if b["bound"] == "tensor":
            ach, peak, unit = fl / (b["us"] * 1e-6) / 1e12, pk["bf16_tflops"], "TFLOP/s"
        else:
            ach, peak, unit = by / (b["us"] * 1e-6) / 1e9, pk["hbm_gbs"], "GB/s"
        roofline = {"kernel": kname, "bound": b["bound"],
                    "achieved": round(ach, 1), "peak": peak, "unit": unit,
                    "frac": round(ach / peak, 3), "traffic": traffic,
                    "peak_source": pk_src,
                    "algorithmic": {"flops": fl, "bytes": by, "distinct_experts": D}}
        fwd_fl, fwd_by = costs["forward"]
        t_roof = max(fwd_fl / (pk["bf16_tflops"] * 1e12), fwd_by / (pk["hbm_gbs"] * 1e9))
        breakdown["forward_roofline_frac"] = round(t_roof / (ms * 1e-3), 3)
        # the forward runs back to back for the whole measurement, so the
        # tensor peak it can hold is the sustained one (seconds under the
        # power cap); reported beside the burst-peak fraction
        if "bf16_tflops_sustained" in pk:
            t_roof_s = max(fwd_fl / (pk["bf16_tflops_sustained"] * 1e12),
                           fwd_by / (pk["hbm_gbs"] * 1e9))
            breakdown["forward_roofline_frac_sustained"] = round(t_roof_s / (ms * 1e-3), 3)
        breakdown["forward_tflops"] = round(fwd_fl / (ms * 1e-3) / 1e12, 1)

    # ---- end to end through the C ABI with host buffers, every rank
    h_host = inp["hidden"].cpu().pin_memory()
    l_host = inp["logits"].cpu().pin_memory()
    o_host = torch.empty((T, H), dtype=tdt).pin_memory()
    # the same work as the device step: the MoERouter slice outputs (when the
    # workload has a slice) go to device buffers, as in the timed forward
    p_host = p
    ws_h = moe._ws(moe.moe_workspace_size_host(T, H, F, E, K, mdt), dev)

    def fwd_host():
        moe.moe_ffn_forward_host(h_host, l_host, inp["w_gate_up"], inp["w_down"], p_host, a,
                                 o_host, ws_h, inp["correction_bias"], inp["expert_ids"],
                                 inp["b_gate_up"], inp["b_down"], router_probs=probs,
                                 weight_scale=wsc)

    if world > 1:
        dist.barrier()
    et, _ = timed(fwd_host, args.steps, args.warmup)
    e_ms = reduce_max(sum(et) / len(et))
    eb = 4 if cfg.dtype == "f32" else 2
    e2e = {"value": job_throughput(T, world, e_ms), "unit": "tokens/s",
           # bytes of the whole job (every rank copies its own inputs and result)
           "h2d_bytes_per_step": world * (T * H * eb + T * E * 4),
           "d2h_bytes_per_step": world * T * H * eb}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args, cfg, inp)


    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg.dtype, "data": "synthetic",
            "config": workload_config(
                args, cfg, world,
                path="indexed" if indexed else "gathered gate_up" if gathered else "staged",
                l2="flushed before every timed step (512 MiB write, then 512 MiB read so no "
                   "dirty lines are written back inside the step)",
                soak_steps=soak),
            "gpu_launches": launches,
            "launches_per_step": launches // args.steps,
            "status": int(status),
            "roofline": roofline, "e2e": e2e, "cpu_baseline": cpu,
            "clocks": clk.summary(), "breakdown": breakdown,
            "inputs_sha256": inputs_sha256(inp),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_stage(args, moe, cfg, inp, p, a, ws, flush, timed):
    """One stage alone on the workload's inputs, as the forward runs it (for
    profiler captures)."""
    import torch

    from mixture_experts_ffn_gb300 import synth

    T, H, F, E, K = cfg.T, cfg.H, cfg.F, cfg.E, cfg.K
    dev = inp["hidden"].device
    gathered = cfg.dtype != "f32" and H % 8 == 0 and F % 8 == 0
    p = moe.config_params(cfg.replace(local_count=0))[0]
    tw, ti, _, _ = moe.moe_route(inp["logits"], p, inp["correction_bias"], inp["expert_ids"])
    perm = moe.moe_permute(ti, E, inp["hidden"])
    act_out = torch.empty((T * K, F), dtype=inp["hidden"].dtype, device=dev)
    y = torch.empty((T * K, H), dtype=inp["hidden"].dtype, device=dev)

    def gemm_act():
        if gathered:
            return moe.moe_grouped_gemm_act_gathered(inp["hidden"], perm["row_to_route"], K,
                                                     inp["w_gate_up"], perm["seg_end"], F, a,
                                                     inp["b_gate_up"], out=act_out)
        return moe.moe_grouped_gemm_act(perm["expert_input"], inp["w_gate_up"], perm["seg_end"],
                                        F, a, inp["b_gate_up"], out=act_out)

    gemm_act()
    moe.moe_grouped_gemm_down(act_out, inp["w_down"], perm["seg_end"], inp["b_down"], out=y)
    fns = {
        "indexed_mlp": lambda: moe.moe_indexed_mlp(inp["hidden"], inp["w_gate_up"], inp["w_down"],
                                                   tw, ti),
        "route": lambda: moe.moe_route(inp["logits"], p, topk_weights=tw, topk_ids=ti),
        "route_permute": lambda: moe.moe_route_permute(inp["logits"], p, inp["correction_bias"],
                                                       inp["expert_ids"], ws=perm["ws"]),
        "permute": lambda: moe.moe_permute(ti, E, inp["hidden"], ws=perm["ws"],
                                           with_gather=not gathered),
        "gemm_act": gemm_act,
        "gemm_down": lambda: moe.moe_grouped_gemm_down(act_out, inp["w_down"], perm["seg_end"],
                                                       inp["b_down"], out=y),
        "combine": lambda: moe.moe_combine(y, tw, perm["route_to_row"]),
    }
    extra = {}
    if args.stage == "shared_mlp":
        # the shared expert (dense gated MLP, intermediate size --shared-s) on
        # the workload's tokens
        S = args.shared_s
        sw = synth.make_shared_expert(cfg, S, dev)
        sh_out = torch.empty_like(inp["hidden"])
        sh_ws = moe._ws(moe.moe_shared_expert_workspace_size(
            T, H, S, {"bf16": moe.MOE_BF16, "f16": moe.MOE_F16, "f32": moe.MOE_F32}[cfg.dtype]), dev)
        fns["shared_mlp"] = lambda: moe.moe_shared_expert_mlp(
            inp["hidden"], sw["shared_w_gate_up"], sw["shared_w_down"], out=sh_out, ws=sh_ws)
        b = 4 if cfg.dtype == "f32" else 2
        extra = {"S": S, "flops": 6.0 * T * H * S,
                 "bytes": 3 * S * H * b + 2 * T * H * b + 2 * T * S * b}
    if args.stage == "gemm_act_split":
        extra = {}
        # the gated gate_up GEMM with the gate and up projections in two
        # tensors (SwiGLU fusion 0), on the permuted copy of the activations
        wg = inp["w_gate_up"][:, :F].contiguous()
        wu = inp["w_gate_up"][:, F:].contiguous()
        bg = bu = None
        if inp["b_gate_up"] is not None:
            bg = inp["b_gate_up"][:, :F].contiguous()
            bu = inp["b_gate_up"][:, F:].contiguous()
        a0 = moe.act_params(a.kind, 0 if a.kind == synth.ACT_SWIGLU else a.swiglu_fusion,
                            a.limit, a.alpha, a.beta)
        fns["gemm_act_split"] = lambda: moe.moe_grouped_gemm_act_split(
            perm["expert_input"], wg, wu, perm["seg_end"], a0, bg, bu, out=act_out)
        # and the whole forward with the split weights (same workspace sizes)
        f_out = torch.empty_like(inp["hidden"])
        f_ws = moe._ws(moe.moe_workspace_size(T, H, F, E, K, {"bf16": moe.MOE_BF16,
                       "f16": moe.MOE_F16, "f32": moe.MOE_F32}[cfg.dtype]), dev)
        split_fwd = lambda: moe.moe_ffn_forward_split(  # noqa: E731
            inp["hidden"], inp["logits"], wg, wu, inp["w_down"], p, a0, inp["correction_bias"],
            inp["expert_ids"], bg, bu, inp["b_down"], out=f_out, ws=f_ws)
        fwd = lambda: moe.moe_ffn_forward(  # noqa: E731
            inp["hidden"], inp["logits"], inp["w_gate_up"], inp["w_down"], p, a,
            inp["correction_bias"], inp["expert_ids"], inp["b_gate_up"], inp["b_down"],
            out=f_out, ws=f_ws)
        extra["forward_split_us"] = [round(1e3 * x, 2) for x in timed(split_fwd, args.steps,
                                                                       args.warmup)[0]]
        extra["forward_stacked_us"] = [round(1e3 * x, 2) for x in timed(fwd, args.steps,
                                                                         args.warmup)[0]]
        b = 4 if cfg.dtype == "f32" else 2
        M = T * K
        extra.update({"flops": 2.0 * M * 2 * F * H,
                      "bytes": E * 2 * F * H * b + M * H * b + M * F * b})
    if args.stage == "swiglu":
        # the standalone clamped SwiGLU on the gated intermediate of this
        # workload: [T*K, 2F] -> [T*K, F] with the row layout of its act
        rows, tdt = T * K, inp["hidden"].dtype
        fusion = cfg.swiglu_fusion if cfg.swiglu_fusion in (1, 2) else 2
        lim, al, be = (cfg.limit, cfg.alpha, cfg.beta) if cfg.act == "swiglu" else (7.0, 1.702, 1.0)
        g_in = torch.randn((rows, 2 * F), device=dev).to(tdt)
        s_out = torch.empty((rows, F), dtype=tdt, device=dev)
        fns["swiglu"] = lambda: moe.swiglu(g_in, None, fusion, lim, al, be, out=s_out)
        eb = g_in.element_size()
        extra = {"rows": rows, "I": F, "fusion": fusion, "flops": 0.0,
                 "bytes": rows * 3 * F * eb}
    if args.stage == "fp8_gemm":
        # block-scaled FP8 masked grouped GEMM, DeepSeek-V3-style expert-parallel
        # shapes: 8 local experts of up to 256 rows, N 4096 (2F), K 7168 (H)
        E8, mm, N8, K8 = 8, 256, 4096, 7168
        f8 = synth.make_fp8_masked(E8, mm, N8, K8, seed=3, device=dev)
        f8_out = torch.empty((E8, mm, N8), dtype=torch.bfloat16, device=dev)
        f8_ws = moe._ws(256, dev)
        fns["fp8_gemm"] = lambda: moe.moe_grouped_gemm_fp8_masked(
            f8["a"], f8["a_scale"], f8["b"], f8["b_scale"], f8["counts"], out=f8_out, ws=f8_ws)
        rows = int(f8["counts"].clamp(0, mm).sum())
        extra = {"E": E8, "max_m": mm, "N": N8, "K": K8, "rows": rows,
                 "flops": 2.0 * rows * N8 * K8,
                 "bytes": E8 * N8 * K8 + rows * K8 + rows * N8 * 2
                 + (E8 * mm + E8 * (N8 // 128)) * (K8 // 128) * 4,
                 "tensor_peak_dtype": "fp8 (measured bf16 x 2, the nominal fp8 / bf16 ratio)"}
    st, nl = timed(fns[args.stage], args.steps, args.warmup)
    line = {"stage": args.stage, "workload": args.workload,
            "us": [round(1e3 * x, 2) for x in st], "launches": nl}
    if extra:
        pk, pk_src = load_peaks()
        tpk = pk["bf16_tflops"] * (2.0 if args.stage == "fp8_gemm" else 1.0)
        us = 1e3 * sorted(st)[len(st) // 2]
        tf = extra["flops"] / (us * 1e-6) / 1e12
        gbs = extra["bytes"] / (us * 1e-6) / 1e9
        bound = ("tensor" if extra["flops"] / (tpk * 1e12)
                 > extra["bytes"] / (pk["hbm_gbs"] * 1e9) else "hbm")
        extra.update({"us_median": round(us, 2), "tflops": round(tf, 1), "gbs": round(gbs, 1),
                      "bound": bound,
                      "frac": round(tf / tpk if bound == "tensor" else gbs / pk["hbm_gbs"], 3),
                      "peak_source": pk_src})
        line.update(extra)
    print(json.dumps(line), flush=True)


def cpu_baseline(args, cfg, inp):
    """The oracle, as it stands, on a bounded token sample (host cores)."""
    from mixture_experts_ffn_gb300 import synth
    from oracle import cases
    from oracle import moe_oracle as O

    n = {k: cases.to_np(v) for k, v in inp.items() if k not in ("w_gate_up", "w_down")}
    # each expert's weights reach the host when the oracle asks for them (the
    # whole stacks in float32 would not fit a host's memory on the largest
    # workload); fetching them is inside the timed call
    w1, w2 = HostExperts(inp["w_gate_up"]), HostExperts(inp["w_down"])
    toks = synth.subset_tokens(cfg.T, min(args.cpu_tokens, cfg.T))
    t0 = time.perf_counter()
    O.ffn_forward(n["hidden"], n["logits"], w1, w2, K=cfg.K, F=cfg.F, scoring=cfg.scoring,
                  renormalize=cfg.renormalize, G=cfg.G, TG=cfg.TG, rsf=cfg.rsf,
                  correction_bias=n["correction_bias"], expert_ids=n["expert_ids"],
                  act=cfg.act, fusion=cfg.swiglu_fusion, limit=cfg.limit, alpha=cfg.alpha,
                  beta=cfg.beta, b_gate_up=n["b_gate_up"], b_down=n["b_down"], dtype=cfg.dtype,
                  local_start=cfg.local_start, local_count=cfg.local_count,
                  route_scale=cfg.route_scale, tokens=toks)
    sec = time.perf_counter() - t0
    return {"value": round(len(toks) / sec, 2), "unit": "tokens/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{len(toks)} of the {cfg.T} tokens of the workload (all their routes), "
                      f"numpy float64 with its BLAS threads, {sec:.1f} s (each distinct expert's "
                      f"weights copied to the host and converted inside the timed call)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=None,
                    help="oracle token sample per --impl reference step (default: 2 on the "
                         "DeepSeek-V3-style workload, 8 on gpt-oss-style, else all tokens)")
    ap.add_argument("--cpu-tokens", type=int, default=None,
                    help="oracle token sample of the cpu_baseline leg (default: 8 on the "
                         "DeepSeek-V3-style workload, 64 on gpt-oss-style, else all tokens)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak-s", type=float, default=1.0,
                    help="untimed forward steps run for this long before the timed ones")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="workload recipe (mixture_experts_ffn_gb300.synth.CONFIGS); the bench "
                         "line of record is the default one")
    ap.add_argument("--override", default="",
                    help="KEY=VAL[,KEY=VAL] changes to the workload recipe (profiling of "
                         "reduced cases only; the bench line of record uses none)")
    ap.add_argument("--stage", default=None,
                    choices=["route", "route_permute", "permute", "gemm_act", "gemm_down",
                             "combine", "indexed_mlp", "shared_mlp", "fp8_gemm",
                             "gemm_act_split", "swiglu"],
                    help="time one stage alone (for profiler captures)")
    ap.add_argument("--shared-s", type=int, default=2048,
                    help="intermediate size of the shared expert timed by --stage shared_mlp "
                         "(DeepSeek-V3: 2048)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world, local = dist_env()
    # token samples of the oracle: it converts and applies each distinct
    # expert's weights in float64, so its time grows with the experts hit
    # (about 0.3 s per DeepSeek-V3-sized expert on 8 cores)
    if args.ref_tokens is None:  # per --impl reference step
        args.ref_tokens = {"deepseek_v3_bf16": 2, "gpt_oss_bf16": 8}.get(args.workload, 4096)
    if args.cpu_tokens is None:  # the cpu_baseline leg
        args.cpu_tokens = {"deepseek_v3_bf16": 8, "gpt_oss_bf16": 64}.get(args.workload, 4096)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
