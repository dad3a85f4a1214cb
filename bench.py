#!/usr/bin/env python
"""MoE-layer forward throughput on GB300: one JSON line.

Workload: the Mixtral-8x7B-shaped MoE layer (d_model 4096, 8 experts, top-2,
SwiGLU d_ff 14336, bf16 weights and activations, float32 accumulation) on a
batch of T = 4096 seeded synthetic tokens.  One step = one pass of the whole
layer (router, top-k, softmax, dispatch, expert FFN, combine) over the batch.
The weights (2.8 GB) are larger than L2, so no flush is needed between steps.

Contract: W untimed warm-up steps, then exactly K steps timed with CUDA
events on the launching stream, bracketed by a barrier and a device
synchronize on both sides; the max over ranks is reported.  Under torchrun
each rank runs its own replica on its own GPU over its own tokens (token
parallel, no collective on the data path): weak scaling.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the CPU oracle (float64 numpy) on the host cores on
a bounded sample of the same workload.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

STAGES = ["router", "dispatch", "gather", "expert_up", "expert_down", "combine", "rmsnorm"]

# name -> (synth shape name, default tokens, label, decode-size sweep)
WORKLOADS = {
    "mixtral": ("MIXTRAL", 4096, "Mixtral-8x7B-shaped MoE layer", (1, 16, 128, 512)),
    "qwen2_moe": ("QWEN2", 8192, "Qwen2-MoE-shaped MoE layer (Zipf(1.1) router offset)", (1, 64, 2048)),
    "deepseek_moe": ("DEEPSEEK", 16384, "DeepSeek-MoE-16B-shaped MoE layer", ()),
    "deepseek_moe_masked": ("DEEPSEEK_MASKED", 16384,
                            "DeepSeek-MoE-16B-shaped MoE layer, experts e%4==3 masked", ()),
    "stack": ("MIXTRAL", 64, "32-layer Mixtral-shaped decode stack (RMSNorm, MoE, residual)", ()),
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="mixtral",
                    help="layer workload (default: the Mixtral-shaped layer the metric is quoted on)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="tokens per step (default per workload; batch per step for the stack)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--top-k", type=int, default=None,
                    help="experts per token (default: the shape's); equal to the expert count "
                         "selects soft routing (every expert, softmax over all logits)")
    ap.add_argument("--weights", choices=["bf16", "int8"], default="bf16",
                    help="expert weight format: bf16, or int8 64x64 blocks (converted on the host, "
                         "dequantised to f16 by converter warps of the tensor-core GEMMs)")
    ap.add_argument("--layers", type=int, default=None,
                    help="stack workload: layers per step (default 32, the decode stack; fewer "
                         "only for small profiler captures)")
    ap.add_argument("--no-sweep", action="store_true", help="skip the decode-size sweep")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the block of the other workloads (Qwen2- and DeepSeek-shaped "
                         "layers, int8 weights, the decode stack) in the default run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- helpers


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def algorithmic(shape, T, counts, weights="bf16"):
    """Algorithmic bytes and FLOPs of one layer call (active experts only).

    int8 expert weights: one byte per weight plus 8 bytes (scale, zero point)
    per 64x64 block."""
    d, f, E, k = shape.d_model, shape.d_ff, shape.n_experts, shape.top_k
    s = 2 if shape.dtype == "bf16" else 4
    w = d * f * (1.0 + 8.0 / 4096) if weights == "int8" else d * f * s   # one expert matrix
    active = int((counts > 0).sum())
    return {
        "active_experts": active,
        "bytes": int(active * 3 * w + d * E * s + 2 * T * d * s + T * k * 8),
        "flops": 2 * T * d * E + 6 * T * k * d * f,
        # per kernel
        "up_flops": 4 * T * k * d * f, "down_flops": 2 * T * k * d * f,
        "up_bytes": int(active * 2 * w + T * d * s + T * k * f * s),
        "down_bytes": int(active * w + T * k * f * s + T * k * d * s),
    }


def make_layer(sef, shape, wr, wg, wu, wd, weights, **kw):
    """A library handle over bf16 weights, or over their int8 conversion
    (the library's converter, on the host)."""
    if weights == "int8":
        parts = [tuple(t.to(wr.device) for t in sef.quantize_int8_block64(w)) for w in (wg, wu, wd)]
        return sef.MoELayer(wr, None, None, None, shape.top_k, int8=parts, **kw)
    return sef.MoELayer(wr, wg, wu, wd, shape.top_k, **kw)


def source_sha(*rel):
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


_TC = ("sparse_expert_ffn_gb300/csrc/gemm_tc.cu", "sparse_expert_ffn_gb300/csrc/tc_common.cuh")
_DEC = ("sparse_expert_ffn_gb300/csrc/gemm_dec.cu", "sparse_expert_ffn_gb300/csrc/tc_common.cuh")
KERNEL_SOURCES = {
    "grouped_gemm_tc<kGateUp>": _TC,
    "grouped_gemm_tc<kDown>": _TC,
    "grouped_gemm_dec<kGateUp>": _DEC,
    "grouped_gemm_dec<kDown>": _DEC,
    "ffn_gemv_i8<up>": ("sparse_expert_ffn_gb300/csrc/gemv_i8.cu", "sparse_expert_ffn_gb300/csrc/tc_common.cuh"),
    "ffn_gemv_i8<down>": ("sparse_expert_ffn_gb300/csrc/gemv_i8.cu", "sparse_expert_ffn_gb300/csrc/tc_common.cuh"),
    "ffn_up_stream": ("sparse_expert_ffn_gb300/csrc/ffn_stream.cu", "sparse_expert_ffn_gb300/csrc/common.cuh"),
    "ffn_down_stream": ("sparse_expert_ffn_gb300/csrc/ffn_stream.cu", "sparse_expert_ffn_gb300/csrc/common.cuh"),
}


def traffic_key(workload, T, shape, weights="bf16"):
    """The name a committed ncu summary gives a kernel's workload: the
    workload and token count, plus the experts per token when they differ
    from the shape's own and the weight format when it is not bf16, so that
    one configuration's bytes are never reported for another's."""
    import synth
    base = getattr(synth, WORKLOADS[workload][0]) if workload in WORKLOADS else shape
    key = f"{workload}_T{T}"
    if shape.top_k != base.top_k:
        key += f"_k{shape.top_k}"
    if weights != "bf16":
        key += f"_{weights}"
    return key


def measured_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source.

    A summary line reads:  traffic-per-launch: <kernel> <workload> bytes=<B> source-sha=<sha>
    """
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir) or kernel not in KERNEL_SOURCES:
        return None
    sha = source_sha(*KERNEL_SOURCES[kernel])
    pat = re.compile(r"traffic-per-launch:\s+(\S+)\s+(\S+)\s+bytes=(\d+)\s+source-sha=(\w+)")
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, fn)) as fh:
            for line in fh:
                m = pat.search(line)
                if m and m.group(1) == kernel and m.group(2) == workload and m.group(4) == sha:
                    return int(m.group(3))
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.marks = {}
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "100", "-i", gpu_id],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.p = None

    def _read(self):
        for line in self.p.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, name):
        self.marks[name] = time.time()

    def stop(self):
        if self.p:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self, start="timed_start", end="timed_end"):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        t0, t1 = self.marks.get(start, 0), self.marks.get(end, time.time())
        win = [s for t, s in self.samples if t0 - 0.15 <= t <= t1 + 0.15] or [s for _, s in self.samples]

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(s[1]) for s in win if num(s[1]) is not None]
        mx = [num(s[2]) for s in win if num(s[2]) is not None]
        pw = [num(s[3]) for s in win if num(s[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4)
                          if len(s) > 5 + i and s[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(win)}


# ----------------------------------------------------------------------------- our arm


def dist_setup(args, backend="nccl"):
    """Rank layout from the torchrun environment; one rank per GPU."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device="cuda"):
    """The largest value of v over all ranks (the slowest rank's time)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base_seed, rank):
    """Each rank runs its own replica layer on its own synthetic tokens."""
    return base_seed + rank


def job_throughput(world, tokens_per_rank, steps, max_ms):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (max_ms / 1e3)


def time_steps(layer, x, y, steps, warmup, world, stream, profile=False):
    """W warm-up steps, then K steps between CUDA events; returns (ms, per-stage dict)."""
    import ctypes

    import torch
    import sparse_expert_ffn_gb300 as sef
    for _ in range(warmup):
        layer.forward(x, y)
    torch.cuda.synchronize()
    lib = sef.library()
    if profile:
        lib.colibri_profile_enable(layer.handle, 1)
    n0 = layer.launch_count
    barrier(world)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        layer.forward(x, y, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = a.elapsed_time(b)
    launches = layer.launch_count - n0
    stages = None
    if profile:
        tot = (ctypes.c_double * 7)()
        cnt = (ctypes.c_uint64 * 7)()
        lib.colibri_profile_read(layer.handle, tot, cnt)
        lib.colibri_profile_enable(layer.handle, 0)
        stages = {STAGES[i]: {"ms_total": tot[i], "launches": int(cnt[i])}
                  for i in range(7) if cnt[i]}
    assert layer.check() == 0, "device-side failure during the timed region"
    return ms, launches, stages


L2_BYTES = 129 * 1024 * 1024   # GB300 L2


def time_steps_flushed(layer, x, y, steps, warmup, stream, scratch):
    """Like time_steps for one rank, but L2 is flushed before every step
    (a write of `scratch`, larger than L2) and only the steps are timed, each
    between its own pair of CUDA events: for workloads whose active weights
    would otherwise be served from L2 on the next step."""
    import torch
    for _ in range(warmup):
        layer.forward(x, y, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        scratch.zero_()
        a.record(stream)
        layer.forward(x, y, stream=stream)
        b.record(stream)
    torch.cuda.synchronize()
    assert layer.check() == 0, "device-side failure during the timed region"
    return sum(a.elapsed_time(b) for a, b in ev)


def kernel_name(stage, shape, T, weights):
    """The library kernel behind a profiled stage of a layer call."""
    grouped = shape.dtype == "bf16" and shape.d_model % 256 == 0
    i8 = "_i8" if weights == "int8" else ""
    # int8 codes for at most three tokens: the CUDA-core GEMV, when its
    # gate/up stage has an item (64 hidden units of one expert) per SM
    import torch
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152
    if (weights == "int8" and grouped and T <= 3 and shape.top_k * shape.d_ff // 64 >= n_sms
            and stage in ("expert_up", "expert_down")):
        return "ffn_gemv_i8<up>" if stage == "expert_up" else "ffn_gemv_i8<down>"
    # decode-sized batches (at most 16 pairs per expert on average) run the
    # GEMMs with the weights as the MMA's M operand
    gk = "grouped_gemm_dec" if T * shape.top_k <= 16 * shape.n_experts else "grouped_gemm_tc"
    return {("expert_up", True): gk + "<kGateUp>", ("expert_down", True): gk + "<kDown>",
            ("expert_up", False): "ffn_up_stream" + i8,
            ("expert_down", False): "ffn_down_stream" + i8}.get((stage, grouped), stage)


def dominant_roofline(stages, alg, kname, pk, traffic=None):
    """Roofline of the stage with the largest share of the profiled region.

    `alg` holds the algorithmic FLOPs and bytes of each GEMM summed over the
    launches profiled (one layer call, or every layer of a stack step).  The
    kernel is tensor-bound when its FLOPs take longer at the tensor peak than
    its bytes at the HBM peak (prefill), HBM-bound otherwise (decode sizes)."""
    dom = max(stages, key=lambda s: stages[s]["ms_total"])
    per_launch_s = stages[dom]["ms_total"] / stages[dom]["launches"] / 1e3
    launches_per_call = stages[dom]["launches"] / alg["calls"]
    fl = {"expert_up": alg["up_flops"], "expert_down": alg["down_flops"]}.get(dom, 0) / alg["calls"] / launches_per_call
    by = {"expert_up": alg["up_bytes"], "expert_down": alg["down_bytes"]}.get(dom, alg["bytes"]) / alg["calls"] / launches_per_call
    tensor = fl / (pk["bf16_tflops"] * 1e12) >= by / (pk["hbm_gbs"] * 1e9) and fl > 0
    if tensor:
        achieved = fl / per_launch_s / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / pk["bf16_tflops"], 4),
                "peak_kind": f"bf16 dense burst, {pk['source']}"}
    else:
        achieved = by / per_launch_s / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 4), "peak_kind": f"HBM copy, {pk['source']}"}
    roof["kernel"] = kname(dom)
    roof["share_of_step"] = round(stages[dom]["ms_total"] / sum(v["ms_total"] for v in stages.values()), 4)
    roof["traffic"] = traffic(roof["kernel"]) if traffic else None
    roof["algorithmic_per_launch"] = int(fl if tensor else by)
    return roof


def layer_roofline(alg, step_s, pk):
    """The whole layer's roofline: max(bytes / HBM, FLOPs / tensor peak) over the step time."""
    t_hbm = alg["bytes"] / (pk["hbm_gbs"] * 1e9)
    t_tc = alg["flops"] / (pk["bf16_tflops"] * 1e12)
    return {"bound": "hbm" if t_hbm >= t_tc else "tensor",
            "roofline_time_us": round(1e6 * max(t_hbm, t_tc), 1),
            "step_us": round(step_s * 1e6, 1),
            "frac": round(max(t_hbm, t_tc) / step_s, 4)}


def profile_stages(lib, handles):
    """Per-stage totals of the library's event profiling, summed over handles."""
    import ctypes
    stages = {}
    for hdl in handles:
        tot = (ctypes.c_double * 7)()
        cnt = (ctypes.c_uint64 * 7)()
        lib.colibri_profile_read(hdl, tot, cnt)
        lib.colibri_profile_enable(hdl, 0)
        for i in range(7):
            if cnt[i]:
                st = stages.setdefault(STAGES[i], {"ms_total": 0.0, "launches": 0})
                st["ms_total"] += tot[i]
                st["launches"] += int(cnt[i])
    return stages


def steps_for(t_step_s, floor, target_s=0.08, cap=4000):
    """Enough steps for a timed region of about target_s (so that the clock
    sampler, every 100 ms, sees it), at least `floor`."""
    return int(min(cap, max(floor, math.ceil(target_s / max(t_step_s, 1e-7)))))


def measure_layer(sef, shape, T, weights, seed, dev, stream, pk, steps, warmup, clocks, tag,
                  world=1, name=None, scratch=None):
    """One layer workload: time K steps (L2 flushed before every step when
    the active weights would fit twice in L2), profile the stages, and return
    the entry of the bench line's `workloads` block (and the flush buffer)."""
    import torch

    import synth
    wr = synth.router_weight(shape, seed, 0, dev)
    wg, wu, wd = synth.expert_weights(shape, seed, 0, dev)
    layer = make_layer(sef, shape, wr, wg, wu, wd, weights,
                       router_bias=synth.router_offset(shape), max_tokens=max(T, 128))
    del wr, wg, wu, wd
    torch.cuda.empty_cache()
    try:
        x = synth.tokens(shape, T, seed, 0, dev)
        y = torch.empty_like(x)
        layer.forward(x, y, stream=stream)
        counts = layer.routing()["counts"].cpu().numpy()
        alg = algorithmic(shape, T, counts, weights)
        flush = world == 1 and alg["bytes"] < 2 * L2_BYTES
        if flush and scratch is None:
            scratch = torch.empty(4 * L2_BYTES, dtype=torch.uint8, device=dev)
        # calibrate the step count
        t_cal = (time_steps_flushed(layer, x, y, 3, 1, stream, scratch) if flush else
                 time_steps(layer, x, y, 3, 1, world, stream)[0]) / 3 / 1e3
        k = steps_for(t_cal, steps)
        if clocks:
            clocks.mark(tag + "_start")
        if flush:
            ms = time_steps_flushed(layer, x, y, k, warmup, stream, scratch)
        else:
            ms, _, _ = time_steps(layer, x, y, k, warmup, world, stream)
        if clocks:
            clocks.mark(tag + "_end")
        ms = max_over_ranks(ms, world)
        _, _, stages = time_steps(layer, x, y, min(k, 200), 1, world, stream, profile=True)
        t_step = ms / k / 1e3
        alg["calls"] = min(k, 200)
        for key_ in ("up_flops", "down_flops", "up_bytes", "down_bytes", "bytes", "flops"):
            alg[key_] = alg[key_] * alg["calls"]
        roof = dominant_roofline(stages, alg, lambda st_: kernel_name(st_, shape, T, weights), pk,
                                 lambda kn: measured_traffic(kn, traffic_key(name or shape.name, T, shape, weights)))
        for key_ in ("up_flops", "down_flops", "up_bytes", "down_bytes", "bytes", "flops"):
            alg[key_] = alg[key_] // alg["calls"]
        entry = {"tokens_per_s": round(world * T / t_step, 1),
                 "us_per_step": round(t_step * 1e6, 2),
                 "steps": k,
                 "layer_roofline": layer_roofline(alg, t_step, pk),
                 "roofline": roof,
                 "active_experts": alg["active_experts"],
                 "stages_us": {s_: round(v["ms_total"] * 1e3 / alg["calls"], 1) for s_, v in stages.items()},
                 "clocks": clocks.summary(tag + "_start", tag + "_end") if clocks else None}
        if flush:
            entry["l2"] = "flushed before every step (512 MB write, untimed); steps timed one by one"
        else:
            entry["l2"] = "inputs larger than L2"
        return entry, scratch
    finally:
        layer.close()


def build_stack(sef, B, seed, dev, weights="bf16", n_layers=None):
    import torch

    import synth
    shape = synth.MIXTRAL
    layers = []
    for l in range(n_layers or synth.STACK_LAYERS):
        wr = synth.router_weight(shape, seed, l, dev)
        wg, wu, wd = synth.expert_weights(shape, seed, l, dev)
        layers.append(make_layer(sef, shape, wr, wg, wu, wd, weights, max_tokens=max(B, 1)))
        del wr, wg, wu, wd
    torch.cuda.empty_cache()
    return layers


def measure_stack(sef, layers, B, seed, dev, stream, pk, steps, warmup, clocks, tag, world=1,
                  weights="bf16", exact=False):
    """One decode-stack step = h reset to the batch's input, then the 32
    layers (RMSNorm -> MoE -> residual), over B single-token sequences.
    Times exactly `steps` steps when `exact`, else enough steps for ~0.15 s
    (at least `steps`).  Returns (entry, launches in the timed region, steps
    timed, the batch's input)."""
    import torch

    import synth
    shape = synth.MIXTRAL
    lib = sef.library()
    gamma = torch.ones(shape.d_model, dtype=torch.bfloat16, device=dev)
    h0 = synth.tokens(shape, B, seed, 0, dev)
    h = h0.clone()

    def step():
        h.copy_(h0)       # every step starts from the same hidden state
        for layer in layers:
            layer.forward_stack_layer(h, gamma, synth.STACK_EPS, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()

    def timed(k, profile):
        for layer in layers:
            lib.colibri_profile_enable(layer.handle, 1 if profile else 0)
        n0 = sum(l.launch_count for l in layers)
        barrier(world)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(k):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(a.elapsed_time(b), world), sum(l.launch_count for l in layers) - n0

    if exact:
        k = steps
    else:
        ms_cal, _ = timed(2, False)
        k = steps_for(ms_cal / 2 / 1e3, steps, target_s=0.15, cap=200)
    if clocks:
        clocks.mark(tag + "_start")
    ms, launches = timed(k, False)
    if clocks:
        clocks.mark(tag + "_end")
    time.sleep(0.5)
    kp = min(k, 10)
    ms_prof, _ = timed(kp, True)
    stages = profile_stages(lib, [l.handle for l in layers])
    # per-layer algorithmic work of one step (every step routes alike: h is reset)
    alg = {"calls": kp, "up_flops": 0, "down_flops": 0, "up_bytes": 0, "down_bytes": 0,
           "bytes": 0, "flops": 0}
    active = 0
    for layer in layers:
        a_l = algorithmic(shape, B, layer.routing()["counts"].cpu().numpy(), weights)
        active += a_l["active_experts"]
        for key_ in ("up_flops", "down_flops", "up_bytes", "down_bytes", "bytes", "flops"):
            alg[key_] += a_l[key_]
        assert layer.check() == 0
    # RMSNorm reads and writes the hidden state once more per layer
    alg["bytes"] += len(layers) * (2 * B * shape.d_model * 2 + shape.d_model * 2)
    step_s = ms / k / 1e3
    per_step = dict(alg)
    for key_ in ("up_flops", "down_flops", "up_bytes", "down_bytes", "bytes", "flops"):
        alg[key_] *= kp
    roof = dominant_roofline(stages, alg, lambda st_: kernel_name(st_, shape, B, weights), pk,
                             lambda kn: measured_traffic(kn, traffic_key("stack", B, shape, weights)))
    entry = {"tokens_per_s": round(world * B / step_s, 1),
             "ms_per_step": round(step_s * 1e3, 4),
             "steps": k,
             "stack_roofline": {"bound": "hbm", "bytes_per_step": int(per_step["bytes"]),
                                "achieved_gbs": round(per_step["bytes"] / step_s / 1e9, 1),
                                "peak": pk["hbm_gbs"],
                                "frac": round(per_step["bytes"] / step_s / 1e9 / pk["hbm_gbs"], 4),
                                "active_experts_per_step": active},
             "roofline": roof,
             "stages_us_per_step": {s_: round(v["ms_total"] * 1e3 / kp, 1) for s_, v in stages.items()},
             "ms_per_step_profiled": round(ms_prof / kp, 4),
             "clocks": clocks.summary(tag + "_start", tag + "_end") if clocks else None,
             "l2": f"inputs larger than L2 ({sum(l.bytes[0] for l in layers) / 1e9:.0f} GB of weights)"}
    return entry, int(launches), k, h0


def gpu_id_of(dev):
    import torch
    props = torch.cuda.get_device_properties(dev)
    uid = str(getattr(props, "uuid", "") or "")
    return (uid if uid.startswith("GPU-") else "GPU-" + uid) if uid else str(dev.index or 0)


def run_ours(args):
    import numpy as np
    import torch

    import sparse_expert_ffn_gb300 as sef
    import synth

    world, rank, local = dist_setup(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    shape_name, T_default, label, sweep_T = WORKLOADS[args.workload]
    shape = getattr(synth, shape_name)
    if args.top_k:
        from dataclasses import replace
        shape = replace(shape, top_k=args.top_k)
        label += ", soft routing" if args.top_k == shape.n_experts else f", top-{args.top_k}"
    T = args.tokens or T_default
    pk = peaks()
    clocks = ClockSampler(gpu_id_of(dev)) if rank == 0 else None

    # weights: layer seed per rank (replicas over independent synthetic layers)
    seed = rank_seed(args.seed, rank)
    wr = synth.router_weight(shape, seed, 0, dev)
    wg, wu, wd = synth.expert_weights(shape, seed, 0, dev)
    max_t = max(T, 128)
    layer = make_layer(sef, shape, wr, wg, wu, wd, args.weights,
                       router_bias=synth.router_offset(shape), max_tokens=max_t)
    weight_gb = (wg.numel() + wu.numel() + wd.numel()) * (1 if args.weights == "int8" else wg.element_size()) / 1e9
    del wg, wu, wd
    torch.cuda.empty_cache()
    x = synth.tokens(shape, T, seed, 0, dev)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream()

    if clocks:
        clocks.mark("warm_start")
    layer.forward(x, y)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark("timed_start")
    ms, launches, _ = time_steps(layer, x, y, args.steps, args.warmup, world, stream)
    if clocks:
        clocks.mark("timed_end")
    ms = max_over_ranks(ms, world)
    # Per-stage kernel times: the same K steps again with an event pair around
    # every launch (the events also stop consecutive kernels from overlapping
    # their launch, so this pass runs a little slower than the headline one).
    time.sleep(1.0)   # same power state as the headline pass
    ms_prof, _, stages = time_steps(layer, x, y, args.steps, 1, world, stream, profile=True)
    ms_prof = max_over_ranks(ms_prof, world)
    r = layer.routing()
    counts = r["counts"].cpu().numpy()
    alg = algorithmic(shape, T, counts, args.weights)
    step_ms = ms / args.steps
    value = job_throughput(world, T, args.steps, ms)

    # roofline of the dominant kernel (largest share of the profiled region)
    alg_run = dict(alg, calls=args.steps)
    for key_ in ("up_flops", "down_flops", "up_bytes", "down_bytes", "bytes", "flops"):
        alg_run[key_] = alg[key_] * args.steps
    wkey = traffic_key(args.workload, T, shape, args.weights)
    roof = dominant_roofline(stages, alg_run, lambda st_: kernel_name(st_, shape, T, args.weights), pk,
                             lambda kn: measured_traffic(kn, wkey))
    whole = layer_roofline(alg, step_ms / 1e3, pk)

    # end to end through the public C API on pinned host buffers: every step
    # uploads x and downloads y; the pipelined calls overlap one step's copies
    # with another step's layer, and the clock stops once the last y is home
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        layer.forward_host(xh, yh)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        layer.forward_host_async(xh, yh)
    layer.host_wait()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e = {"value": round(world * T * e2e_steps / e2e_s, 1), "unit": "tokens/s",
           "h2d_bytes_per_step": int(xh.numel() * xh.element_size()),
           "d2h_bytes_per_step": int(yh.numel() * yh.element_size())}

    # decode-size sweep (context; the headline is the T above)
    sweep = {}
    scratch = None
    if not args.no_sweep:
        for Ts in [t for t in sweep_T if t <= max_t]:
            xs = synth.tokens(shape, Ts, seed, 0, dev)
            ys = torch.empty_like(xs)
            layer.forward(xs, ys, stream=stream)
            cs = layer.routing()["counts"].cpu().numpy()
            a_s = algorithmic(shape, Ts, cs, args.weights)
            # active weights that fit twice in L2 would be served from it on
            # the next step: flush L2 between steps, time the steps alone
            flush = world == 1 and a_s["bytes"] < 2 * L2_BYTES
            if flush:
                if scratch is None:
                    scratch = torch.empty(4 * L2_BYTES, dtype=torch.uint8, device=dev)
                ms_s = time_steps_flushed(layer, xs, ys, args.steps, args.warmup, stream, scratch)
            else:
                ms_s, _, _ = time_steps(layer, xs, ys, args.steps, args.warmup, world, stream)
            _, _, st_s = time_steps(layer, xs, ys, args.steps, 1, world, stream, profile=True)
            ms_s = max_over_ranks(ms_s, world)
            t_step = ms_s / args.steps / 1e3
            entry = {"tokens_per_s": round(world * Ts / t_step, 1),
                     "us_per_step": round(t_step * 1e6, 1),
                     "hbm_frac_of_measured": round(a_s["bytes"] / t_step / 1e9 / pk["hbm_gbs"], 4),
                     "active_experts": a_s["active_experts"],
                     "stages_us": {k: round(v["ms_total"] * 1e3 / args.steps, 1)
                                   for k, v in st_s.items()}}
            if flush:
                entry["l2"] = "flushed before every step (512 MB write, untimed); steps timed one by one"
            sweep[f"T{Ts}"] = entry
    layer.close()
    del x, y
    torch.cuda.empty_cache()

    # the other workloads, each timed and clock-sampled on its own (default run only)
    workloads = None
    if (not args.no_workloads and args.workload == "mixtral" and args.tokens is None
            and not args.top_k and args.weights == "bf16"):
        workloads = {}
        wsteps, wwarm = max(3, min(args.steps, 10)), max(3, min(args.warmup, 5))
        plan = [("qwen2_moe", synth.QWEN2, 1, "bf16"), ("qwen2_moe", synth.QWEN2, 64, "bf16"),
                ("qwen2_moe", synth.QWEN2, 2048, "bf16"), ("qwen2_moe", synth.QWEN2, 8192, "bf16"),
                ("deepseek_moe", synth.DEEPSEEK, 16384, "bf16"),
                ("deepseek_moe_masked", synth.DEEPSEEK_MASKED, 16384, "bf16"),
                ("mixtral", synth.MIXTRAL, 1, "int8"), ("mixtral", synth.MIXTRAL, 4096, "int8")]
        for wl, shp, Tw, wt in plan:
            tag = f"{wl}_T{Tw}" + ("" if wt == "bf16" else f"_{wt}")
            entry, scratch = measure_layer(sef, shp, Tw, wt, seed, dev, stream, pk, wsteps, wwarm,
                                           clocks, tag, world, name=wl, scratch=scratch)
            entry["workload"] = f"{WORKLOADS[wl][2]}, T={Tw} tokens" + \
                ("" if wt == "bf16" else f", {wt} expert weights")
            workloads[tag] = entry
        scratch = None
        torch.cuda.empty_cache()
        layers = build_stack(sef, max(synth.STACK_BATCHES), seed, dev)
        try:
            for B in synth.STACK_BATCHES:
                entry, _, _, _ = measure_stack(sef, layers, B, seed, dev, stream, pk, wsteps, wwarm,
                                               clocks, f"stack_B{B}", world)
                entry["workload"] = f"{WORKLOADS['stack'][2]}, batch {B}"
                workloads[f"stack_B{B}"] = entry
        finally:
            for l_ in layers:
                l_.close()
            torch.cuda.empty_cache()
    if clocks:
        clocks.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(shape, T, seed=seed, target_s=args.cpu_seconds)

    out = {
        "metric": "MoE-layer tokens/s at 1 GB300; % of HBM (decode) / bf16 TC (prefill) roofline",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{label}, T={T} tokens" + (", int8 expert weights" if args.weights == "int8" else ""),
                   "weights": args.weights,
                   "d_model": shape.d_model, "d_ff": shape.d_ff, "n_experts": shape.n_experts,
                   "top_k": shape.top_k, "tokens_per_gpu": T, "parallelism": f"token-parallel x{world}",
                   "l2": f"inputs larger than L2 ({weight_gb:.2f} GB of expert weights per step)"},
        "roofline": roof,
        "layer_roofline": whole,
        "stages_us_per_step": {k: round(v["ms_total"] * 1e3 / args.steps, 1) for k, v in stages.items()},
        "ms_per_step_profiled": round(ms_prof / args.steps, 4),
        "active_experts": alg["active_experts"],
        "gpu_launches": int(launches),
        "e2e": e2e,
        "clocks": clocks.summary() if clocks else None,
        "cpu_baseline": cpu,
        "sweep": sweep,
    }
    if workloads is not None:
        out["workloads"] = workloads
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_stack(args):
    """One step = 32 Mixtral-shaped layers, each RMSNorm -> MoE -> residual,
    over a batch of B single-token sequences; weight-streaming bound."""
    import torch

    import sparse_expert_ffn_gb300 as sef
    import synth

    world, rank, local = dist_setup(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    shape, B = synth.MIXTRAL, args.tokens or 64
    pk = peaks()
    seed = rank_seed(args.seed, rank)
    clocks = ClockSampler(gpu_id_of(dev)) if rank == 0 else None
    stream = torch.cuda.current_stream()
    layers = build_stack(sef, B, seed, dev, args.weights, args.layers)
    entry, launches, k, h0 = measure_stack(sef, layers, B, seed, dev, stream, pk, args.steps,
                                           args.warmup, clocks, "timed", world, args.weights,
                                           exact=True)
    step_ms = entry["ms_per_step"]

    # end to end through the public API on pinned host buffers: every step
    # uploads the batch's hidden state, runs the 32 layers in place and
    # downloads the result
    gamma = torch.ones(shape.d_model, dtype=torch.bfloat16, device=dev)
    hh = h0.cpu().pin_memory()
    oh = torch.empty_like(hh).pin_memory()
    h = torch.empty_like(h0)
    e2e_steps = max(3, min(k, 20))

    def host_step():
        h.copy_(hh, non_blocking=True)
        for layer in layers:
            layer.forward_stack_layer(h, gamma, synth.STACK_EPS, stream=stream)
        oh.copy_(h, non_blocking=True)

    host_step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        host_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e = {"value": round(world * B * e2e_steps / e2e_s, 1), "unit": "tokens/s",
           "h2d_bytes_per_step": int(hh.numel() * hh.element_size()),
           "d2h_bytes_per_step": int(oh.numel() * oh.element_size())}
    if clocks:
        clocks.stop()
    for layer in layers:
        layer.close()
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = stack_cpu_baseline(B, seed, target_s=args.cpu_seconds)

    out = {
        "metric": "MoE-layer tokens/s at 1 GB300; % of HBM (decode) / bf16 TC (prefill) roofline",
        "value": entry["tokens_per_s"], "unit": "tokens/s",
        "n_gpus": world, "steps": k, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{WORKLOADS['stack'][2]}, batch {B}" + (", int8 expert weights" if args.weights == "int8" else ""),
                   "weights": args.weights, "layers": args.layers or synth.STACK_LAYERS,
                   "batch": B, "parallelism": f"token-parallel x{world}",
                   "l2": entry["l2"]},
        "roofline": entry["roofline"],
        "stack_roofline": entry["stack_roofline"],
        "stages_us_per_step": entry["stages_us_per_step"],
        "ms_per_step_profiled": entry["ms_per_step_profiled"],
        "gpu_launches": launches,
        "e2e": e2e,
        "clocks": entry["clocks"],
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


# ----------------------------------------------------------------------------- oracle (CPU)


def _host_inputs(shape, T, seed):
    """Workload inputs on the host: generated on the GPU when one is present
    (the counter-based generator gives the same values either way)."""
    import torch

    import synth
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wr = synth.router_weight(shape, seed, 0, dev).cpu()
    wg, wu, wd = synth.expert_weights(shape, seed, 0, dev)
    wg, wu, wd = wg.cpu(), wu.cpu(), wd.cpu()
    x = synth.tokens(shape, T, seed, 0, dev).cpu()
    return x, wr, wg, wu, wd


def _oracle_weights(wr, wg, wu, wd):
    import oracle
    return (oracle.to_f64(wr), oracle.to_f64(wg), oracle.to_f64(wu), oracle.to_f64(wd))


def cpu_baseline(shape, T, seed=0, target_s=15.0):
    """The oracle, as it stands, on a bounded sample of the workload's tokens."""
    import oracle
    import synth
    xh, wr, wg, wu, wd = _host_inputs(shape, T, seed)
    W = _oracle_weights(wr, wg, wu, wd)
    del wg, wu, wd
    x64 = oracle.to_f64(xh)
    # calibrate on 16 tokens, then size the sample to ~target_s seconds
    off = synth.router_offset(shape)
    off = None if off is None else off.double().numpy()
    t0 = time.perf_counter()
    oracle.moe_layer(x64[:64], *W, shape.top_k, off)
    per_tok = (time.perf_counter() - t0) / 64
    n = int(min(x64.shape[0], max(16, target_s / max(per_tok, 1e-9))))
    t0 = time.perf_counter()
    oracle.moe_layer(x64[:n], *W, shape.top_k, off)
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(n / dt, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} of the {x64.shape[0]} tokens, whole layer (float64 numpy, BLAS "
                      f"threads = all {cores} cores), {dt:.1f} s"}


def stack_cpu_baseline(B, seed=0, target_s=15.0):
    """The oracle's stack layer (RMSNorm, MoE, residual), as it stands, on
    the batch's hidden state, for as many of the 32 layers as fit in about
    target_s (at least one), scaled to a 32-layer step.  Converting a layer's
    weights to float64 for the oracle is not timed."""
    import numpy as np
    import torch

    import oracle
    import synth
    shape = synth.MIXTRAL
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    h = oracle.to_f64(synth.tokens(shape, B, seed, 0, dev).cpu())
    g = np.ones(shape.d_model)
    spent, done = 0.0, 0
    for l in range(synth.STACK_LAYERS):
        wr = synth.router_weight(shape, seed, l, dev).cpu()
        wg, wu, wd = synth.expert_weights(shape, seed, l, dev)
        W = _oracle_weights(wr, wg.cpu(), wu.cpu(), wd.cpu())
        del wg, wu, wd
        t0 = time.perf_counter()
        h = oracle.stack_layer(h, g, synth.STACK_EPS, *W, shape.top_k)["h_out"]
        spent += time.perf_counter() - t0
        done += 1
        del W
        if spent * (done + 1) / done > target_s:
            break
    step_s = spent / done * synth.STACK_LAYERS
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(B / step_s, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"the first {done} of the 32 layers at batch {B} ({spent:.1f} s, float64 "
                      f"numpy, BLAS threads = all {cores} cores), scaled to a 32-layer step"}


def run_reference(args):
    import numpy as np

    import oracle
    import synth
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = "mixtral" if args.workload == "stack" else args.workload
    shape_name, T_default, label, _ = WORKLOADS[wl]
    shape = getattr(synth, shape_name)
    T = args.tokens or T_default
    xh, wr, wg, wu, wd = _host_inputs(shape, T, args.seed)
    off = synth.router_offset(shape)
    off = None if off is None else off.double().numpy()
    W = _oracle_weights(wr, wg, wu, wd)
    del wg, wu, wd
    x64 = oracle.to_f64(xh)
    t0 = time.perf_counter()
    oracle.moe_layer(x64[:8], *W, shape.top_k, off)
    per_tok = (time.perf_counter() - t0) / 8
    # each step: a bounded sample sized so that W + K steps take ~2 minutes
    n = int(max(4, min(T, 120.0 / max(per_tok, 1e-9) / max(1, args.steps + args.warmup))))
    for i in range(args.warmup):
        oracle.moe_layer(x64[:n], *W, shape.top_k, off)
    t0 = time.perf_counter()
    for i in range(args.steps):
        lo = (i * n) % max(1, T - n)
        oracle.moe_layer(x64[lo:lo + n], *W, shape.top_k, off)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = f"{n} tokens per step out of the T={T} batch, whole layer, float64 numpy"
    out = {"impl": "reference",
           "metric": "MoE-layer tokens/s at 1 GB300; % of HBM (decode) / bf16 TC (prefill) roofline",
           "value": round(value, 3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": f"{label}, T={T} tokens",
                      "d_model": shape.d_model, "d_ff": shape.d_ff, "n_experts": shape.n_experts,
                      "top_k": shape.top_k, "tokens_per_gpu": T, "parallelism": "none (host CPU)"},
           "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "stack":
        run_stack(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
