"""Benchmark of the one-launch Event Tensor MoE megakernel on GB300.

Default workload (the pages' MoE-layer benchmark shape): Qwen3-30B-A3B-shaped
MoE layer (hidden 2048, 128 experts, top-8, intermediate 768, SwiGLU),
prefill T=4096 with Zipf(1.2)-skewed routing, bf16 weights, fp32 accumulation,
synthetic seeded inputs.  A step is one MoE layer forward (router, top-k,
counts/exp_indptr scan, permute, GroupGEMM gate/up+SwiGLU, GroupGEMM down,
combine) = ONE kernel launch of the megakernel; the benchmark line takes the
mixed scheduler (routing walked statically, expert tiles from the queue), the
fastest of the three on this workload (--sched static or dynamic for the
others; every one of them is also timed in the ablation).

One JSON line on stdout (rank 0).  Extra keys report the decode sizes,
the static/dynamic/unfused ablation, the split-K task graph and the chain.

Multi-GPU: replicas only (token-sharded data parallelism, no collective on
the data path); each rank runs its own T=4096 batch, `value` sums all ranks.

--impl reference times the fp64 C++ oracle (the only reference this method
has) on a bounded token sample on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s and µs/layer on 1 GB300; % of HBM/bf16-tensor roofline"
H, E, K, I = 2048, 128, 8, 768
FLOPS_PER_TOKEN = 2 * K * (H * 2 * I + I * H) + 2 * H * E   # 75,497,472 + 524,288
EXPERT_BYTES = (2 * I * H + H * I) * 2                       # 9,437,184
ROUTER_BYTES = H * E * 2                                     # 524,288
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of ONE launch of the
# benchmark line's kernel (mixed scheduler, prefill T=4096), from one ncu capture.
# Valid only for the kernel sources it was taken on: reported as null once any
# of them changes.
MEGAKERNEL_SOURCES = ("moe_kernel.cu", "moe_api.cu", "etc_internal.h", "etc_event.cuh", "etc_ptx.cuh")
NCU_TRAFFIC = {"sources_sha256_16": "f5d7382a32b87ca3", "bytes_per_launch": 1218420224 + 251629312}


def megakernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for name in MEGAKERNEL_SOURCES:
        with open(os.path.join(ROOT, "moe_layer_scheduling_gb300", "csrc", name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# distributed helpers (replicas)
# ---------------------------------------------------------------------------

def dist_init():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.samples = []
        self.proc = None
        self.uuid = uuid
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                self.samples.append((time.time(), float(parts[0]), float(parts[1]),
                                     float(parts[2]) if parts[2] not in ("[N/A]", "N/A") else 0.0,
                                     parts[4:8]))
            except ValueError:
                continue

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        if len(win) < 3:
            win = [s for s in self.samples if s[3] > 0] or self.samples
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i, v in enumerate(s[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": max(s[2] for s in win),
                "reasons": reasons, "samples": len(win)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def make_layer(T, weights, skew):
    from moe_layer_scheduling_gb300 import inputs
    if skew:
        return inputs.prefill_skew_layer(T, weights)
    return inputs.decode_layer(T, weights)


def time_gpu(fn, steps, warmup, world, stream=None, between=None):
    """Returns seconds per step (max over ranks), device-timed with CUDA events."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    if between is None:
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(steps):
            fn()
        e.record()
        torch.cuda.synchronize()
        sec = s.elapsed_time(e) / 1e3 / steps
    else:
        total = 0.0
        for i in range(steps):
            between(i)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            fn()
            e.record()
            torch.cuda.synchronize()
            total += s.elapsed_time(e) / 1e3
        sec = total / steps
    barrier(world)
    return max_over_ranks(sec, world)


def time_e2e_pipelined(B, plan, x_host, weights, T, H, steps, warmup, world, dev):
    """End to end through the C ABI with host buffers.  Every step copies its input from
    pinned host memory to the device, runs the layer and copies its output back into pinned
    host memory.  Steps are pipelined over two device buffers and three streams, as a
    serving loop runs them: step i's input copy and step i-1's output copy overlap step
    i's kernel.  Returns (seconds per step, max over ranks; the last output on the host)."""
    import torch
    gw, wgu, wd = weights
    cs, ks, os_ = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    xb = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    ob = [torch.empty(T, H, dtype=torch.float32, device=dev) for _ in range(2)]
    oh = [torch.empty(T, H, dtype=torch.float32).pin_memory() for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_k = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        for i in range(n):
            b = i % 2
            if i >= 2:
                cs.wait_event(ev_k[b])  # step i-2's kernel has read xb[b]
            with torch.cuda.stream(cs):
                xb[b].copy_(x_host, non_blocking=True)
            ev_in[b].record(cs)
            ks.wait_event(ev_in[b])
            if i >= 2:
                ks.wait_event(ev_out[b])  # step i-2's output has left ob[b]
            B.etc_moe_forward(plan, xb[b], gw, wgu, wd, T, ob[b], stream=ks)
            ev_k[b].record(ks)
            os_.wait_event(ev_k[b])
            with torch.cuda.stream(os_):
                oh[b].copy_(ob[b], non_blocking=True)
            ev_out[b].record(os_)

    run(warmup)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(cs)  # every stream is idle here
    run(steps)
    e.record(os_)  # after the last output copy, which follows every earlier step
    torch.cuda.synchronize()
    sec = s.elapsed_time(e) / 1e3 / steps
    barrier(world)
    return max_over_ranks(sec, world), oh[(steps - 1) % 2].clone()


def run_ours(args, rank, world):
    import numpy as np
    import torch

    from moe_layer_scheduling_gb300 import binding as B
    from moe_layer_scheduling_gb300 import build as libbuild
    from moe_layer_scheduling_gb300 import inputs

    libbuild.build()
    peaks, peak_src = load_peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    if not uuid.startswith("GPU-"):
        uuid = "GPU-" + uuid
    sampler = ClockSampler(uuid)
    sampler.start()

    weights = inputs.qwen_weights(0)
    gw, wgu, wd = weights.gate_w.to(dev), weights.w_gate_up.to(dev), weights.w_down.to(dev)
    T = args.tokens
    wl = make_layer(T, weights, skew=True)
    bias = wl.weights.router_bias.to(dev)
    x = wl.x.to(dev)
    out = torch.empty(T, H, dtype=torch.float32, device=dev)
    launches0 = B.etc_launch_count()
    results = {}
    plans = {}
    for name, sched in (("dynamic", B.ETC_SCHED_DYNAMIC), ("static", B.ETC_SCHED_STATIC),
                        ("mixed", B.ETC_SCHED_MIXED)):
        plans[name] = B.etc_moe_plan(H, E, K, I, t_max=T, sched=sched, router_bias=bias)

    # ---- headline: the one-launch megakernel (--sched), inputs resident in HBM ----
    plan = plans[args.sched]
    step = lambda: B.etc_moe_forward(plan, x, gw, wgu, wd, T, out)  # noqa: E731
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches_before = B.etc_launch_count()
    s.record()
    for _ in range(args.steps):
        step()
    e.record()
    torch.cuda.synchronize()
    t1 = time.time()
    launches_timed = B.etc_launch_count() - launches_before
    barrier(world)
    sec = max_over_ranks(s.elapsed_time(e) / 1e3 / args.steps, world)
    assert B.etc_plan_check(plan) == B.ETC_OK, B.etc_last_error()
    # keep the GPU loaded ~1.5 s more for the clock record if the timed region was short
    if t1 - t0 < args.clock_window:
        tl = time.time()
        while time.time() - tl < args.clock_window:
            for _ in range(20):
                step()
            torch.cuda.synchronize()
        t1 = time.time()
    clocks = sampler.summary(t0, t1)

    flops = T * FLOPS_PER_TOKEN
    achieved_tflops = flops / sec / 1e12
    if megakernel_source_hash() == NCU_TRAFFIC["sources_sha256_16"]:
        traffic = NCU_TRAFFIC["bytes_per_launch"]
        traffic_src = ("bytes per launch, ncu dram__bytes_read.sum + dram__bytes_write.sum of one "
                       "launch of this kernel on this workload")
    else:
        traffic, traffic_src = None, "kernel sources changed since the ncu capture"
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    results["prefill_T4096"] = {"us": sec * 1e6, "tok_s": T / sec, "tflops": achieved_tflops}

    # routing realised on this workload
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    B.etc_moe_debug_routing(plan, 0, None, None, None, counts, None, None)
    torch.cuda.synchronize()
    cnt = counts.cpu().numpy()

    # ---- e2e through the C ABI with host buffers (H2D of x, D2H of out, every step) ----
    x_host = wl.x.pin_memory()
    e2e_sec, last_host = time_e2e_pipelined(B, plan, x_host, (gw, wgu, wd), T, H, args.steps,
                                            max(2, args.warmup), world, dev)
    ref_out = out.float().cpu()
    rms = float(ref_out.pow(2).mean().sqrt())
    assert float((last_host - ref_out).abs().max()) <= 1e-3 * rms, "e2e output differs"

    extra = {}
    if not args.no_extra:
        extra = run_extras(args, dev, weights, gw, wgu, wd, bias, x, out, T, plans, peaks, world)

    for p in plans.values():
        p.close()
    per_rank_units = T
    value = per_rank_units * world / sec
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": sec * 1e3,
        "us_per_layer": sec * 1e6,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded normal weights/activations, Zipf(1.2) router bias)",
        "config": {
            "workload": "qwen3_30b_a3b_moe_prefill_T4096_zipf1.2",
            "hidden": H, "experts": E, "top_k": K, "inter": I, "tokens_per_gpu": T,
            "global_tokens": T * world, "scheduler": f"{args.sched} megakernel (1 launch/layer)",
            "parallelism": f"replicas x{world} (token-sharded, no collective)",
            "l2": "inputs larger than L2 (1.2 GB of expert weights touched per step)",
            "experts_with_tokens": int((cnt > 0).sum()), "max_rows_per_expert": int(cnt.max()),
        },
        "roofline": {
            "bound": "tensor", "achieved": achieved_tflops, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved_tflops / peak, "traffic": traffic,
            "traffic_source": traffic_src,
            "kernel": f"etc_moe_megakernel ({args.sched})",
            "peak_source": f"bf16_tflops (burst) of {peak_src} MEASURED_PEAKS.json"
            if peak_src == "measured" else "fallback 1.9 PFLOP/s",
            "algorithmic_flops_per_launch": flops,
        },
        "e2e": {"value": T * world / e2e_sec, "unit": "tokens/s",
                "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 4,
                "pipelining": "two device buffers; a step's input and output copies overlap "
                              "the neighbouring steps' kernels"},
        "gpu_launches": int(launches_timed),
        "clocks": clocks,
    }
    line.update(extra)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, wl, budget_s=args.cpu_budget)
    sampler.stop()
    return line


def run_extras(args, dev, weights, gw, wgu, wd, bias, x, out, T, plans, peaks, world):
    import numpy as np
    import torch

    from moe_layer_scheduling_gb300 import binding as B
    from moe_layer_scheduling_gb300 import inputs
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    tflops_peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    res = {}
    steps = max(5, min(args.steps, 50))
    # --- Table 2 analogue on the prefill workload: static / dynamic / unfused ---
    abl = {}
    for name in ("static", "dynamic", "mixed"):
        p = plans[name]
        sec = time_gpu(lambda: B.etc_moe_forward(p, x, gw, wgu, wd, T, out), steps, 3, world)
        abl[name] = {"us": sec * 1e6, "tflops": T * FLOPS_PER_TOKEN / sec / 1e12}
    p = plans["static"]
    sec = time_gpu(lambda: B.etc_moe_forward_unfused(p, x, gw, wgu, wd, T, out), steps, 3, world)
    abl["unfused_per_stage"] = {"us": sec * 1e6, "tflops": T * FLOPS_PER_TOKEN / sec / 1e12}
    for name in ("static", "dynamic", "mixed"):
        abl[name]["vs_unfused"] = abl["unfused_per_stage"]["us"] / abl[name]["us"]
    # the same call on CTA-pair tiles, with the ordered (deterministic) combine,
    # with swap-AB wide tiles, and (mixed) without heavy experts
    for name, sched, kw in (
            ("static_pair_tiles", B.ETC_SCHED_STATIC, dict(debug_flags=B.ETC_DEBUG_PAIR_MOE)),
            ("static_ordered_combine", B.ETC_SCHED_STATIC, dict(combine=B.ETC_COMBINE_ORDERED)),
            ("static_swap_ab_wide_tiles", B.ETC_SCHED_STATIC, dict(debug_flags=B.ETC_DEBUG_WIDE_SWAP_AB)),
            ("mixed_no_heavy_experts", B.ETC_SCHED_MIXED, dict(debug_flags=B.ETC_DEBUG_NO_HEAVY))):
        pv = B.etc_moe_plan(H, E, K, I, t_max=T, sched=sched, router_bias=bias, **kw)
        sec = time_gpu(lambda: B.etc_moe_forward(pv, x, gw, wgu, wd, T, out), steps, 3, world)
        assert B.etc_plan_check(pv) == B.ETC_OK, B.etc_last_error()
        abl[name] = {"us": sec * 1e6, "tflops": T * FLOPS_PER_TOKEN / sec / 1e12}
        pv.close()
    res["ablation_prefill_T4096"] = abl

    # --- decode sizes: 8 rotating weight copies defeat the 129 MB L2 ---
    copies = [(gw, wgu, wd)]
    for _ in range(7):
        copies.append((gw.clone(), wgu.clone(), wd.clone()))
    dec = {}
    for Td in (1, 8, 32, 64):
        xd = inputs.decode_layer(Td, weights).x.to(dev)
        od = torch.empty(Td, H, dtype=torch.float32, device=dev)
        row = {}
        for name, sched in (("dynamic", B.ETC_SCHED_DYNAMIC), ("static", B.ETC_SCHED_STATIC),
                            ("mixed", B.ETC_SCHED_MIXED)):
            pd = B.etc_moe_plan(H, E, K, I, t_max=64, sched=sched)
            idx = [0]

            def f():
                g, a, b = copies[idx[0] % len(copies)]
                idx[0] += 1
                B.etc_moe_forward(pd, xd, g, a, b, Td, od)

            sec = time_gpu(f, 8 * 4, 8, world)
            cnt = torch.empty(E, dtype=torch.int32, device=dev)
            B.etc_moe_debug_routing(pd, 0, None, None, None, cnt, None, None)
            torch.cuda.synchronize()
            D = int((cnt.cpu().numpy() > 0).sum())
            bytes_ = D * EXPERT_BYTES + ROUTER_BYTES + 4 * Td * H
            row[name] = {"us": sec * 1e6, "tok_s": Td / sec, "hbm_gbs": bytes_ / sec / 1e9,
                         "hbm_frac": bytes_ / sec / 1e9 / hbm, "touched_experts": D}
            if name == "static":
                # the per-stage build on the same inputs, timed the same way:
                # the same 8 rotating weight copies, so its weights also come from HBM
                idx[0] = 0

                def fu():
                    g, a, b = copies[idx[0] % len(copies)]
                    idx[0] += 1
                    B.etc_moe_forward_unfused(pd, xd, g, a, b, Td, od)

                secu = time_gpu(fu, 8 * 4, 8, world)
                row["unfused"] = {"us": secu * 1e6, "tok_s": Td / secu, "hbm_gbs": bytes_ / secu / 1e9,
                                  "hbm_frac": bytes_ / secu / 1e9 / hbm, "touched_experts": D}
            pd.close()
        for name in ("static", "dynamic", "mixed"):
            row[name]["vs_unfused"] = row["unfused"]["us"] / row[name]["us"]
        dec[f"T{Td}"] = row
    del copies
    res["decode"] = dec

    # --- split-K task graph (Figure 3), A fp32 [8192 x 16384] ---
    A = torch.empty(8192, 16384, device=dev).uniform_(-1, 1)
    C = torch.empty(8192, device=dev)
    sk = {}
    for name, sched in (("static", 0), ("dynamic", 1)):
        sec = time_gpu(lambda: B.etc_splitk_rowsum(A, 4, C, sched=sched), 20, 3, world)
        gbs = (A.numel() * 4 + C.numel() * 4) / sec / 1e9
        sk[name] = {"us": sec * 1e6, "gbs": gbs, "hbm_frac": gbs / hbm}
    res["splitk_8192x16384"] = sk
    del A

    # --- chain: 4 blocks, 200 seeded token counts in [1, 512], one launch each ---
    blocks = inputs.chain_blocks(4)
    bd = dict(norm=[b.norm_w.to(dev) for b in blocks], gate=[b.gate_w.to(dev) for b in blocks],
              gu=[b.w_gate_up.to(dev) for b in blocks], dn=[b.w_down.to(dev) for b in blocks])
    seq = inputs.chain_t_sequence(200, 1, 512, 7)
    xs = torch.randn(512, H, device=dev).to(torch.bfloat16)
    oc = torch.empty(512, H, dtype=torch.float32, device=dev)
    ch = {}
    for name, sched in (("dynamic", 1), ("static", 0)):
        pc = B.etc_moe_plan(H, E, K, I, t_max=512, sched=sched, n_blocks=4)
        for Tc in seq[:3]:
            B.etc_chain_forward(pc, xs, bd["norm"], bd["gate"], None, bd["gu"], bd["dn"], Tc, oc)
        torch.cuda.synchronize()
        l0 = pc and B.etc_plan_stats(pc)["launches"]
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for Tc in seq:
            B.etc_chain_forward(pc, xs, bd["norm"], bd["gate"], None, bd["gu"], bd["dn"], Tc, oc)
        e.record()
        torch.cuda.synchronize()
        assert B.etc_plan_check(pc) == B.ETC_OK, B.etc_last_error()
        tot = s.elapsed_time(e) / 1e3
        ch[name] = {"us_per_call": tot / len(seq) * 1e6, "us_per_layer": tot / len(seq) / 4 * 1e6,
                    "tok_s": sum(seq) / tot, "launches_per_call": (B.etc_plan_stats(pc)["launches"] - l0) / len(seq)}
        pc.close()
    res["chain_4blocks_200calls"] = ch

    # --- dense MLP (the appendix's Table 4, MLP-1 = Qwen3-8B shape), same megakernel ---
    res["dense_mlp"] = run_mlp_rows(dev, tflops_peak, world)
    return res


def run_mlp_rows(dev, tflops_peak, world, names=("MLP-1",)):
    """Dense MLP at Table 4 shapes: static / dynamic one-launch and the two-launch ablation.
    Weights (> L2) are read from HBM on every call."""
    import torch

    from moe_layer_scheduling_gb300 import binding as B
    from moe_layer_scheduling_gb300 import inputs
    rows = {}
    for nm in names:
        S, Hm, Im = inputs.MLP_SHAPES[nm]
        w, x = inputs.mlp_layer(nm)
        wgu, wd, xd = w.w_gate_up.to(dev), w.w_down.to(dev), x.to(dev)
        out = torch.empty(S, Hm, device=dev)
        flops = 6.0 * S * Hm * Im
        row = {"S": S, "H": Hm, "I": Im, "gflop": flops / 1e9}
        for mode, sched, unf, fl in (("static", B.ETC_SCHED_STATIC, False, 0),
                                     ("dynamic", B.ETC_SCHED_DYNAMIC, False, 0),
                                     ("unfused_two_launches", B.ETC_SCHED_STATIC, True, 0),
                                     ("static_single_cta_tiles", B.ETC_SCHED_STATIC, False,
                                      B.ETC_DEBUG_NO_PAIR)):
            pm = B.etc_mlp_plan(Hm, Im, S, sched=sched, debug_flags=fl)
            fn = B.etc_mlp_forward_unfused if unf else B.etc_mlp_forward
            sec = time_gpu(lambda: fn(pm, xd, wgu, wd, S, out), 10, 3, world)
            assert B.etc_plan_check(pm) == B.ETC_OK, B.etc_last_error()
            tf = flops / sec / 1e12
            row[mode] = {"us": sec * 1e6, "tflops": tf, "tensor_frac_of_measured": tf / tflops_peak}
            pm.close()
        rows[nm] = row
        del wgu, wd, xd, out
    return rows


def cpu_baseline(args, wl, budget_s=15.0):
    """The fp64 oracle as it stands, on a bounded token sample of the same workload."""
    import oracle
    w = wl.weights
    n = 8
    t = 0.0
    cores = oracle.get_threads()
    while True:
        xs = wl.x[:n]
        t0 = time.time()
        oracle.moe_layer(xs, w.gate_w, w.w_gate_up, w.w_down, w.top_k, bias=w.router_bias)
        t = time.time() - t0
        if t >= budget_s / 3 or n >= wl.T:
            break
        n = min(wl.T, n * 4)
    return {"value": n / t, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} of the {wl.T} tokens of the same prefill workload "
                      f"(router, top-k, dispatch, {w.top_k} expert FFNs and combine per token), "
                      f"fp64, {t:.1f} s"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: bounded samples of the same workload per step."""
    import oracle
    from moe_layer_scheduling_gb300 import inputs
    if rank != 0:
        return None
    weights = inputs.qwen_weights(0)
    wl = inputs.prefill_skew_layer(args.tokens, weights)
    w = wl.weights
    n = args.ref_tokens
    xs = wl.x[:n]
    for _ in range(args.warmup):
        oracle.moe_layer(xs, w.gate_w, w.w_gate_up, w.w_down, w.top_k, bias=w.router_bias)
    t0 = time.time()
    for _ in range(args.steps):
        oracle.moe_layer(xs, w.gate_w, w.w_gate_up, w.w_down, w.top_k, bias=w.router_bias)
    sec = (time.time() - t0) / args.steps
    v = n / sec
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded workload)",
        "config": {"workload": "qwen3_30b_a3b_moe_prefill_T4096_zipf1.2", "hidden": H,
                   "experts": E, "top_k": K, "inter": I, "tokens_per_step_sample": n},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": oracle.get_threads(),
                         "kind": "oracle", "sample": f"{n} tokens of the T={args.tokens} workload per step"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_single(args):
    """One workload only, no extras (used for profiling captures): decode, splitk or mlp."""
    import torch

    from moe_layer_scheduling_gb300 import binding as B
    from moe_layer_scheduling_gb300 import build as libbuild
    from moe_layer_scheduling_gb300 import inputs
    libbuild.build()
    dev = torch.device("cuda")
    sched = {"static": B.ETC_SCHED_STATIC, "dynamic": B.ETC_SCHED_DYNAMIC,
             "mixed": B.ETC_SCHED_MIXED}[args.sched]
    if args.workload == "mlp":
        if sched == B.ETC_SCHED_MIXED:
            raise SystemExit("the dense MLP takes static or dynamic scheduling")
        S, Hm, Im = inputs.MLP_SHAPES[args.mlp]
        w, x = inputs.mlp_layer(args.mlp)
        wgu, wd, xd = w.w_gate_up.to(dev), w.w_down.to(dev), x.to(dev)
        out = torch.empty(S, Hm, device=dev)
        plan = B.etc_mlp_plan(Hm, Im, S, sched=sched,
                              debug_flags=B.ETC_DEBUG_NO_PAIR if args.tiles == "single" else 0)
        sec = time_gpu(lambda: B.etc_mlp_forward(plan, xd, wgu, wd, S, out), args.steps,
                       args.warmup, 1)
        plan.close()
        return {"workload": f"dense_mlp_{args.mlp}_S{S}_H{Hm}_I{Im}", "sched": args.sched,
                "tiles": args.tiles, "us": sec * 1e6, "tflops": 6.0 * S * Hm * Im / sec / 1e12}
    if args.workload == "splitk":
        if sched == B.ETC_SCHED_MIXED:
            raise SystemExit("split-K takes static or dynamic scheduling")
        A = inputs.splitk_matrix(8192, 16384, 0).to(dev)
        C = torch.empty(8192, device=dev)
        sec = time_gpu(lambda: B.etc_splitk_rowsum(A, 4, C, sched=sched), args.steps, args.warmup, 1)
        return {"workload": "splitk_8192x16384_4tiles", "sched": args.sched, "us": sec * 1e6,
                "gbs": A.numel() * 4 / sec / 1e9}
    w = inputs.qwen_weights(0)
    wl = inputs.decode_layer(args.tokens, w)
    plan = B.etc_moe_plan(H, E, K, I, t_max=args.tokens, sched=sched)
    x, gw, wgu, wd = wl.x.to(dev), w.gate_w.to(dev), w.w_gate_up.to(dev), w.w_down.to(dev)
    out = torch.empty(args.tokens, H, device=dev)
    sec = time_gpu(lambda: B.etc_moe_forward(plan, x, gw, wgu, wd, args.tokens, out), args.steps,
                   args.warmup, 1)
    plan.close()
    return {"workload": wl.name, "sched": args.sched, "us": sec * 1e6,
            "note": "same weights every step (L2-warm for small T)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--ref-tokens", type=int, default=32)
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--workload", default="prefill", choices=["prefill", "decode", "splitk", "mlp"],
                    help="prefill = the benchmark line; decode/splitk/mlp = one workload (profiling)")
    ap.add_argument("--mlp", default="MLP-1", help="Table 4 shape for --workload mlp")
    ap.add_argument("--sched", default=None, choices=["static", "dynamic", "mixed"],
                    help="scheduler of the benchmark line (prefill; default mixed) or of the single "
                         "workload (default static)")
    ap.add_argument("--tiles", default="default", choices=["default", "single"],
                    help="--workload mlp: 'single' runs its wide tiles on single CTAs instead of CTA "
                         "pairs (the form ncu can capture: it cannot launch the pair kernel's "
                         "cooperative cluster launch)")
    ap.add_argument("--clock-window", type=float, default=1.5,
                    help="seconds of load kept up for the clock record (0 for profiler runs)")
    args = ap.parse_args()
    if args.sched is None:
        args.sched = "mixed" if args.workload == "prefill" and args.impl == "ours" else "static"
    rank, world, _ = dist_init()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    elif args.workload != "prefill":
        line = run_single(args)
    else:
        line = run_ours(args, rank, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
