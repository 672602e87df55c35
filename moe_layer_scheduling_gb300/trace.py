"""Task-trace summary of one megakernel call (a profiling aid).

Runs one MoE layer with the library's ETC_DEBUG_TRACE flag and prints, per
task type, how many tasks ran, their summed and mean busy time on the worker
warps, and when the stage started and ended relative to the first task;
also the time from the first to the last task and how busy the SMs' workers
were, over the whole call and per 20 us window.

    python -m moe_layer_scheduling_gb300.trace --tokens 4096 --skew --sched dynamic
    python -m moe_layer_scheduling_gb300.trace --mlp MLP-1 --sched static   # dense MLP
"""
from __future__ import annotations

import argparse
import json
from collections import defaultdict


def summarize(recs: list[dict], window_ns: int = 20000) -> dict:
    if not recs:
        return {}
    t0 = min(r["t_dispatch"] or r["t_start"] for r in recs)
    t_end = max(r["t_end"] for r in recs)
    by = defaultdict(list)
    for r in recs:
        by[r["type"]].append(r)
    stages = {}
    for name, rs in by.items():
        busy = [r["t_end"] - r["t_start"] for r in rs]
        wait = [r["t_start"] - r["t_dispatch"] for r in rs if r["t_dispatch"]]
        stages[name] = {
            "tasks": len(rs),
            "busy_us_sum": sum(busy) / 1e3,
            "busy_us_mean": sum(busy) / len(busy) / 1e3,
            "queue_us_mean": (sum(wait) / len(wait) / 1e3) if wait else None,
            "first_start_us": (min(r["t_start"] for r in rs) - t0) / 1e3,
            "last_end_us": (max(r["t_end"] for r in rs) - t0) / 1e3,
        }
    sms = {r["sm"] for r in recs}
    busy_total = sum(r["t_end"] - r["t_start"] for r in recs)
    span = t_end - t0
    # fraction of the SMs' workers inside a task, per window of the call
    win = window_ns if span > window_ns else max(span, 1)
    n_win = max(1, -(-span // win))
    busy_win = [0.0] * n_win
    for r in recs:
        a, b = r["t_start"] - t0, r["t_end"] - t0
        for i in range(max(0, a // win), min(n_win, b // win + 1)):
            lo, hi = i * win, (i + 1) * win
            busy_win[i] += max(0, min(b, hi) - max(a, lo))
    n_sm = max(len(sms), 1)
    return {"span_us": span / 1e3, "sms": len(sms),
            "worker_busy_frac": busy_total / (span * n_sm) if span else None,
            "busy_frac_per_window": {"window_us": win / 1e3,
                                     "values": [round(v / (win * n_sm), 2) for v in busy_win]},
            "stages": stages}


def main():
    import torch

    from . import binding as B
    from . import inputs

    ap = argparse.ArgumentParser()
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--skew", action="store_true", help="Zipf(1.2) router bias (prefill workload)")
    ap.add_argument("--sched", default="dynamic", choices=["static", "dynamic", "mixed"])
    ap.add_argument("--repeat", type=int, default=3, help="calls before the traced one")
    ap.add_argument("--raw", default=None, help="also write the task records (JSON) to this file")
    ap.add_argument("--mlp", default=None, help="trace the dense MLP of this Table 4 shape instead")
    ap.add_argument("--no-pair", action="store_true", help="dense MLP: wide tiles on single CTAs")
    ap.add_argument("--pair", action="store_true", help="MoE layer: wide tiles on CTA pairs")
    args = ap.parse_args()
    extra = (B.ETC_DEBUG_NO_PAIR if args.no_pair else 0) | (B.ETC_DEBUG_PAIR_MOE if args.pair else 0)
    dev = torch.device("cuda")
    sched = {"static": B.ETC_SCHED_STATIC, "dynamic": B.ETC_SCHED_DYNAMIC,
             "mixed": B.ETC_SCHED_MIXED}[args.sched]
    if args.mlp:
        if sched == B.ETC_SCHED_MIXED:
            raise SystemExit("the dense MLP takes static or dynamic scheduling")
        mw, mx = inputs.mlp_layer(args.mlp)
        S, Hm = mx.shape
        plan = B.etc_mlp_plan(Hm, mw.inter, S, sched=sched, debug_flags=B.ETC_DEBUG_TRACE | extra)
        xd, wgu, wd = mx.to(dev), mw.w_gate_up.to(dev), mw.w_down.to(dev)
        out = torch.empty(S, Hm, device=dev)
        for _ in range(args.repeat + 1):
            B.etc_mlp_forward(plan, xd, wgu, wd, S, out)
        name = f"dense_mlp_{args.mlp}_S{S}_H{Hm}_I{mw.inter}"
    else:
        plan, name = None, None
    if plan is not None:
        torch.cuda.synchronize()
        assert B.etc_plan_check(plan) == B.ETC_OK, B.etc_last_error()
        _report(B, plan, name, args)
        return
    w = inputs.qwen_weights(0)
    wl = inputs.prefill_skew_layer(args.tokens, w) if args.skew else inputs.decode_layer(args.tokens, w)
    bias = wl.weights.router_bias.to(dev) if wl.weights.router_bias is not None else None
    plan = B.etc_moe_plan(w.hidden, w.n_experts, w.top_k, w.inter, t_max=args.tokens, sched=sched,
                          router_bias=bias, debug_flags=B.ETC_DEBUG_TRACE | extra)
    x = wl.x.to(dev)
    gw, wgu, wd = w.gate_w.to(dev), w.w_gate_up.to(dev), w.w_down.to(dev)
    out = torch.empty(args.tokens, w.hidden, device=dev)
    for _ in range(args.repeat + 1):
        B.etc_moe_forward(plan, x, gw, wgu, wd, args.tokens, out)
    torch.cuda.synchronize()
    assert B.etc_plan_check(plan) == B.ETC_OK, B.etc_last_error()
    _report(B, plan, wl.name, args)


def _report(B, plan, name, args):
    recs = B.etc_moe_debug_trace(plan, max_records=200000)
    if args.raw:
        with open(args.raw, "w") as f:
            json.dump(recs, f)
    s = summarize(recs)
    s["workload"] = name
    s["sched"] = args.sched
    print(json.dumps(s, indent=1))
    plan.close()


if __name__ == "__main__":
    main()
