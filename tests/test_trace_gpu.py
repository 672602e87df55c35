"""The task trace records every task of a call, MoE layer and dense MLP alike."""
from collections import Counter

import pytest
import torch

from moe_layer_scheduling_gb300 import binding as B
from moe_layer_scheduling_gb300 import inputs
from moe_layer_scheduling_gb300.trace import summarize

pytestmark = pytest.mark.gpu


def _check_records(recs):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for r in recs:
        assert r["t_start"] <= r["t_end"]
        assert 0 <= r["sm"] < sms


@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC], ids=["static", "dynamic"])
def test_trace_of_a_tiny_layer_counts_its_tiles(sched):
    wl = inputs.tiny_layer(0)
    w = wl.weights
    plan = B.etc_moe_plan(w.hidden, w.n_experts, w.top_k, w.inter, t_max=wl.T, sched=sched,
                          debug_flags=B.ETC_DEBUG_TRACE)
    out = torch.empty(wl.T, w.hidden, device="cuda")
    B.etc_moe_forward(plan, wl.x.cuda(), w.gate_w.cuda(), w.w_gate_up.cuda(), w.w_down.cuda(),
                      wl.T, out)
    torch.cuda.synchronize()
    assert B.etc_plan_check(plan) == B.ETC_OK
    counts = torch.empty(w.n_experts, dtype=torch.int32, device="cuda")
    B.etc_moe_debug_routing(plan, 0, counts=counts)
    hit = int((counts.cpu() > 0).sum())  # each hit expert has one chunk (at most T rows)
    recs = B.etc_moe_debug_trace(plan)
    _check_records(recs)
    n = Counter(r["type"] for r in recs)
    # narrow tiles: I/64 gate/up tiles and H/128 down tiles per chunk
    assert n["gate_up"] == hit * (w.inter // 64)
    assert n["down"] == hit * (w.hidden // 128)
    assert n["router"] >= 1 and n["perm"] >= 1
    assert summarize(recs)["stages"]["gate_up"]["tasks"] == n["gate_up"]
    plan.close()


def test_trace_of_a_dense_mlp_counts_its_tiles():
    H, I, T = 256, 512, 300  # wide tiles: 3 chunks x I/128 gate/up tiles, H/256 down tiles
    w = inputs.mlp_weights(H, I, seed=31)
    x = inputs.tokens(T, H, seed=32)
    plan = B.etc_mlp_plan(H, I, t_max=T, debug_flags=B.ETC_DEBUG_TRACE)
    out = torch.empty(T, H, device="cuda")
    B.etc_mlp_forward(plan, x.cuda(), w.w_gate_up.cuda(), w.w_down.cuda(), T, out)
    torch.cuda.synchronize()
    assert B.etc_plan_check(plan) == B.ETC_OK
    recs = B.etc_moe_debug_trace(plan)
    _check_records(recs)
    n = Counter(r["type"] for r in recs)
    assert n == Counter({"gate_up": 3 * (I // 128), "down": 3 * (H // 256)})
    plan.close()
