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
    # one token block: the gate/up tiles read x directly, no permute task runs
    assert n["router"] >= 1 and n["perm"] == 0
    assert summarize(recs)["stages"]["gate_up"]["tasks"] == n["gate_up"]
    plan.close()


@pytest.mark.parametrize("pair", [True, False], ids=["pair_tiles", "single_cta_tiles"])
def test_trace_of_a_dense_mlp_counts_its_tiles(pair):
    H, I, T = 256, 512, 300
    w = inputs.mlp_weights(H, I, seed=31)
    x = inputs.tokens(T, H, seed=32)
    plan = B.etc_mlp_plan(H, I, t_max=T, debug_flags=B.ETC_DEBUG_TRACE |
                          (0 if pair else B.ETC_DEBUG_NO_PAIR))
    out = torch.empty(T, H, device="cuda")
    B.etc_mlp_forward(plan, x.cuda(), w.w_gate_up.cuda(), w.w_down.cuda(), T, out)
    torch.cuda.synchronize()
    assert B.etc_plan_check(plan) == B.ETC_OK
    recs = B.etc_moe_debug_trace(plan)
    _check_records(recs)
    n = Counter(r["type"] for r in recs)
    if not pair:
        # wide tiles: 3 chunks of 128 rows x I/128 gate/up tiles, H/256 down tiles
        assert n == Counter({"gate_up": 3 * (I // 128), "down": 3 * (H // 256)})
    else:
        # pair tiles: 2 chunks of 256 rows, the same tile counts per chunk; each
        # tile runs on both CTAs of one pair (SMs 2u and 2u + 1)
        assert n == Counter({"gate_up": 2 * 2 * (I // 128), "down": 2 * 2 * (H // 256)})
        _check_pairs(recs)
    plan.close()


def _check_pairs(recs):
    by_task = {}
    for r in recs:
        by_task.setdefault((r["type"], r["block"], r["a"], r["b"]), []).append(r["sm"])
    for key, sms in by_task.items():
        if key[0] in ("gate_up", "down", "router"):
            assert len(sms) == 2 and sms[0] // 2 == sms[1] // 2 and sms[0] != sms[1], (key, sms)


@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC], ids=["static", "dynamic"])
def test_trace_of_a_pair_tile_layer(sched):
    # Enough rows per expert for wide tiles, run on CTA pairs on request: every
    # router, gate/up and down task appears on the two CTAs of one pair.
    w = inputs.moe_weights(512, 16, 4, 256, seed=5)
    x = inputs.tokens(1100, 512, 55)
    plan = B.etc_moe_plan(512, 16, 4, 256, t_max=1100, sched=sched,
                          debug_flags=B.ETC_DEBUG_TRACE | B.ETC_DEBUG_PAIR_MOE)
    out = torch.empty(1100, 512, device="cuda")
    B.etc_moe_forward(plan, x.cuda(), w.gate_w.cuda(), w.w_gate_up.cuda(), w.w_down.cuda(), 1100, out)
    torch.cuda.synchronize()
    assert B.etc_plan_check(plan) == B.ETC_OK
    counts = torch.empty(16, dtype=torch.int32, device="cuda")
    B.etc_moe_debug_routing(plan, 0, counts=counts)
    chunks = int(((counts.cpu() + 255) // 256).sum())
    recs = B.etc_moe_debug_trace(plan)
    _check_records(recs)
    n = Counter(r["type"] for r in recs)
    assert n["gate_up"] == 2 * chunks * (256 // 128)
    assert n["down"] == 2 * chunks * (512 // 256)
    _check_pairs(recs)
    plan.close()
