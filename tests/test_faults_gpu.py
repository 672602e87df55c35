"""Failure detection on the GPU without a GPU fault.

A wait is made to run out on purpose (an expert or row whose event needs one
notify more than it will ever get); the kernel's bounded wait records a
timeout, every CTA exits, the host reads the status, and the context stays
usable for the next call.
"""
import numpy as np
import pytest
import torch

from _moe_check import compare_layer, run_layer, to_dev
from moe_layer_scheduling_gb300 import binding as B
from moe_layer_scheduling_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC, B.ETC_SCHED_MIXED])
def test_moe_wait_times_out_and_recovers(oracle_lib, sched):
    wl = inputs.tiny_layer(0)
    w = wl.weights
    dw = to_dev(w)
    ref, L, ids, _ = oracle_lib.moe_layer(wl.x, w.gate_w, w.w_gate_up, w.w_down, w.top_k,
                                          want_routing=True)
    victim = int(ids[0, 0])  # an expert that does receive tokens
    plan = B.etc_moe_plan(w.hidden, w.n_experts, w.top_k, w.inter, t_max=4, sched=sched,
                          wait_timeout_ns=100_000_000, debug_flags=B.ETC_DEBUG_FAULT_EXTRA_WAIT,
                          debug_arg=victim)
    x = wl.x.cuda()
    out = torch.zeros(4, w.hidden, dtype=torch.float32, device="cuda")
    B.etc_moe_forward(plan, x, dw["gate_w"], dw["w_gate_up"], dw["w_down"], 4, out)
    torch.cuda.synchronize()  # the kernel ends: no hang
    assert B.etc_plan_check(plan) == B.ETC_ERR_TIMEOUT
    assert "timed out" in B.etc_last_error()
    with pytest.raises(B.EtcError) as ei:  # sticky until reset
        B.etc_moe_forward(plan, x, dw["gate_w"], dw["w_gate_up"], dw["w_down"], 4, out)
    assert ei.value.code == B.ETC_ERR_STATE
    B.etc_plan_reset(plan)
    assert B.etc_plan_check(plan) == B.ETC_OK
    plan.close()
    # the context is healthy: a clean plan computes the right answer
    out, routing, plan2 = run_layer(w, wl.x, sched, dw=dw)
    compare_layer(out, routing, ref, L, ids, w.top_k)
    plan2.close()


def test_splitk_wait_times_out_and_recovers(oracle_lib):
    A = inputs.splitk_matrix(64, 1024, seed=1)
    Ad = A.cuda()
    C = torch.zeros(64, device="cuda")
    rc = B.etc_splitk_rowsum_ex(Ad, 4, C, sched=B.ETC_SCHED_STATIC, wait_timeout_ns=100_000_000,
                                debug_flags=B.ETC_DEBUG_FAULT_EXTRA_WAIT, debug_arg=17)
    assert rc == B.ETC_OK
    torch.cuda.synchronize()
    assert B.etc_splitk_check() == B.ETC_ERR_TIMEOUT
    assert B.etc_splitk_check() == B.ETC_OK  # cleared, counters re-armed
    B.etc_splitk_rowsum(Ad, 4, C)
    torch.cuda.synchronize()
    assert B.etc_splitk_check() == B.ETC_OK
    _, Cref = oracle_lib.splitk(A.numpy(), 4)
    assert np.linalg.norm(C.cpu().numpy() - Cref) <= 1e-5 * np.linalg.norm(Cref)


@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC], ids=["static", "dynamic"])
def test_dense_mlp_wait_times_out_and_recovers(oracle_lib, sched):
    """Dense MLP: chunk 1's down tiles wait for one gate/up tile more than it
    has (static: their counter wait; dynamic: they are never pushed, so a
    queue pop waits).  The bounded waits end the kernel, the status reports
    the timeout, the plan refuses calls until reset, and the context still
    computes a correct MLP."""
    H, I, T = 256, 256, 300  # 3 chunks, the last one ragged
    w = inputs.mlp_weights(H, I, seed=21)
    x = inputs.tokens(T, H, seed=22)
    xd, wgu, wd = x.cuda(), w.w_gate_up.cuda(), w.w_down.cuda()
    plan = B.etc_mlp_plan(H, I, t_max=T, sched=sched, wait_timeout_ns=100_000_000,
                          debug_flags=B.ETC_DEBUG_FAULT_EXTRA_WAIT, debug_arg=1)
    out = torch.zeros(T, H, device="cuda")
    B.etc_mlp_forward(plan, xd, wgu, wd, T, out)
    torch.cuda.synchronize()  # the kernel ends: no hang
    assert B.etc_plan_check(plan) == B.ETC_ERR_TIMEOUT
    assert "timed out" in B.etc_last_error()
    with pytest.raises(B.EtcError) as ei:  # sticky until reset
        B.etc_mlp_forward(plan, xd, wgu, wd, T, out)
    assert ei.value.code == B.ETC_ERR_STATE
    B.etc_plan_reset(plan)
    assert B.etc_plan_check(plan) == B.ETC_OK
    plan.close()
    good = B.etc_mlp_plan(H, I, t_max=T, sched=sched)
    out = torch.full((T, H), float("nan"), device="cuda")
    B.etc_mlp_forward(good, xd, wgu, wd, T, out)
    torch.cuda.synchronize()
    assert B.etc_plan_check(good) == B.ETC_OK
    ref = oracle_lib.mlp(x, w.w_gate_up, w.w_down)
    got = out.double().cpu().numpy()
    assert np.max(np.abs(got - ref)) <= 2e-2 * np.sqrt(np.mean(ref * ref))
    good.close()
