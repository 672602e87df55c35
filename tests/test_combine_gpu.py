"""The ordered combine (etc_moe_opts.combine = ETC_COMBINE_ORDERED).

Down tiles store each expert row y; a finaliser per token block forms
out[t] = sum_{j=0..k-1} w[t,j] * y[pos[t,j]] in j order.  The result must match
the oracle like the fused combine does, and it must be the same bit for bit
from run to run and for every scheduler and launch form, since no step of it
depends on the order in which tiles finish.
"""
import numpy as np
import pytest
import torch

from _moe_check import compare_layer, dispatch_properties, run_layer, to_dev
from moe_layer_scheduling_gb300 import binding as B
from moe_layer_scheduling_gb300 import inputs

pytestmark = pytest.mark.gpu

ORD = B.ETC_COMBINE_ORDERED
SCHEDS = [(B.ETC_SCHED_STATIC, False), (B.ETC_SCHED_DYNAMIC, False), (B.ETC_SCHED_MIXED, False),
          (B.ETC_SCHED_STATIC, True)]


def _plan(w, T, sched, dw, **kw):
    return B.etc_moe_plan(w.hidden, w.n_experts, w.top_k, w.inter, t_max=T, sched=sched,
                          router_bias=dw["bias"], combine=ORD, **kw)


@pytest.mark.parametrize("case", ["tiny", "decode8", "decode64", "wide1100", "pair1100"])
def test_ordered_combine_parity_and_bitwise_reproducible(oracle_lib, case):
    if case == "tiny":
        wl = inputs.tiny_layer(0)
        w, x, extra = wl.weights, wl.x, 0
    elif case.startswith("decode"):
        w = inputs.qwen_weights(0)
        T = int(case[6:])
        x, extra = inputs.tokens(T, inputs.QWEN_H, 1000 + T), 0
    else:
        w = inputs.moe_weights(512, 16, 4, 256, seed=5)
        w.router_bias = inputs.zipf_bias(16, 1.2, 5)
        x = inputs.tokens(1100, 512, 55)
        extra = B.ETC_DEBUG_PAIR_MOE if case == "pair1100" else 0
    T = x.shape[0]
    dw = to_dev(w)
    ref, L, ids, _ = oracle_lib.moe_layer(x, w.gate_w, w.w_gate_up, w.w_down, w.top_k,
                                          bias=w.router_bias, want_routing=True)
    outs = []
    for sched, unfused in SCHEDS:
        plan = _plan(w, T, sched, dw, debug_flags=extra)
        for _ in range(2):
            out, routing, _ = run_layer(w, x, sched, unfused, plan=plan, dw=dw)
            outs.append(out)
        compare_layer(out, routing, ref, L, ids, w.top_k)
        dispatch_properties(routing, w.n_experts)
        plan.close()
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_ordered_combine_bf16_is_the_rounded_fp32_result(oracle_lib):
    w = inputs.qwen_weights(0)
    x = inputs.tokens(300, inputs.QWEN_H, 4300)
    dw = to_dev(w)
    p32 = _plan(w, 300, B.ETC_SCHED_STATIC, dw)
    p16 = _plan(w, 300, B.ETC_SCHED_DYNAMIC, dw, out_dtype=B.ETC_OUT_BF16)
    a, routing, _ = run_layer(w, x, B.ETC_SCHED_STATIC, plan=p32, dw=dw)
    h, _, _ = run_layer(w, x, B.ETC_SCHED_DYNAMIC, plan=p16, dw=dw)
    p32.close()
    p16.close()
    rounded = torch.from_numpy(a).to(torch.bfloat16).float().numpy()
    assert np.array_equal(h, rounded)
    ref, L, ids, _ = oracle_lib.moe_layer(x, w.gate_w, w.w_gate_up, w.w_down, 8, want_routing=True)
    compare_layer(h, routing, ref, L, ids, 8, out_bf16=True)


@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC])
def test_ordered_combine_chain(oracle_lib, sched):
    # Two chain blocks: the first block's finaliser writes the fp32 residual
    # stream (input + ordered sum) that the second block normalises.
    blocks = inputs.chain_blocks(2)
    bd = dict(norm=[b.norm_w.cuda() for b in blocks], gate=[b.gate_w.cuda() for b in blocks],
              gu=[b.w_gate_up.cuda() for b in blocks], dn=[b.w_down.cuda() for b in blocks])
    x = inputs.tokens(45, 2048, 7345)
    res = []
    for _ in range(2):
        plan = B.etc_chain_plan(2, 2048, 128, 8, 768, t_max=64, sched=sched, combine=ORD)
        out = torch.full((45, 2048), float("nan"), device="cuda")
        B.etc_chain_forward(plan, x.cuda(), bd["norm"], bd["gate"], None, bd["gu"], bd["dn"], 45, out)
        torch.cuda.synchronize()
        assert B.etc_plan_check(plan) == B.ETC_OK, B.etc_last_error()
        plan.close()
        res.append(out.cpu().numpy())
    assert np.array_equal(res[0], res[1])
    ref = oracle_lib.chain(x, blocks, eps=1e-6)
    rms = np.sqrt(np.mean(ref * ref))
    assert np.max(np.abs(res[0] - ref)) <= 2e-2 * rms
