"""Seeded random layer shapes against the oracle.

Each case draws H, E, k, I, T, the router bias (none, Zipf-skewed, or one
expert that every token chooses) and the schedule from a fixed seed, within
the library's shape limits, and runs the full parity check (logits, routing
properties, output within 2e-2 * RMS).  The draws reach the narrow, thin,
direct and wide tile forms, heavy experts, permute parts and ragged tails
that the hand-picked cases leave out.
"""
import numpy as np
import pytest
import torch

from _moe_check import compare_layer, dispatch_properties, run_layer
from moe_layer_scheduling_gb300 import binding as B
from moe_layer_scheduling_gb300 import inputs

pytestmark = pytest.mark.gpu

SCHEDS = [(B.ETC_SCHED_STATIC, False), (B.ETC_SCHED_DYNAMIC, False), (B.ETC_SCHED_MIXED, False),
          (B.ETC_SCHED_STATIC, True)]


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    H = int(rng.choice([128, 256, 384, 512, 1024]))
    E = int(rng.choice([8, 16, 24, 64, 128]))
    k = int(rng.integers(1, min(E, 16) + 1))
    I = int(rng.choice([64, 128, 192, 256, 384]))
    T = int(rng.choice([int(rng.integers(1, 33)), int(rng.integers(33, 300)),
                        int(rng.integers(300, 1500))]))
    # keep the fp64 oracle within a few seconds
    while T > 1 and T * k * H * I * 3 > 4e9:
        T //= 2
    bias_kind = int(rng.integers(0, 3))
    sched, unfused = SCHEDS[int(rng.integers(0, len(SCHEDS)))]
    return H, E, k, I, T, bias_kind, sched, unfused


@pytest.mark.parametrize("seed", range(48))
def test_random_shape(oracle_lib, seed):
    H, E, k, I, T, bias_kind, sched, unfused = _draw(seed)
    w = inputs.moe_weights(H, E, k, I, seed=500 + seed)
    if bias_kind == 1:
        w.router_bias = inputs.zipf_bias(E, 1.2, seed)
    elif bias_kind == 2:
        bias = torch.zeros(E)
        bias[seed % E] = 40.0  # one expert every token chooses
        w.router_bias = bias
    x = inputs.tokens(T, H, 600 + seed)
    out, routing, plan = run_layer(w, x, sched, unfused)
    plan.close()
    ref, L, ids, _ = oracle_lib.moe_layer(x, w.gate_w, w.w_gate_up, w.w_down, k,
                                          bias=w.router_bias, want_routing=True)
    compare_layer(out, routing, ref, L, ids, k)
    dispatch_properties(routing, E)
