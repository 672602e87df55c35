"""GPU parity of the MoE megakernel (static, dynamic, unfused) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from _moe_check import (check_dispatch_vs_oracle, compare_layer, dispatch_properties,
                        read_routing, run_layer, to_dev)
from moe_layer_scheduling_gb300 import binding as B
from moe_layer_scheduling_gb300 import inputs

pytestmark = pytest.mark.gpu

MODES = [(B.ETC_SCHED_STATIC, False), (B.ETC_SCHED_DYNAMIC, False), (B.ETC_SCHED_MIXED, False),
         (B.ETC_SCHED_STATIC, True)]
MODE_IDS = ["static", "dynamic", "mixed", "unfused"]


@pytest.fixture(scope="module")
def qwen():
    return inputs.qwen_weights(0)


@pytest.fixture(scope="module")
def qwen_dev(qwen):
    return to_dev(qwen)


def _full_check(oracle_lib, w, x, sched, unfused, dw=None, t_max=None, debug_flags=0):
    out, routing, plan = run_layer(w, x, sched, unfused, dw=dw, t_max=t_max, debug_flags=debug_flags)
    ref, ref_logits, ref_ids, ref_w = oracle_lib.moe_layer(x, w.gate_w, w.w_gate_up, w.w_down,
                                                           w.top_k, bias=w.router_bias,
                                                           want_routing=True)
    err, tol, nflip = compare_layer(out, routing, ref, ref_logits, ref_ids, w.top_k)
    dispatch_properties(routing, w.n_experts)
    if nflip == 0:
        check_dispatch_vs_oracle(routing, oracle_lib, ref_ids, w.n_experts)
        assert np.allclose(routing["w"], ref_w, atol=2e-6, rtol=0)
    plan.close()
    return err, tol


@pytest.mark.parametrize("sched,unfused", MODES, ids=MODE_IDS)
def test_tiny_layer(oracle_lib, sched, unfused):
    wl = inputs.tiny_layer(0)
    _full_check(oracle_lib, wl.weights, wl.x, sched, unfused)


@pytest.mark.parametrize("sched,unfused", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_decode_layer(oracle_lib, qwen, qwen_dev, sched, unfused, T):
    x = inputs.tokens(T, inputs.QWEN_H, 1000 + T)
    _full_check(oracle_lib, qwen, x, sched, unfused, dw=qwen_dev)


@pytest.mark.parametrize("sched,unfused", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("T,seed", [(33, 1), (200, 2), (517, 3), (6000, 4)])
def test_ragged_token_counts(oracle_lib, sched, unfused, T, seed):
    # Several tiles and a ragged tail on every axis, a skewing bias, odd T;
    # T=6000 has more token blocks (188) than SMs, so CTAs run several
    # routing and permute tasks in one launch.
    w = inputs.moe_weights(256, 16, 4, 192, seed=seed)
    w.router_bias = inputs.zipf_bias(16, 1.2, seed)
    x = inputs.tokens(T, 256, seed + 50)
    _full_check(oracle_lib, w, x, sched, unfused)


SHAPE_EDGES = [
    # (H, E, k, I, T): E not a power of two and k = 1;
    (256, 24, 1, 64, 45),
    # k = E = 16 (every token to every expert, the largest k);
    (256, 16, 16, 128, 40),
    # the largest hidden size: one 24 KB token row fills the permute's row
    # slots, the router's H is split 32 ways;
    (12288, 8, 2, 64, 33),
    # T = t_max with a ragged block, H a multiple of 128 but not a power of two.
    (384, 128, 8, 64, 77),
]


@pytest.mark.parametrize("sched,unfused", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape", SHAPE_EDGES, ids=lambda s: "H%d-E%d-k%d-I%d-T%d" % s)
def test_shape_edges(oracle_lib, sched, unfused, shape):
    H, E, k, I, T = shape
    w = inputs.moe_weights(H, E, k, I, seed=H + E + k)
    x = inputs.tokens(T, H, T + 7)
    _full_check(oracle_lib, w, x, sched, unfused, t_max=T)


@pytest.mark.parametrize("sched,unfused", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("T,seed", [(300, 4), (1100, 5)])
def test_wide_tiles(oracle_lib, sched, unfused, T, seed):
    # Enough rows per expert (T*k >= 64*E) for the 256-weight-row tiles:
    # H=512, E=16, k=4, I=256, a skewing bias, ragged token and chunk tails.
    w = inputs.moe_weights(512, 16, 4, 256, seed=seed)
    w.router_bias = inputs.zipf_bias(16, 1.2, seed)
    x = inputs.tokens(T, 512, seed + 50)
    _full_check(oracle_lib, w, x, sched, unfused)


@pytest.mark.parametrize("sched,unfused", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("T,seed", [(300, 4), (1100, 5)])
def test_wide_tiles_on_cta_pairs(oracle_lib, sched, unfused, T, seed):
    # The same wide calls on CTA pairs (one cta_group::2 MMA per tile over two
    # SMs, chunks of up to 256 rows), ragged chunk and token tails.
    w = inputs.moe_weights(512, 16, 4, 256, seed=seed)
    w.router_bias = inputs.zipf_bias(16, 1.2, seed)
    x = inputs.tokens(T, 512, seed + 50)
    _full_check(oracle_lib, w, x, sched, unfused, debug_flags=B.ETC_DEBUG_PAIR_MOE)


@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC, B.ETC_SCHED_MIXED])
def test_qwen_prefill_on_cta_pairs(oracle_lib, qwen, qwen_dev, sched):
    # Qwen shape at T=1100 on CTA pairs, every token checked against the oracle.
    x = inputs.tokens(1100, inputs.QWEN_H, 1100)
    _full_check(oracle_lib, qwen, x, sched, False, dw=qwen_dev, debug_flags=B.ETC_DEBUG_PAIR_MOE)


@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC, B.ETC_SCHED_MIXED])
def test_qwen_wide_tiles_full_parity(oracle_lib, qwen, qwen_dev, sched):
    # Qwen shape at T=1100: wide tiles, every token checked against the oracle.
    x = inputs.tokens(1100, inputs.QWEN_H, 1100)
    _full_check(oracle_lib, qwen, x, sched, False, dw=qwen_dev)


@pytest.fixture(scope="module")
def prefill(oracle_lib, qwen):
    """The benchmark's prefill workload and the oracle's result for all its tokens."""
    wl = inputs.prefill_skew_layer(4096, qwen)
    w = wl.weights
    ref, Lref, ids_ref, _ = oracle_lib.moe_layer(wl.x, w.gate_w, w.w_gate_up, w.w_down, w.top_k,
                                                 bias=w.router_bias, want_routing=True)
    return wl, ref, Lref, ids_ref


@pytest.mark.parametrize("sched,unfused", MODES, ids=MODE_IDS)
def test_prefill_skew_full_size(oracle_lib, qwen_dev, prefill, sched, unfused):
    # T=4096 with Zipf(1.2)-biased routing, in the launch configuration the
    # benchmark times: empty experts and experts with thousands of rows.
    # Routing, dispatch and the output of every one of the 4096 tokens are
    # checked against the oracle.
    wl, ref, Lref, ids_ref = prefill
    w = wl.weights
    dw = dict(qwen_dev)
    dw["bias"] = w.router_bias.cuda()
    out, routing, plan = run_layer(w, wl.x, sched, unfused, dw=dw)
    plan.close()
    counts = np.bincount(ids_ref.ravel(), minlength=w.n_experts)
    assert (counts == 0).any() and counts.max() > 200  # the skew the workload asks for
    dispatch_properties(routing, w.n_experts)
    err, tol, nflip = compare_layer(out, routing, ref, Lref, ids_ref, w.top_k)
    if nflip == 0:
        check_dispatch_vs_oracle(routing, oracle_lib, ids_ref, w.n_experts)


@pytest.mark.parametrize("T", [64, 427])
def test_bf16_output(oracle_lib, qwen, qwen_dev, T):
    # Optional bf16 output: the stated bar plus the rounding of the output itself.
    x = inputs.tokens(T, inputs.QWEN_H, 4000 + T)
    out, routing, plan = run_layer(qwen, x, B.ETC_SCHED_DYNAMIC, dw=qwen_dev,
                                   out_dtype=B.ETC_OUT_BF16)
    plan.close()
    ref, L, ids, _ = oracle_lib.moe_layer(x, qwen.gate_w, qwen.w_gate_up, qwen.w_down, 8,
                                          want_routing=True)
    compare_layer(out, routing, ref, L, ids, 8, out_bf16=True)


def test_run_to_run_difference_is_bounded(qwen, qwen_dev):
    # The fused combine adds each token's k weighted expert rows with fp32
    # reductions in L2, in whatever order the down tiles finish: two runs of the
    # same call may differ, but only by the rounding of a reordered k-term fp32
    # sum, at most 2k * 2^-24 * sum_j |w_j y_j| per element.  sum_j |w_j y_j|
    # is taken as 8x the output's largest magnitude (room for cancellation);
    # a lost or doubled contribution would be ~|w_j y_j|, far above this.
    T, k = 517, qwen.top_k
    x = inputs.tokens(T, inputs.QWEN_H, 5170)
    plan = B.etc_moe_plan(2048, 128, k, 768, t_max=T, sched=B.ETC_SCHED_DYNAMIC)
    outs = [run_layer(qwen, x, B.ETC_SCHED_DYNAMIC, plan=plan, dw=qwen_dev)[0] for _ in range(3)]
    plan.close()
    scale = 8 * np.max(np.abs(outs[0])) * 2 * k * 2.0 ** -24
    for o in outs[1:]:
        assert np.max(np.abs(o.astype(np.float64) - outs[0])) <= scale


@pytest.mark.parametrize("T,E,k", [(300, 64, 6), (1, 128, 8), (2, 128, 8), (5, 128, 8), (8, 128, 8),
                                   (34, 128, 8), (37, 8, 2), (70, 128, 16), (41, 8, 8)])
def test_route_from_logits_bit_exact(oracle_lib, T, E, k):
    # Identical fp32 logits on both sides, with deliberate exact ties: ids,
    # counts, exp_indptr and the permutation must match bit for bit, and
    # x_perm must hold the routed rows.  Token blocks of 1-2, 3-8 and more
    # tokens take the three top-k methods (rank count, warp, thread groups).
    H = 256
    rng = np.random.default_rng(5 + T)
    L = rng.integers(-8, 8, size=(T, E)).astype(np.float32) * 0.25  # many ties
    if T > 8:
        L[7] = 0.0  # a token whose logits are all equal
        L[8, :] = -0.0
        L[8, 3] = 0.0
    else:
        L[0] = 0.0
    x = inputs.tokens(T, H, 6)
    plan = B.etc_moe_plan(H, E, k, 128, t_max=T)
    B.etc_moe_route_from_logits(plan, torch.from_numpy(L).cuda(), x.cuda(), T)
    torch.cuda.synchronize()
    assert B.etc_plan_check(plan) == B.ETC_OK
    w = type("W", (), dict(n_experts=E, top_k=k))
    r = read_routing(plan, T, w)
    ids_ref, w_ref = oracle_lib.route_f32(L, k)
    assert np.array_equal(r["ids"], ids_ref)
    assert np.array_equal(r["logits"], L)
    check_dispatch_vs_oracle(r, oracle_lib, ids_ref, E)
    assert np.allclose(r["w"], w_ref, atol=1e-6, rtol=0)
    assert r["ids"][7 if T > 8 else 0].tolist() == list(range(k))
    xp = torch.empty(T * k, H, dtype=torch.bfloat16, device="cuda")
    B.etc_moe_debug_buffer(plan, 0, xp)
    torch.cuda.synchronize()
    _, _, _, row_token = oracle_lib.dispatch(ids_ref, E)
    assert torch.equal(xp.cpu(), x[torch.from_numpy(row_token.astype(np.int64))])
    plan.close()


def test_zero_tokens_is_a_noop(qwen, qwen_dev):
    plan = B.etc_moe_plan(2048, 128, 8, 768, t_max=16)
    before = B.etc_launch_count()
    x = torch.empty(0, 2048, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(0, 2048, dtype=torch.bfloat16, device="cuda")
    B.etc_moe_forward(plan, x.data_ptr() or 256, qwen_dev["gate_w"], qwen_dev["w_gate_up"],
                      qwen_dev["w_down"], 0, out.data_ptr() or 256)
    assert B.etc_launch_count() == before
    with pytest.raises(B.EtcError):
        B.etc_moe_forward(plan, torch.empty(17, 2048, dtype=torch.bfloat16, device="cuda"),
                          qwen_dev["gate_w"], qwen_dev["w_gate_up"], qwen_dev["w_down"], 17,
                          torch.empty(17, 2048, dtype=torch.bfloat16, device="cuda"))
    plan.close()


def test_all_tokens_on_one_expert(oracle_lib):
    # A bias that sends every token to experts {5, 2}: one expert gets T rows,
    # the rest none; several 128-row chunks of one expert.
    w = inputs.moe_weights(256, 8, 2, 128, seed=21)
    bias = torch.full((8,), -50.0)
    bias[5], bias[2] = 50.0, 40.0
    w.router_bias = bias
    x = inputs.tokens(300, 256, 22)
    for sched in (B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC):
        _full_check(oracle_lib, w, x, sched, False)


@pytest.mark.parametrize("sched", [B.ETC_SCHED_DYNAMIC, B.ETC_SCHED_MIXED], ids=["dynamic", "mixed"])
def test_heavy_experts(oracle_lib, sched):
    # Experts 5 (all 600 tokens) and 2 (552 of them) reach the heavy threshold
    # (ceil(0.85 T) = 510 rows; queued schedules only): they run over all of
    # x, with weight 0 for the 48 tokens that did not choose expert 2; the
    # other six experts keep their permuted rows.  The result must match the
    # oracle, and the same call with heavy experts switched off up to the
    # rounding of the tiles' fp32 accumulation.
    unfused = False
    w = inputs.moe_weights(256, 8, 2, 256, seed=31)
    bias = torch.zeros(8)
    bias[5], bias[2] = 50.0, 1.0
    w.router_bias = bias
    x = inputs.tokens(600, 256, 32)
    _, _, ref_ids, _ = oracle_lib.moe_layer(x, w.gate_w, w.w_gate_up, w.w_down, 2, bias=bias,
                                            want_routing=True)
    cnt = np.bincount(np.asarray(ref_ids).reshape(-1), minlength=8)
    assert cnt[5] == 600 and 510 <= cnt[2] < 600 and (cnt[[0, 1, 3, 4, 6, 7]] > 0).all()
    _full_check(oracle_lib, w, x, sched, unfused)
    out_h, _, plan = run_layer(w, x, sched, unfused)
    plan.close()
    out_p, _, plan = run_layer(w, x, sched, unfused, debug_flags=B.ETC_DEBUG_NO_HEAVY)
    plan.close()
    # (a tile's MMAs see the token rows in other positions: fp32 accumulation
    # may round differently, far below the bf16 operands' own rounding)
    diff = np.max(np.abs(out_h.astype(np.float64) - out_p))
    assert diff <= 1e-5 * np.max(np.abs(out_p)), diff


@pytest.mark.parametrize("flags", [0, B.ETC_DEBUG_WIDE_SWAP_AB, B.ETC_DEBUG_NO_HEAVY,
                                   B.ETC_DEBUG_WIDE_SWAP_AB | B.ETC_DEBUG_NO_HEAVY],
                         ids=["default", "swap_ab", "no_heavy", "swap_ab_no_heavy"])
@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_MIXED], ids=["static", "mixed"])
def test_wide_tile_forms(oracle_lib, sched, flags):
    # Wide tiles in every form the flags select: full chunks token-major or
    # swap-AB, with and without a heavy expert (expert 3 takes every token),
    # several full 128-row chunks and ragged ones; all against the oracle.
    w = inputs.moe_weights(512, 16, 4, 256, seed=41)
    bias = inputs.zipf_bias(16, 1.2, 41)
    bias[3] = 40.0
    w.router_bias = bias
    x = inputs.tokens(700, 512, 42)
    _full_check(oracle_lib, w, x, sched, False, debug_flags=flags)


@pytest.mark.parametrize("T", [20, 600])
@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_MIXED], ids=["static", "mixed"])
def test_saturated_gate_activations(oracle_lib, sched, T):
    # Gate rows scaled by 100: pre-activations reach past -88 and +88, where
    # SiLU sits on its asymptotes (0 and the identity) and the epilogue's
    # denominator 1 + exp(-g) leaves the normal range of the fast division.
    # T=20 runs the one-block direct tiles, T=600 the wide ones.
    w = inputs.moe_weights(256, 8, 2, 128, seed=51)
    wgu = w.w_gate_up.float()
    wgu[:, :128, :] *= 100.0
    w.w_gate_up = wgu.to(torch.bfloat16)
    x = inputs.tokens(T, 256, 52)
    g = np.einsum("th,eih->tei", x.float().numpy(), w.w_gate_up[:, :128, :].float().numpy())
    assert g.min() < -90.0 and g.max() > 90.0
    _full_check(oracle_lib, w, x, sched, False)


def test_identical_experts_closed_form(oracle_lib):
    # Routing-independent closed form: with every expert equal the layer is one FFN.
    w = inputs.moe_weights(256, 16, 4, 128, seed=23)
    w.w_gate_up = w.w_gate_up[:1].expand(16, -1, -1).contiguous()
    w.w_down = w.w_down[:1].expand(16, -1, -1).contiguous()
    x = inputs.tokens(40, 256, 24)
    out, routing, plan = run_layer(w, x, B.ETC_SCHED_DYNAMIC)
    plan.close()
    ref = np.stack([oracle_lib.expert_ffn(x[t], w.w_gate_up[0], w.w_down[0]) for t in range(40)])
    rms = np.sqrt(np.mean(ref * ref))
    assert np.max(np.abs(out - ref)) <= 2e-2 * rms


def test_dynamic_token_counts_same_plan(oracle_lib, qwen, qwen_dev):
    # One plan, one compiled kernel, T changing on every call: exactly one
    # launch per call and correct results (Figure 4: template instantiated per call).
    plan = B.etc_moe_plan(2048, 128, 8, 768, t_max=512, sched=B.ETC_SCHED_DYNAMIC)
    seq = inputs.chain_t_sequence(24, 1, 512, seed=7)
    launches0 = B.etc_plan_stats(plan)["launches"]
    for i, T in enumerate(seq):
        x = inputs.tokens(T, 2048, 3000 + i)
        out, routing, _ = run_layer(qwen, x, B.ETC_SCHED_DYNAMIC, plan=plan, dw=qwen_dev)
        if i % 6 == 0:
            ref, L, ids, _ = oracle_lib.moe_layer(x, qwen.gate_w, qwen.w_gate_up, qwen.w_down, 8,
                                                  want_routing=True)
            compare_layer(out, routing, ref, L, ids, 8)
        dispatch_properties(routing, 128)
    assert B.etc_plan_stats(plan)["launches"] - launches0 == len(seq)
    plan.close()


def test_poisoned_workspace_gives_same_result(oracle_lib):
    # NaN-filled intermediates before the call: any stale read would show.
    wl = inputs.tiny_layer(0)
    w = wl.weights
    dw = to_dev(w)
    plan = B.etc_moe_plan(w.hidden, w.n_experts, w.top_k, w.inter, t_max=4,
                          debug_flags=B.ETC_DEBUG_POISON)
    out, routing, _ = run_layer(w, wl.x, 0, plan=plan, dw=dw)
    ref, L, ids, _ = oracle_lib.moe_layer(wl.x, w.gate_w, w.w_gate_up, w.w_down, w.top_k,
                                          want_routing=True)
    compare_layer(out, routing, ref, L, ids, w.top_k)
    plan.close()
