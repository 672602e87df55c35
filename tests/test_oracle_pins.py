"""Pins for the fp64 oracle: closed forms, brute force, invariants and the
pages' structural split-K example.  CPU only.

Each pin is chosen so that a plausible slip in the oracle (a dropped bias, a
wrong tie-break, gate/up swapped, a transposed weight, an unstable permutation,
a dropped column tile, a missing residual) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax

from moe_layer_scheduling_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f64(t):
    return t.float().double().numpy()


# ---------------------------------------------------------------------------
# Independent brute-force formulation (dense over all experts, numpy matmuls,
# full softmax then renormalise, selection by a Python sort).
# ---------------------------------------------------------------------------

def brute_moe(x, gate_w, w_gate_up, w_down, k, bias=None):
    X = _f64(x) if isinstance(x, torch.Tensor) else x
    Wg = _f64(gate_w)
    logits = X @ Wg
    if bias is not None:
        logits = logits + bias.double().numpy()[None, :]
    T, E = logits.shape
    I = w_gate_up.shape[1] // 2
    out = np.zeros((T, X.shape[1]))
    probs = softmax(logits, axis=1)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))[:k]
        p = probs[t, order]
        p = p / p.sum()
        for wj, e in zip(p, order):
            Wgu = _f64(w_gate_up[e])
            Wd = _f64(w_down[e])
            gu = Wgu @ X[t]
            g, u = gu[:I], gu[I:]
            a = g * (1.0 / (1.0 + np.exp(-g))) * u
            out[t] += wj * (Wd @ a)
    return out, logits


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# ---------------------------------------------------------------------------
# Router
# ---------------------------------------------------------------------------

def test_router_logits_match_matmul(oracle_lib):
    w = inputs.moe_weights(64, 16, 4, 32, seed=3)
    x = inputs.tokens(5, 64, seed=4)
    bias = torch.linspace(-1, 1, 16, dtype=torch.float32)
    L = oracle_lib.router_logits(x, w.gate_w, bias)
    ref = _f64(x) @ _f64(w.gate_w) + bias.double().numpy()
    assert _rel(L, ref) < 1e-13
    L0 = oracle_lib.router_logits(x, w.gate_w)
    assert _rel(L0, _f64(x) @ _f64(w.gate_w)) < 1e-13
    # orientation: Wg is [H, E]; a one-hot token picks row h of Wg
    xh = torch.zeros(1, 64, dtype=torch.bfloat16)
    xh[0, 7] = 1.0
    assert np.array_equal(oracle_lib.router_logits(xh, w.gate_w)[0], _f64(w.gate_w)[7])


# ---------------------------------------------------------------------------
# Routing: top-k, ties, softmax-over-top-k
# ---------------------------------------------------------------------------

def test_route_ties_go_to_lower_id(oracle_lib):
    L = np.array([[1.0, 3.0, 3.0, 2.0, 3.0],
                  [0.0, 0.0, 0.0, 0.0, 0.0],
                  [-1.0, -0.0, 0.0, -2.0, 5.0]])
    ids, w = oracle_lib.route(L, 2)
    assert ids.tolist() == [[1, 2], [0, 1], [4, 1]]
    assert np.allclose(w[0], [0.5, 0.5]) and np.allclose(w[1], [0.5, 0.5])
    ids3, _ = oracle_lib.route(L, 3)
    assert ids3.tolist() == [[1, 2, 4], [0, 1, 2], [4, 1, 2]]
    ids32, _ = oracle_lib.route_f32(L.astype(np.float32), 3)
    assert np.array_equal(ids32, ids3)


def test_route_k_equals_E_is_full_softmax(oracle_lib):
    rng = np.random.default_rng(1)
    L = rng.standard_normal((7, 12))
    ids, w = oracle_lib.route(L, 12)
    full = softmax(L, axis=1)
    for t in range(7):
        assert sorted(ids[t].tolist()) == list(range(12))
        assert np.allclose(w[t], full[t, ids[t]], rtol=1e-14, atol=0)
        assert abs(w[t].sum() - 1.0) < 1e-14
        assert np.all(np.diff(L[t, ids[t]]) <= 0)  # descending order


def test_route_k1_weight_is_one_and_renormalised_softmax(oracle_lib):
    rng = np.random.default_rng(2)
    L = rng.standard_normal((9, 16)) * 3
    ids1, w1 = oracle_lib.route(L, 1)
    assert np.array_equal(ids1[:, 0], np.argmax(L, axis=1))
    assert np.all(w1 == 1.0)
    ids, w = oracle_lib.route(L, 4)
    p = softmax(L, axis=1)
    for t in range(9):
        ref = p[t, ids[t]] / p[t, ids[t]].sum()
        assert np.allclose(w[t], ref, rtol=1e-13, atol=0)
        # the selected logits dominate every unselected one
        sel = set(ids[t].tolist())
        assert min(L[t, list(sel)]) >= max(L[t, [e for e in range(16) if e not in sel]])


# ---------------------------------------------------------------------------
# Dispatch: counts / exp_indptr / stable permutation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k,seed", [(1, 8, 2, 0), (37, 16, 4, 1), (200, 128, 8, 2)])
def test_dispatch_invariants_and_stable_sort(oracle_lib, T, E, k, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, indptr, pos, row_token = oracle_lib.dispatch(ids, E)
    assert counts.sum() == T * k
    assert indptr[0] == 0 and indptr[-1] == T * k
    assert np.all(np.diff(indptr) == counts)
    assert np.array_equal(np.sort(pos.ravel()), np.arange(T * k))  # bijection
    # brute force: stable argsort of the flat slot list by expert id
    flat = ids.ravel()
    order = np.argsort(flat, kind="stable")
    ref_pos = np.empty(T * k, dtype=np.int64)
    ref_pos[order] = np.arange(T * k)
    assert np.array_equal(pos.ravel(), ref_pos)
    for e in range(E):
        rows = np.arange(indptr[e], indptr[e + 1])
        toks = row_token[rows]
        assert np.all(np.diff(toks) > 0)  # ascending tokens within the expert
        assert set(toks.tolist()) == {t for t in range(T) if e in ids[t]}


def test_dispatch_all_tokens_on_one_expert(oracle_lib):
    T, E, k = 10, 4, 1
    ids = np.full((T, k), 2, dtype=np.int32)
    counts, indptr, pos, row_token = oracle_lib.dispatch(ids, E)
    assert counts.tolist() == [0, 0, 10, 0]
    assert indptr.tolist() == [0, 0, 0, 10, 10]
    assert pos[:, 0].tolist() == list(range(10))
    assert row_token.tolist() == list(range(10))


# ---------------------------------------------------------------------------
# Expert FFN: hand-computed closed forms
# ---------------------------------------------------------------------------

def test_expert_ffn_hand_values(oracle_lib):
    # H=2, I=1: gate row [1, 0], up row [0, 2], down [[3], [-1]]
    x = torch.tensor([1.0, 0.5], dtype=torch.bfloat16)
    wgu = torch.tensor([[1.0, 0.0], [0.0, 2.0]], dtype=torch.bfloat16)
    wd = torch.tensor([[3.0], [-1.0]], dtype=torch.bfloat16)
    y = oracle_lib.expert_ffn(x, wgu, wd)
    g, u = 1.0, 1.0
    a = g / (1 + math.exp(-g)) * u
    assert np.allclose(y, [3 * a, -a], rtol=1e-15, atol=0)
    # gate and up are not interchangeable: swapping the halves changes the result
    y2 = oracle_lib.expert_ffn(torch.tensor([2.0, 1.0], dtype=torch.bfloat16), wgu, wd)
    g, u = 2.0, 2.0
    assert np.allclose(y2, [3 * g / (1 + math.exp(-g)) * u, -g / (1 + math.exp(-g)) * u])
    x3 = torch.tensor([-1.0, 1.0], dtype=torch.bfloat16)  # g=-1, u=2
    a3 = -1.0 / (1 + math.exp(1.0)) * 2.0
    assert np.allclose(oracle_lib.expert_ffn(x3, wgu, wd), [3 * a3, -a3], rtol=1e-15)
    # silu(0) = 0 kills the row whatever the up projection
    x0 = torch.tensor([0.0, 1.0], dtype=torch.bfloat16)
    assert np.all(oracle_lib.expert_ffn(x0, wgu, wd) == 0.0)


def test_expert_ffn_matches_matmul(oracle_lib):
    w = inputs.moe_weights(48, 3, 1, 40, seed=9)
    x = inputs.tokens(1, 48, seed=10)[0]
    y = oracle_lib.expert_ffn(x, w.w_gate_up[1], w.w_down[1])
    gu = _f64(w.w_gate_up[1]) @ _f64(x)
    g, u = gu[:40], gu[40:]
    ref = _f64(w.w_down[1]) @ (g / (1 + np.exp(-g)) * u)
    assert _rel(y, ref) < 1e-13


# ---------------------------------------------------------------------------
# Dense MLP: the same FFN on every row with one weight set
# ---------------------------------------------------------------------------

def test_mlp_hand_values(oracle_lib):
    # H=2, I=1: gate row [1, 0], up row [0, 1], down [[1], [2]]
    wgu = torch.tensor([[1.0, 0.0], [0.0, 1.0]], dtype=torch.bfloat16)
    wd = torch.tensor([[1.0], [2.0]], dtype=torch.bfloat16)
    x = torch.tensor([[2.0, 3.0], [0.0, 5.0], [-1.0, 1.0]], dtype=torch.bfloat16)
    y = oracle_lib.mlp(x, wgu, wd)
    a0 = 2.0 / (1 + math.exp(-2.0)) * 3.0
    a2 = -1.0 / (1 + math.exp(1.0)) * 1.0
    assert np.allclose(y, [[a0, 2 * a0], [0.0, 0.0], [a2, 2 * a2]], rtol=1e-15, atol=0)


def test_mlp_matches_matmul(oracle_lib):
    rng = np.random.default_rng(5)
    T, H, I = 7, 64, 48
    x = torch.from_numpy(rng.standard_normal((T, H), dtype=np.float32)).to(torch.bfloat16)
    w = inputs.mlp_weights(H, I, seed=6)
    y = oracle_lib.mlp(x, w.w_gate_up, w.w_down)
    gu = _f64(x) @ _f64(w.w_gate_up).T
    g, u = gu[:, :I], gu[:, I:]
    ref = (g / (1 + np.exp(-g)) * u) @ _f64(w.w_down).T
    assert y.shape == (T, H)
    assert _rel(y, ref) < 1e-13


def test_mlp_row_subset_is_those_rows(oracle_lib):
    w = inputs.mlp_weights(32, 64, seed=7)
    x = inputs.tokens(6, 32, seed=8)
    full = oracle_lib.mlp(x, w.w_gate_up, w.w_down)
    rows = [4, 0, 5, 4]
    sub = oracle_lib.mlp(x, w.w_gate_up, w.w_down, rows=rows)
    assert np.array_equal(sub, full[rows])
    # rows are independent: permuting the input permutes the output
    perm = [3, 1, 5, 0, 2, 4]
    assert np.array_equal(oracle_lib.mlp(x[perm], w.w_gate_up, w.w_down), full[perm])


def test_mlp_is_a_one_expert_layer(oracle_lib):
    # one expert, top-1: the routing weight is exactly 1 and the layer is the MLP
    w = inputs.mlp_weights(48, 40, seed=9)
    x = inputs.tokens(5, 48, seed=10)
    gate_w = torch.zeros(48, 1, dtype=torch.bfloat16)
    moe = oracle_lib.moe_layer(x, gate_w, w.w_gate_up[None], w.w_down[None], 1)
    assert np.array_equal(oracle_lib.mlp(x, w.w_gate_up, w.w_down), moe)


# ---------------------------------------------------------------------------
# Whole layer
# ---------------------------------------------------------------------------

def test_tiny_layer_matches_brute_force(oracle_lib):
    wl = inputs.tiny_layer(0)
    w = wl.weights
    out, logits, ids, wts = oracle_lib.moe_layer(wl.x, w.gate_w, w.w_gate_up, w.w_down, w.top_k,
                                                  want_routing=True)
    ref, ref_logits = brute_moe(wl.x, w.gate_w, w.w_gate_up, w.w_down, w.top_k)
    assert _rel(logits, ref_logits) < 1e-13
    assert _rel(out, ref) < 1e-12
    assert np.allclose(wts.sum(axis=1), 1.0, atol=1e-15)


@pytest.mark.parametrize("T,seed,with_bias", [(1, 5, False), (13, 6, True), (33, 7, True)])
def test_random_layers_match_brute_force(oracle_lib, T, seed, with_bias):
    w = inputs.moe_weights(64, 16, 4, 32, seed=seed)
    x = inputs.tokens(T, 64, seed=seed + 100)
    bias = inputs.zipf_bias(16, 1.2, seed) if with_bias else None
    out = oracle_lib.moe_layer(x, w.gate_w, w.w_gate_up, w.w_down, 4, bias=bias)
    ref, _ = brute_moe(x, w.gate_w, w.w_gate_up, w.w_down, 4, bias=bias)
    assert _rel(out, ref) < 1e-12


def test_identical_experts_reduce_to_one_ffn(oracle_lib):
    # Closed form independent of routing: weights sum to 1, so the layer equals
    # the shared expert's FFN on every token.
    w = inputs.moe_weights(64, 8, 3, 32, seed=11)
    wgu = w.w_gate_up[:1].expand(8, -1, -1).contiguous()
    wd = w.w_down[:1].expand(8, -1, -1).contiguous()
    x = inputs.tokens(6, 64, seed=12)
    out = oracle_lib.moe_layer(x, w.gate_w, wgu, wd, 3)
    for t in range(6):
        y = oracle_lib.expert_ffn(x[t], wgu[0], wd[0])
        assert _rel(out[t], y) < 1e-13


def test_bias_steers_routing(oracle_lib):
    w = inputs.moe_weights(32, 8, 2, 16, seed=13)
    x = inputs.tokens(4, 32, seed=14)
    bias = torch.full((8,), -100.0)
    bias[5] = 100.0
    bias[2] = 50.0
    _, _, ids, wts = oracle_lib.moe_layer(x, w.gate_w, w.w_gate_up, w.w_down, 2, bias=bias,
                                         want_routing=True)
    assert np.all(ids[:, 0] == 5) and np.all(ids[:, 1] == 2)
    assert np.all(wts[:, 0] > 0.999)


def test_zero_down_projection_gives_zero(oracle_lib):
    w = inputs.moe_weights(32, 4, 2, 16, seed=15)
    x = inputs.tokens(3, 32, seed=16)
    out = oracle_lib.moe_layer(x, w.gate_w, w.w_gate_up, torch.zeros_like(w.w_down), 2)
    assert np.all(out == 0.0)


# ---------------------------------------------------------------------------
# Chain
# ---------------------------------------------------------------------------

def _small_chain(n_blocks, H=64, E=8, k=2, I=32):
    blocks = []
    for b in range(n_blocks):
        w = inputs.moe_weights(H, E, k, I, 100 + b)
        w.norm_w = inputs.tokens(1, H, 200 + b)[0].abs() + 0.5
        w.norm_w = w.norm_w.to(torch.bfloat16)
        blocks.append(w)
    return blocks


def test_chain_matches_blockwise_brute_force(oracle_lib):
    blocks = _small_chain(3)
    x = inputs.tokens(5, 64, 300)
    out, ids, _ = oracle_lib.chain(x, blocks, eps=1e-6, want_routing=True)
    cur = _f64(x)
    for b in blocks:
        rms = np.sqrt(np.mean(cur * cur, axis=1, keepdims=True) + 1e-6)
        normed = cur / rms * _f64(b.norm_w)[None, :]
        delta, _ = brute_moe(normed, b.gate_w, b.w_gate_up, b.w_down, b.top_k)
        cur = cur + delta
    assert _rel(out, cur) < 1e-12


def test_chain_given_its_own_routing_is_the_plain_chain(oracle_lib):
    # Routing given as exactly what the chain selects itself changes nothing.
    blocks = _small_chain(3)
    x = inputs.tokens(6, 64, 303)
    out, ids, logits = oracle_lib.chain(x, blocks, want_routing=True)
    out2, ids2, logits2 = oracle_lib.chain(x, blocks, want_routing=True, ids_in=ids)
    assert np.array_equal(out, out2) and np.array_equal(ids, ids2) and np.array_equal(logits, logits2)


def test_chain_given_routing_matches_brute_force(oracle_lib):
    # Any given routing: each block uses the given experts, weighted by the
    # softmax of its own logits over them (renormalised full softmax).
    blocks = _small_chain(3)
    T, E, k = 5, 8, 2
    x = inputs.tokens(T, 64, 304)
    given = np.zeros((3, T, k), dtype=np.int32)
    for b in range(3):
        for t in range(T):
            given[b, t] = [(t + 3 * b) % E, (t + 3 * b + 5) % E]
    out, ids, _ = oracle_lib.chain(x, blocks, want_routing=True, ids_in=given)
    assert np.array_equal(ids, given)
    cur = _f64(x)
    for b, blk in enumerate(blocks):
        rms = np.sqrt(np.mean(cur * cur, axis=1, keepdims=True) + 1e-6)
        X = cur / rms * _f64(blk.norm_w)[None, :]
        L = X @ _f64(blk.gate_w)
        probs = softmax(L, axis=1)
        I = blk.w_gate_up.shape[1] // 2
        delta = np.zeros_like(X)
        for t in range(T):
            sel = list(given[b, t])
            p = probs[t, sel] / probs[t, sel].sum()
            for wj, e in zip(p, sel):
                gu = _f64(blk.w_gate_up[e]) @ X[t]
                g, u = gu[:I], gu[I:]
                delta[t] += wj * (_f64(blk.w_down[e]) @ (g / (1.0 + np.exp(-g)) * u))
        cur = cur + delta
    assert _rel(out, cur) < 1e-12


def test_chain_zero_experts_is_identity(oracle_lib):
    blocks = _small_chain(4)
    for b in blocks:
        b.w_down = torch.zeros_like(b.w_down)
    x = inputs.tokens(7, 64, 301)
    out = oracle_lib.chain(x, blocks)
    assert np.array_equal(out, _f64(x))


def test_chain_rmsnorm_constant_rows(oracle_lib):
    # For a constant row c*1 with unit gain, RMSNorm gives sign(c)/sqrt(1+eps/c^2);
    # one block with identical experts therefore adds FFN of that vector.
    H = 64
    blocks = _small_chain(1, H=H)
    b = blocks[0]
    b.norm_w = torch.ones(H, dtype=torch.bfloat16)
    b.w_gate_up = b.w_gate_up[:1].expand(8, -1, -1).contiguous()
    b.w_down = b.w_down[:1].expand(8, -1, -1).contiguous()
    x = torch.full((2, H), 4.0, dtype=torch.bfloat16)
    x[1] = -0.5
    out = oracle_lib.chain(x, blocks, eps=1e-6)
    for t, c in enumerate([4.0, -0.5]):
        v = np.full(H, np.sign(c) / math.sqrt(1 + 1e-6 / c ** 2))
        gu = _f64(b.w_gate_up[0]) @ v
        g, u = gu[:32], gu[32:]
        ref = c + _f64(b.w_down[0]) @ (g / (1 + np.exp(-g)) * u)
        assert _rel(out[t], ref) < 1e-12


# ---------------------------------------------------------------------------
# Split-K row sum and its event graph
# ---------------------------------------------------------------------------

def test_splitk_closed_forms(oracle_lib):
    n = 1024
    B, C = oracle_lib.splitk(np.ones((3, n), dtype=np.float32), 4)
    assert np.all(C == n) and np.all(B == n / 4)
    A = np.tile(np.arange(n, dtype=np.float32), (2, 1))
    B, C = oracle_lib.splitk(A, 4)
    assert np.all(C == n * (n - 1) / 2)
    q = n // 4
    for j in range(4):
        assert B[0, j] == sum(range(j * q, (j + 1) * q))


def test_splitk_random_vs_fsum(oracle_lib):
    A = inputs.splitk_matrix(16, 4096, seed=0).numpy()
    B, C = oracle_lib.splitk(A, 4)
    for i in range(16):
        exact = math.fsum(A[i].astype(np.float64))
        assert abs(C[i] - exact) <= 1e-12 * np.abs(A[i]).sum()
        for j in range(4):
            ex = math.fsum(A[i, j * 1024:(j + 1) * 1024].astype(np.float64))
            assert abs(B[i, j] - ex) <= 1e-12 * np.abs(A[i]).sum()


def _golden(name):
    d = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            d.setdefault(key, []).append(vals)
    return d


def test_event_graph_from_the_pages(oracle_lib):
    g = _golden("splitk_event_graph.txt")
    wait = int(g["wait_count"][0][0])
    n_split = int(g["n_split"][0][0])
    out_map, in_map = g["out_edges"][0][0], g["in_edges"][0][0]
    rng = np.random.default_rng(0)
    part = rng.standard_normal((50, n_split))
    Cs = []
    for seed in range(5):
        C, notes, early, order = oracle_lib.event_sim(part, wait, out_map, in_map, seed)
        assert np.all(notes == int(g["notifies_per_event"][0][0]))
        assert early == 0
        # final(i) runs only after its n_split partials, and exactly once
        seen = np.zeros(50, dtype=int)
        finals = 0
        for task in order:
            if task >= 0:
                seen[task // n_split] += 1
            else:
                i = -task - 1
                assert seen[i] == n_split
                finals += 1
        assert finals == 50
        Cs.append(C)
    for C in Cs[1:]:
        assert np.array_equal(C, Cs[0])  # order-independent result
    ref = np.array([sum(part[i, j] for j in range(n_split)) for i in range(50)])
    assert np.array_equal(Cs[0], ref)


def test_event_graph_detects_wrong_wait_count(oracle_lib):
    part = np.ones((8, 4))
    _, _, early, _ = oracle_lib.event_sim(part, 3, "ij->i", "i->i", 1)
    assert early > 0                   # a final would start before its 4th partial
    C, _, _, order = oracle_lib.event_sim(part, 5, "ij->i", "i->i", 1)
    assert np.all(np.isnan(C))         # wait_count 5 never reaches zero: no final runs
    assert np.all(order >= 0)


def test_event_graph_instantiation_shapes(oracle_lib):
    # Figure 4: the same template instantiated at batch 1 and batch 2.
    g = _golden("splitk_event_graph.txt")
    for b, shape in g["instantiate"]:
        b = int(b)
        rows, cols = (int(v) for v in shape.split("x"))
        part = np.ones((rows, cols))
        C, notes, early, order = oracle_lib.event_sim(part, cols, "ij->i", "i->i", 3)
        assert rows == b and len(notes) == b and np.all(notes == cols) and early == 0
        assert len(order) == b * cols + b
    trace = [int(v) for v in g["two_producer_trace"][0]]
    C, notes, early, order = oracle_lib.event_sim(np.ones((1, 2)), trace[0], "ij->i", "i->i", 0)
    assert notes[0] == trace[0] and early == 0 and C[0] == 2.0
