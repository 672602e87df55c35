"""Shared GPU-vs-oracle checks for the MoE layer tests.

Tolerances (north-star): logits |dL| <= 1e-4 * (|L_ref| + RMS(L_ref));
layer output max |gpu - oracle| <= 2e-2 * RMS(oracle); routing (ids, counts,
exp_indptr, permutation) bit-exact given identical fp32 logits, ties to the
lower expert id.
"""
import numpy as np
import torch

from moe_layer_scheduling_gb300 import binding as B

LOGIT_RTOL = 1e-4
OUT_TOL = 2e-2


def to_dev(w, dev="cuda"):
    return dict(x=None, gate_w=w.gate_w.to(dev), w_gate_up=w.w_gate_up.to(dev),
                w_down=w.w_down.to(dev),
                bias=None if w.router_bias is None else w.router_bias.to(dev))


def run_layer(w, x_cpu, sched, unfused=False, t_max=None, debug_flags=0, plan=None, dw=None,
              out_dtype=B.ETC_OUT_F32):
    """Runs one layer through the C ABI; returns (out, routing dict, plan)."""
    T = x_cpu.shape[0]
    dw = dw or to_dev(w)
    if plan is None:
        plan = B.etc_moe_plan(w.hidden, w.n_experts, w.top_k, w.inter, t_max=t_max or T,
                              sched=sched, router_bias=dw["bias"], debug_flags=debug_flags,
                              out_dtype=out_dtype)
    x = x_cpu.cuda()
    out = torch.full((T, w.hidden), float("nan"), dtype=plan.out_dtype, device="cuda")
    before = B.etc_launch_count()
    fn = B.etc_moe_forward_unfused if unfused else B.etc_moe_forward
    fn(plan, x, dw["gate_w"], dw["w_gate_up"], dw["w_down"], T, out)
    torch.cuda.synchronize()
    assert B.etc_plan_check(plan) == B.ETC_OK, B.etc_last_error()
    # unfused: one launch per stage that has work; the top-k stage is empty
    # when the top-k runs inside the router tiles, the combine finaliser when
    # the fp32 output is complete after the down tiles
    n = B.etc_launch_count() - before
    assert (5 <= n <= 7) if unfused else n == 1
    return out.float().cpu().numpy(), read_routing(plan, T, w), plan


def read_routing(plan, T, w, block=0):
    E, k = w.n_experts, w.top_k
    r = dict(logits=torch.empty(T, E, device="cuda"),
             ids=torch.empty(T, k, dtype=torch.int32, device="cuda"),
             w=torch.empty(T, k, device="cuda"),
             counts=torch.empty(E, dtype=torch.int32, device="cuda"),
             exp_indptr=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
             pos=torch.empty(T, k, dtype=torch.int32, device="cuda"))
    B.etc_moe_debug_routing(plan, block, r["logits"], r["ids"], r["w"], r["counts"],
                            r["exp_indptr"], r["pos"])
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in r.items()}


def topk_is_valid(logits, ids):
    """Property: ids[t] are the k largest of logits[t], ordered by (value desc, id asc)."""
    T, E = logits.shape
    k = ids.shape[1]
    bad = []
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))[:k]
        if not np.array_equal(order, ids[t]):
            bad.append(t)
    return bad


def near_tie(L_ref_row, k, ids_a, ids_b, gap):
    """True if the two selections differ only among experts whose oracle logits
    sit within `gap` of the k-th largest one."""
    srt = np.sort(L_ref_row)[::-1]
    kth = srt[k - 1]
    diff = set(ids_a.tolist()) ^ set(ids_b.tolist())
    return all(abs(L_ref_row[e] - kth) <= gap for e in diff)


def compare_layer(out, routing, ref_out, ref_logits, ref_ids, k, max_flip_frac=0.01,
                  out_bf16=False):
    """Returns (max_err, tol, n_flipped) after asserting every spec bar.

    With a bf16 output the bound also allows the rounding of the output itself:
    the stated bar is for the fp32 result, and round-to-nearest-even to bf16
    (8 significant bits) moves a value by at most half a unit in the last place
    of the result, 2^(floor(log2|y|) - 8) for the rounded value y, i.e. between
    2^-9 |y| and 2^-8 |y| (elementwise).
    """
    L, Lref = routing["logits"].astype(np.float64), ref_logits
    rms_L = np.sqrt(np.mean(Lref * Lref))
    assert np.all(np.abs(L - Lref) <= LOGIT_RTOL * (np.abs(Lref) + rms_L)), \
        f"logits off: max {np.max(np.abs(L - Lref))}"
    assert topk_is_valid(routing["logits"], routing["ids"]) == []
    flips = [t for t in range(out.shape[0]) if not np.array_equal(routing["ids"][t], ref_ids[t])]
    gap = 4 * LOGIT_RTOL * (np.abs(Lref).max() + rms_L)
    for t in flips:
        assert near_tie(Lref[t], k, routing["ids"][t], ref_ids[t], gap), f"token {t} routed apart"
    assert len(flips) <= max(1, int(max_flip_frac * out.shape[0]))
    keep = np.ones(out.shape[0], dtype=bool)
    keep[flips] = False
    rms = float(np.sqrt(np.mean(ref_out * ref_out)))
    tol = OUT_TOL * rms
    assert np.all(np.isfinite(out))
    if keep.any():
        d = np.abs(out[keep] - ref_out[keep])
        if out_bf16:
            d = d - bf16_half_ulp(out[keep])
        err = float(np.max(d))
    else:
        err = 0.0
    assert err <= tol, f"max |gpu - oracle| = {err:.4e} > {tol:.4e}"
    # weights: softmax over the selected logits, fp32 on the GPU
    return err, tol, len(flips)


def bf16_half_ulp(y):
    """Half a unit in the last place of bf16 values y (0 where y == 0)."""
    a = np.abs(np.asarray(y, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def dispatch_properties(routing, E):
    """counts / exp_indptr / pos are the stable counting sort of the GPU's own ids
    (checked as properties here, never by feeding GPU output to the oracle)."""
    ids = routing["ids"]
    T, k = ids.shape
    counts = np.bincount(ids.ravel(), minlength=E)
    assert np.array_equal(routing["counts"], counts)
    assert np.array_equal(routing["exp_indptr"], np.concatenate([[0], np.cumsum(counts)]))
    order = np.argsort(ids.ravel(), kind="stable")
    pos = np.empty(T * k, dtype=np.int64)
    pos[order] = np.arange(T * k)
    assert np.array_equal(routing["pos"].ravel(), pos)


def check_dispatch_vs_oracle(routing, oracle_lib, ref_ids, E):
    """With no routing flips the dispatch must equal the oracle's, bit for bit."""
    counts, indptr, pos, _ = oracle_lib.dispatch(ref_ids, E)
    assert np.array_equal(routing["counts"], counts)
    assert np.array_equal(routing["exp_indptr"], indptr)
    assert np.array_equal(routing["pos"], pos)
