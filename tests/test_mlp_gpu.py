"""GPU parity of the dense MLP megakernel (static, dynamic, unfused) against the fp64 oracle.

The dense MLP shapes are those of the appendix's Table 4 (paper summary page of
"Event Tensor: A Unified Abstraction for Compiling Dynamic Megakernel").  The
output tolerance is the layer tolerance: max |gpu - oracle| <= 2e-2 * RMS(oracle).
"""
import numpy as np
import pytest
import torch

from moe_layer_scheduling_gb300 import binding as B
from moe_layer_scheduling_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 2e-2
MODES = [(B.ETC_SCHED_STATIC, False), (B.ETC_SCHED_DYNAMIC, False), (B.ETC_SCHED_STATIC, True)]
MODE_IDS = ["static", "dynamic", "unfused"]


def _run(plan, xd, wgu, wd, T, unfused, out_dtype=torch.float32):
    out = torch.full((max(T, 1), xd.shape[1]), float("nan"), device="cuda", dtype=out_dtype)
    fn = B.etc_mlp_forward_unfused if unfused else B.etc_mlp_forward
    fn(plan, xd, wgu, wd, T, out)
    torch.cuda.synchronize()
    assert B.etc_plan_check(plan) == B.ETC_OK
    return out[:T].double().cpu().numpy()


def _close(out, ref):
    rms = np.sqrt(np.mean(ref * ref))
    err = np.max(np.abs(out - ref))
    assert np.isfinite(out).all()
    assert err <= TOL * rms, (err, rms)
    return err / rms


@pytest.mark.parametrize("sched,unfused", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("H,I,T", [
    (512, 1024, 300),   # wide tiles: 3 chunks, the last one ragged (44 rows)
    (512, 1024, 64),    # the smallest call on wide tiles: one partial chunk
    (512, 1024, 5),     # narrow tiles
    (384, 320, 200),    # narrow tiles forced by the shape (H % 256, I % 128 != 0)
    (256, 128, 1),      # one token, one down tile per chunk row
])
def test_mlp_parity(oracle_lib, sched, unfused, H, I, T):
    w = inputs.mlp_weights(H, I, seed=H + I)
    x = inputs.tokens(T, H, seed=T)
    plan = B.etc_mlp_plan(H, I, t_max=T, sched=sched)
    before = B.etc_launch_count()
    out = _run(plan, x.cuda(), w.w_gate_up.cuda(), w.w_down.cuda(), T, unfused)
    assert B.etc_launch_count() - before == (2 if unfused else 1)
    _close(out, oracle_lib.mlp(x, w.w_gate_up, w.w_down))
    plan.close()


@pytest.mark.parametrize("sched,unfused", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("H,I,T", [(512, 1024, 300), (512, 1024, 64)])
def test_mlp_parity_single_cta_wide_tiles(oracle_lib, sched, unfused, H, I, T):
    # Wide calls with CTA pairs disabled (256-weight-row tiles on one SM).
    w = inputs.mlp_weights(H, I, seed=H + I)
    x = inputs.tokens(T, H, seed=T)
    plan = B.etc_mlp_plan(H, I, t_max=T, sched=sched, debug_flags=B.ETC_DEBUG_NO_PAIR)
    out = _run(plan, x.cuda(), w.w_gate_up.cuda(), w.w_down.cuda(), T, unfused)
    _close(out, oracle_lib.mlp(x, w.w_gate_up, w.w_down))
    plan.close()


@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC], ids=["static", "dynamic"])
def test_mlp_bf16_output_and_determinism(oracle_lib, sched):
    H, I, T = 512, 768, 257
    w = inputs.mlp_weights(H, I, seed=3)
    x = inputs.tokens(T, H, seed=4)
    xd, wgu, wd = x.cuda(), w.w_gate_up.cuda(), w.w_down.cuda()
    ref = oracle_lib.mlp(x, w.w_gate_up, w.w_down)
    p32 = B.etc_mlp_plan(H, I, t_max=T, sched=sched)
    p16 = B.etc_mlp_plan(H, I, t_max=T, sched=sched, out_dtype=B.ETC_OUT_BF16)
    a = _run(p32, xd, wgu, wd, T, False)
    b = _run(p32, xd, wgu, wd, T, False)
    # each output element is written once, by the tile that owns it
    assert np.array_equal(a, b)
    h = _run(p16, xd, wgu, wd, T, False, out_dtype=torch.bfloat16)
    _close(h, ref)
    # the bf16 output is the fp32 one rounded to nearest even
    assert np.array_equal(h, torch.from_numpy(a).float().to(torch.bfloat16).double().numpy())
    p32.close()
    p16.close()


@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC], ids=["static", "dynamic"])
def test_mlp_changing_T_on_one_plan(oracle_lib, sched):
    # The chunk counters are re-armed by each call's last down tiles: a run of
    # calls with different T (and narrow/wide tiles) on one plan stays correct.
    H, I = 512, 1024
    w = inputs.mlp_weights(H, I, seed=5)
    x = inputs.tokens(700, H, seed=6)
    xd, wgu, wd = x.cuda(), w.w_gate_up.cuda(), w.w_down.cuda()
    ref = oracle_lib.mlp(x, w.w_gate_up, w.w_down)
    plan = B.etc_mlp_plan(H, I, t_max=700, sched=sched)
    for T in (700, 129, 7, 128, 700, 63, 300):
        out = _run(plan, xd, wgu, wd, T, False)
        _close(out, ref[:T])
    # T = 0 launches nothing
    before = B.etc_launch_count()
    B.etc_mlp_forward(plan, xd, wgu, wd, 0, torch.empty(1, H, device="cuda"))
    assert B.etc_launch_count() == before
    plan.close()


def test_mlp_and_moe_plans_are_not_interchangeable():
    mlp = B.etc_mlp_plan(256, 128, t_max=8)
    moe = B.etc_moe_plan(256, 8, 2, 128, 8)
    x = torch.zeros(8, 256, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(8, 256, device="cuda")
    w = torch.zeros(8 * 256 * 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.EtcError) as e:
        B.etc_moe_forward(mlp, x, w, w, w, 8, out)
    assert e.value.code == B.ETC_ERR_INVALID
    with pytest.raises(B.EtcError) as e:
        B.etc_mlp_forward(moe, x, w, w, 8, out)
    assert e.value.code == B.ETC_ERR_INVALID
    with pytest.raises(B.EtcError):
        B.etc_moe_debug_routing(mlp, 0, counts=torch.empty(8, dtype=torch.int32, device="cuda"))
    with pytest.raises(B.EtcError):  # no permuted rows in a dense plan
        B.etc_moe_debug_buffer(mlp, 0, torch.empty(16, dtype=torch.bfloat16, device="cuda"))
    mlp.close()
    moe.close()


@pytest.fixture(scope="module")
def mlp1(oracle_lib):
    S, H, I = inputs.MLP_SHAPES["MLP-1"]
    w, x = inputs.mlp_layer("MLP-1")
    # Rows checked against the oracle: the first and the last 256-row chunk
    # whole (a pair tile's chunk; two 128-row chunks of single-CTA tiles),
    # and 256 more sampled from the rest.
    rng = np.random.default_rng(17)
    rows = np.unique(np.concatenate([np.arange(0, 256), np.arange(S - 256, S),
                                     rng.choice(np.arange(256, S - 256), 256, replace=False)]))
    ref = oracle_lib.mlp(x, w.w_gate_up, w.w_down, rows=rows)
    return S, H, I, w, x, w.w_gate_up.cuda(), w.w_down.cuda(), x.cuda(), rows, ref


@pytest.mark.parametrize("sched,unfused", MODES, ids=MODE_IDS)
def test_mlp1_full_size(oracle_lib, mlp1, sched, unfused):
    # Table 4's MLP-1 (Qwen3-8B: S=8192, H=4096, I=12288) in the launch
    # configuration the benchmark times; the oracle computes 768 of the rows.
    S, H, I, w, x, wgu, wd, xd, rows, ref = mlp1
    plan = B.etc_mlp_plan(H, I, t_max=S, sched=sched)
    out = _run(plan, xd, wgu, wd, S, unfused)
    assert len(rows) == 768
    _close(out[rows], ref)
    assert np.isfinite(out).all()
    plan.close()


def _draw_mlp(seed):
    """A seeded dense MLP shape within the plan's limits (H multiple of 128, I of 64)."""
    rng = np.random.default_rng(5000 + seed)
    H = int(rng.choice([128, 256, 384, 512, 768, 1024]))
    I = int(rng.choice([64, 128, 192, 256, 320, 512, 1024]))
    T = int(rng.choice([int(rng.integers(1, 33)), int(rng.integers(33, 300)), int(rng.integers(300, 900))]))
    sched = B.ETC_SCHED_DYNAMIC if rng.integers(0, 2) else B.ETC_SCHED_STATIC
    flags = B.ETC_DEBUG_NO_PAIR if rng.integers(0, 2) else 0
    return H, I, T, sched, flags


@pytest.mark.parametrize("seed", range(24))
def test_mlp_random_shape(oracle_lib, seed):
    """Seeded (H, I, T), schedule and tile form (CTA pairs or single-CTA) against the oracle:
    ragged chunks, narrow and wide tiles, one and many chunks."""
    H, I, T, sched, flags = _draw_mlp(seed)
    w = inputs.mlp_weights(H, I, seed=700 + seed)
    x = inputs.tokens(T, H, seed=800 + seed)
    plan = B.etc_mlp_plan(H, I, t_max=T, sched=sched, debug_flags=flags)
    out = _run(plan, x.cuda(), w.w_gate_up.cuda(), w.w_down.cuda(), T, False)
    _close(out, oracle_lib.mlp(x, w.w_gate_up, w.w_down))
    plan.close()
