"""GPU parity of the split-K row-sum megakernel against the fp64 oracle.

Tolerance (north-star): relative error <= 1e-5, read as
||C - C_ref||_2 / ||C_ref||_2 <= 1e-5 and, per row, |C_i - C_ref_i| <= 1e-5 * sum_c |A_ic|.
"""
import numpy as np
import pytest
import torch

from moe_layer_scheduling_gb300 import binding as B
from moe_layer_scheduling_gb300 import inputs

pytestmark = pytest.mark.gpu


def _check(C, A, oracle_lib, n_split):
    _, Cref = oracle_lib.splitk(A, n_split)
    C = np.asarray(C, dtype=np.float64)
    assert np.linalg.norm(C - Cref) <= 1e-5 * max(np.linalg.norm(Cref), 1e-30)
    bound = 1e-5 * np.abs(A.astype(np.float64)).sum(axis=1)
    assert np.all(np.abs(C - Cref) <= bound + 1e-30)


def _run(A_np, n_split, sched):
    A = torch.from_numpy(A_np).cuda()
    C = torch.full((A.shape[0],), float("nan"), device="cuda")
    before = B.etc_launch_count()
    B.etc_splitk_rowsum(A, n_split, C, sched=sched)
    torch.cuda.synchronize()
    assert B.etc_splitk_check() == B.ETC_OK, B.etc_last_error()
    assert B.etc_launch_count() - before == 1
    return C.cpu().numpy()


@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC])
@pytest.mark.parametrize("n_rows,n_cols,n_split", [
    (37, 64, 4), (1, 16, 4), (5, 4, 1), (300, 4096, 4), (9, 256, 64), (1000, 12, 3), (8, 65536, 4),
])
def test_splitk_small_and_ragged(oracle_lib, sched, n_rows, n_cols, n_split):
    A = inputs.splitk_matrix(n_rows, n_cols, seed=n_rows + n_cols).numpy()
    C = _run(A, n_split, sched)
    _check(C, A, oracle_lib, n_split)


@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC])
def test_splitk_full_size(oracle_lib, sched):
    # Figure 3's task graph at the benchmarked size: A fp32 [8192 x 16384], 4 column tiles.
    A = inputs.splitk_matrix(8192, 16384, seed=0).numpy()
    C = _run(A, 4, sched)
    _check(C, A, oracle_lib, 4)


def test_splitk_repeated_calls_rearm_the_events(oracle_lib):
    # Counters are re-armed by each final sum: many calls in a row stay correct.
    A = inputs.splitk_matrix(513, 1024, seed=3).numpy()
    for sched in (0, 1, 0, 1, 1, 0):
        C = _run(A, 4, sched)
        _check(C, A, oracle_lib, 4)


def test_splitk_closed_form_on_gpu():
    n = 16384
    A = np.ones((64, n), dtype=np.float32)
    C = _run(A, 4, B.ETC_SCHED_STATIC)
    assert np.all(C == n)
    A = np.tile(np.arange(1024, dtype=np.float32), (8, 1))
    C = _run(A, 4, B.ETC_SCHED_DYNAMIC)
    assert np.all(C == 1024 * 1023 / 2)


@pytest.mark.parametrize("seed", range(24))
def test_splitk_random_shape(oracle_lib, seed):
    """Seeded row counts, split counts and tile widths (n_cols = n_split * tile, tile a
    multiple of 4 up to 16384) under both schedules, against the oracle."""
    rng = np.random.default_rng(6000 + seed)
    n_split = int(rng.choice([1, 2, 3, 4, 5, 8, 16, 64]))
    tile = 4 * int(rng.integers(1, 4097 if n_split <= 4 else 257))
    n_rows = int(rng.choice([int(rng.integers(1, 40)), int(rng.integers(40, 3000))]))
    while n_rows * n_split * tile > 2e7:  # keep the fp64 oracle quick
        n_rows = max(1, n_rows // 2)
    sched = B.ETC_SCHED_DYNAMIC if rng.integers(0, 2) else B.ETC_SCHED_STATIC
    A = inputs.splitk_matrix(n_rows, n_split * tile, seed=6100 + seed).numpy()
    C = _run(A, n_split, sched)
    _check(C, A, oracle_lib, n_split)
