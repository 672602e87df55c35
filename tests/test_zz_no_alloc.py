"""The split-K entry point that allocates nothing.

It serves callers that cannot call cudaMalloc when they need the operation
(allocator or memory-pool callbacks that must not re-enter the allocator,
runtimes that reserve all device memory up front).  Its result must match the
oracle's fp64 row sums within the split-K tolerance, and the allocating entry
point's result, on two calls in a row (the second reuses the fixed scratch the
first left behind); each call must leave an OK status that etc_splitk_check
reads without allocating, must not change the device's free memory, and sizes
beyond its fixed scratch must be refused.  This file is collected last on
purpose.
"""
import numpy as np
import pytest
import torch

from moe_layer_scheduling_gb300 import binding as B
from moe_layer_scheduling_gb300 import inputs

pytestmark = pytest.mark.gpu

REL_TOL = 1e-5  # the split-K tolerance used by the other split-K tests


def _close(C, Cref, A):
    C, Cref = C.double(), Cref.double()
    assert torch.linalg.norm(C - Cref) <= REL_TOL * torch.linalg.norm(Cref)
    bound = REL_TOL * A.double().abs().sum(dim=1)
    assert torch.all((C - Cref).abs() <= bound)


@pytest.mark.parametrize("sched", [B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC])
@pytest.mark.parametrize("n_rows,n_cols,n_split", [(8192, 16384, 4), (777, 1024, 4), (5, 64, 1)])
def test_noalloc_matches_the_oracle_and_the_allocating_entry_point(oracle_lib, sched, n_rows, n_cols,
                                                                   n_split):
    A_cpu = inputs.splitk_matrix(n_rows, n_cols, seed=11)
    A = A_cpu.cuda()
    _, C_oracle = oracle_lib.splitk(A_cpu.numpy(), n_split)
    C_oracle = torch.from_numpy(np.asarray(C_oracle, dtype=np.float64))
    ref = torch.empty(n_rows, device="cuda")
    B.etc_splitk_rowsum(A, n_split, ref, sched=sched)
    for _ in range(2):
        C = torch.full((n_rows,), float("nan"), device="cuda")
        B.etc_splitk_rowsum_noalloc(A, n_split, C, sched=sched)
        torch.cuda.synchronize()
        assert B.etc_splitk_check() == B.ETC_OK, B.etc_last_error()
        assert torch.isfinite(C).all()
        _close(C.cpu(), C_oracle, A_cpu)
        _close(C.cpu(), ref.cpu().double(), A_cpu)


def test_noalloc_call_allocates_no_device_memory():
    A = inputs.splitk_matrix(4096, 8192, seed=12).cuda()
    C = torch.empty(4096, device="cuda")
    B.etc_splitk_rowsum_noalloc(A, 4, C)  # the first call on a device does its set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    torch_bytes0 = torch.cuda.memory_allocated()
    for sched in (B.ETC_SCHED_STATIC, B.ETC_SCHED_DYNAMIC):
        B.etc_splitk_rowsum_noalloc(A, 4, C, sched=sched)
        torch.cuda.synchronize()
        assert B.etc_splitk_check() == B.ETC_OK, B.etc_last_error()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == torch_bytes0


def test_noalloc_refuses_sizes_beyond_its_scratch():
    A = torch.zeros(65537, 4, device="cuda")
    C = torch.empty(65537, device="cuda")
    with pytest.raises(B.EtcError) as e:
        B.etc_splitk_rowsum_noalloc(A, 1, C)
    assert e.value.code == B.ETC_ERR_INVALID and "scratch" in str(e.value)
    A = torch.zeros(8192, 64 * 4, device="cuda")
    C = torch.empty(8192, device="cuda")
    with pytest.raises(B.EtcError):
        B.etc_splitk_rowsum_noalloc(A, 64, C)  # 8192 * 64 partial sums > 262144
