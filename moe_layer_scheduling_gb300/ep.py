"""Expert parallelism across GPUs: the host-side plan of the dispatch and combine.

On one GPU the layer's expert tiles wait on per-expert counters whose
wait_count is the number of rows the router gave the expert, and expert e fires
exactly the tiles of its row range [exp_indptr[e], exp_indptr[e+1]) ("Event
Tensor: A Unified Abstraction for Compiling Dynamic Megakernel", podcast
transcript, cues 7 and 9).  Across W ranks the same two mechanisms carry over,
with the experts sharded in contiguous ranges (rank r owns experts
[r*E/W, (r+1)*E/W)) and each rank routing its own tokens:

  1. count exchange: each rank tells every owner how many rows it will send to
     each of the owner's experts;
  2. data-dependent event init on the owner: wait_count[e] = the rows all
     sources send to e;
  3. dispatch: a source writes its rows straight into the owner's receive
     buffer, at the slots the prefix sums below give it (expert-major, then
     source rank, then ascending token), and takes its row count off the
     owner's counter of that expert: the notify that, at zero, fires the
     expert's tiles;
  4. combine: the owner writes each finished expert row back to its source in
     the order it received the rows; the source puts it in the slot (t, j) it
     came from and takes one off its token's counter (k); at zero the token's
     k rows are summed in j order.

This module holds that bookkeeping only (which rows go where, in what order,
and the counter values); it moves no data and does no arithmetic of the layer.
The fused multi-GPU kernel (rows written into peer memory, counters in peer
memory, no multicast) is not built: every box this library is measured on has
one GPU.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def expert_owner(n_experts: int, world: int) -> tuple[np.ndarray, np.ndarray]:
    """(owner rank, index within the owner's shard) of every expert."""
    if world < 1 or n_experts % world:
        raise ValueError(f"{n_experts} experts do not split evenly over {world} ranks")
    per = n_experts // world
    e = np.arange(n_experts)
    return e // per, e % per


@dataclass
class SendPlan:
    """What one source rank sends.  slots[d]: the flat slots t*k + j whose rows
    go to rank d, in send order; counts[d]: rows per local expert of rank d."""
    slots: list[np.ndarray]
    counts: np.ndarray  # [world, experts per rank]


def send_plan(ids: np.ndarray, n_experts: int, world: int) -> SendPlan:
    """Send order of a rank's routed rows: per destination, ascending local
    expert, then ascending token (the stable order of the one-GPU layer)."""
    T, k = ids.shape
    owner, local = expert_owner(n_experts, world)
    per = n_experts // world
    flat = ids.reshape(-1).astype(np.int64)
    slots, counts = [], np.zeros((world, per), dtype=np.int64)
    for d in range(world):
        mine = np.nonzero(owner[flat] == d)[0]          # flat slots, ascending token
        order = np.argsort(local[flat[mine]], kind="stable")
        slots.append(mine[order])
        counts[d] = np.bincount(local[flat[mine]], minlength=per)
    return SendPlan(slots, counts)


@dataclass
class RecvPlan:
    """Where an owner rank puts what it receives.  indptr[e]: first row of
    local expert e; src_off[s, e]: first row of source s's rows of e;
    wait_count[e]: rows expert e waits for (its event's initial value)."""
    indptr: np.ndarray      # [experts per rank + 1]
    src_off: np.ndarray     # [world, experts per rank]
    wait_count: np.ndarray  # [experts per rank]


def recv_plan(counts_from: np.ndarray) -> RecvPlan:
    """counts_from[s, e]: rows source s sends to this rank's local expert e."""
    counts_from = np.asarray(counts_from, dtype=np.int64)
    wait = counts_from.sum(axis=0)
    indptr = np.concatenate([[0], np.cumsum(wait)])
    src_off = indptr[:-1][None, :] + np.cumsum(counts_from, axis=0) - counts_from
    return RecvPlan(indptr, src_off, wait)


def recv_rows(plan: RecvPlan, counts_from: np.ndarray, source: int) -> np.ndarray:
    """Receive-buffer rows, in arrival order, of the rows `source` sends (its
    send order: ascending local expert, then ascending token)."""
    counts_from = np.asarray(counts_from, dtype=np.int64)
    return np.concatenate([np.arange(plan.src_off[source, e], plan.src_off[source, e] + counts_from[source, e])
                           for e in range(counts_from.shape[1])]).astype(np.int64) \
        if counts_from.shape[1] else np.zeros(0, dtype=np.int64)
