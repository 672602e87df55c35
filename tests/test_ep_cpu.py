"""Expert parallelism's dispatch and combine protocol, run as two gloo processes on CPU.

Each rank routes its own tokens, the experts are split between the ranks, and
the plan in moe_layer_scheduling_gb300/ep.py decides which rows go where: the
count exchange, the owner's per-expert event init (wait_count = rows from all
sources), the dispatch into the owner's receive buffer with a notify per
source, the expert FFNs (the oracle's, fp64), and the combine back to the
source in j order.  Every rank's result must equal the one-GPU layer the
oracle computes on that rank's tokens, and every counter must reach zero
exactly.  No GPU is used; the multi-GPU kernel is not built (one GPU per box).
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

from moe_layer_scheduling_gb300 import ep

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plan_on_one_rank_is_the_one_gpu_dispatch(oracle_lib):
    # World size 1: the receive buffer is the one-GPU expert-sorted order.
    ids = np.array([[3, 1], [0, 3], [1, 2], [3, 0]], dtype=np.int32)
    sp = ep.send_plan(ids, 4, 1)
    rp = ep.recv_plan(sp.counts)
    counts, indptr, pos, row_token = oracle_lib.dispatch(ids, 4)
    assert np.array_equal(rp.wait_count, counts)
    assert np.array_equal(rp.indptr, indptr)
    rows = ep.recv_rows(rp, sp.counts, 0)
    # the row each sent slot lands in is the one-GPU pos of that slot
    assert np.array_equal(rows, pos.reshape(-1)[sp.slots[0]])


def test_plan_counts_and_offsets_by_hand():
    # E = 4 over 2 ranks: rank 0 owns experts 0, 1; rank 1 owns 2, 3.
    ids = np.array([[2, 0], [3, 2], [1, 0]], dtype=np.int32)
    sp = ep.send_plan(ids, 4, 2)
    assert sp.counts.tolist() == [[2, 1], [2, 1]]
    # to rank 0: expert 0 from tokens 0, 2 (slots 1, 5), then expert 1 (slot 4)
    assert sp.slots[0].tolist() == [1, 5, 4]
    # to rank 1: expert 2 from tokens 0, 1 (slots 0, 3), then expert 3 (slot 2)
    assert sp.slots[1].tolist() == [0, 3, 2]
    # an owner receiving [2, 1] from source 0 and [1, 3] from source 1
    rp = ep.recv_plan(np.array([[2, 1], [1, 3]]))
    assert rp.wait_count.tolist() == [3, 4]
    assert rp.indptr.tolist() == [0, 3, 7]
    assert rp.src_off.tolist() == [[0, 3], [2, 4]]
    assert ep.recv_rows(rp, np.array([[2, 1], [1, 3]]), 1).tolist() == [2, 4, 5, 6]


_RANK = r"""
import json, sys
import numpy as np
import torch
import torch.distributed as dist
sys.path.insert(0, {root!r})
import oracle
from moe_layer_scheduling_gb300 import ep, inputs

dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
H, E, k, I = 64, 8, 2, 32
per = E // world
w = inputs.moe_weights(H, E, k, I, seed=3)
w.router_bias = inputs.zipf_bias(E, 1.2, 3)
T = [7, 12][rank]
x = inputs.tokens(T, H, 50 + rank)
L = oracle.router_logits(x, w.gate_w, w.router_bias)
ids, wts = oracle.route(L, k)


def exchange(send, shapes, dtype):
    recv = [torch.empty(s, dtype=dtype) for s in shapes]
    reqs = [dist.irecv(recv[s], src=s) for s in range(world) if s != rank]
    reqs += [dist.isend(send[d], dst=d) for d in range(world) if d != rank]
    for r in reqs:
        r.wait()
    recv[rank] = send[rank].clone()
    return recv


# 1. count exchange
sp = ep.send_plan(ids, E, world)
counts_from = torch.stack(exchange([torch.from_numpy(sp.counts[d]) for d in range(world)],
                                   [(per,)] * world, torch.int64)).numpy()
# 2. data-dependent event init on the owner
rp = ep.recv_plan(counts_from)
event = rp.wait_count.copy()
assert np.array_equal(event, counts_from.sum(axis=0))
# 3. dispatch: rows (bf16 bit patterns) straight into the receive buffer, one notify per source and expert
xbits = x.view(torch.int16)
send_rows = [xbits[torch.from_numpy(sp.slots[d] // k)].contiguous() for d in range(world)]
got = exchange(send_rows, [(int(counts_from[s].sum()), H) for s in range(world)], torch.int16)
buf = torch.zeros(int(rp.indptr[-1]), H, dtype=torch.int16)
fired = []
for s in range(world):
    buf[torch.from_numpy(ep.recv_rows(rp, counts_from, s))] = got[s]
    for e in range(per):
        before = event[e]
        event[e] -= counts_from[s, e]
        if before > 0 and event[e] == 0:
            fired.append(e)
assert (event == 0).all() and sorted(fired) == [e for e in range(per) if rp.wait_count[e] > 0]
# 4. expert FFNs of the owner's rows, expert e on rows [indptr[e], indptr[e+1])
xrows = buf.view(torch.bfloat16)
y = np.zeros((buf.shape[0], H))
for e in range(per):
    ge = rank * per + e
    for r in range(rp.indptr[e], rp.indptr[e + 1]):
        y[r] = oracle.expert_ffn(xrows[r], w.w_gate_up[ge], w.w_down[ge])
# 5. combine: rows back to their sources in arrival order, into slot (t, j); a counter of k per token
back = [torch.from_numpy(y[ep.recv_rows(rp, counts_from, s)]) for s in range(world)]
ret = exchange(back, [(len(sp.slots[d]), H) for d in range(world)], torch.float64)
yslot = np.full((T * k, H), np.nan)
tok_event = np.full(T, k)
for d in range(world):
    yslot[sp.slots[d]] = ret[d].numpy()
    np.subtract.at(tok_event, sp.slots[d] // k, 1)
assert (tok_event == 0).all()
out = np.zeros((T, H))
for j in range(k):
    out += wts[:, j:j + 1] * yslot[j::k]
ref = oracle.moe_layer(x, w.gate_w, w.w_gate_up, w.w_down, k, bias=w.router_bias)
print(json.dumps({{"rank": rank, "T": T, "max_err": float(np.max(np.abs(out - ref))),
                  "scale": float(np.max(np.abs(ref))), "rows_received": int(rp.indptr[-1]),
                  "rows_sent": [len(s) for s in sp.slots]}}), flush=True)
dist.destroy_process_group()
"""


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_ep_dispatch_and_combine_world2_gloo(oracle_lib):
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(r), LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK.format(root=ROOT)], env=env,
                                      cwd=ROOT, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=240)
        assert p.returncode == 0, err[-3000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    outs.sort(key=lambda d: d["rank"])
    # every row sent is received by its owner
    assert sum(o["rows_received"] for o in outs) == sum(sum(o["rows_sent"]) for o in outs) == (7 + 12) * 2
    for o in outs:
        # the same fp64 arithmetic as the one-GPU layer, summed in the same order
        assert o["max_err"] <= 1e-12 * o["scale"], o
