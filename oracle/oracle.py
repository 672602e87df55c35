"""ctypes front end of the fp64 C++ oracle (TEST INFRASTRUCTURE ONLY).

``build()`` compiles ``etc_oracle.cpp`` with the host C++ compiler into
``oracle/_build/libetc_oracle.so``; the functions below marshal numpy arrays and
return numpy results.  Each wrapper names the step of the Event Tensor pages it
restates (see the C++ source for the citations).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "etc_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libetc_oracle.so")
_lib = None
_lock = threading.Lock()

__all__ = [
    "build", "lib", "set_threads", "get_threads", "router_logits", "route", "route_f32",
    "dispatch", "expert_ffn", "mlp", "moe_layer", "chain", "splitk", "event_sim",
]


def build(force: bool = False) -> str:
    """Compile the oracle shared library (plain g++, fp64, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    compile_source(_SRC, tmp)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    """The loaded oracle library.

    ``ETC_ORACLE_LIB`` may name another build of the same source (the mutation
    test uses it to load deliberately broken copies).
    """
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("ETC_ORACLE_LIB") or build()
            _lib = ctypes.CDLL(path)
            _declare(_lib)
    return _lib


def compile_source(src: str, out_path: str) -> str:
    """Compile a C++ source file with the oracle's flags into ``out_path``."""
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", src, "-o", out_path]
    subprocess.run(cmd, check=True)
    return out_path


_P = ctypes.c_void_p
_L = ctypes.c_long
_I = ctypes.c_int


def _declare(L):
    L.oracle_set_threads.argtypes = [_I]
    L.oracle_get_threads.restype = _I
    L.oracle_router_logits.argtypes = [_P, _P, _P, _L, _I, _I, _P]
    L.oracle_route_f64.argtypes = [_P, _L, _I, _I, _P, _P]
    L.oracle_route_f32.argtypes = [_P, _L, _I, _I, _P, _P]
    L.oracle_dispatch.argtypes = [_P, _L, _I, _I, _P, _P, _P, _P]
    L.oracle_expert_ffn.argtypes = [_P, _P, _P, _I, _I, _P]
    L.oracle_mlp.argtypes = [_P, _P, _P, _L, _I, _I, _P, _L, _P]
    L.oracle_moe_layer.argtypes = [_P, _P, _P, _P, _P, _L, _I, _I, _I, _I, _P, _P, _P, _P]
    L.oracle_chain.argtypes = [_P, _I, _P, _P, _P, _P, _P, _L, _I, _I, _I, _I, ctypes.c_double,
                               _P, _P, _P]
    L.oracle_chain_routed.argtypes = [_P, _I, _P, _P, _P, _P, _P, _L, _I, _I, _I, _I,
                                      ctypes.c_double, _P, _P, _P, _P]
    L.oracle_splitk.argtypes = [_P, _L, _L, _I, _P, _P]
    L.oracle_event_sim.argtypes = [_L, _I, _I, ctypes.c_char_p, ctypes.c_char_p,
                                   ctypes.c_ulonglong, _P, _P, _P, _P, _P]
    L.oracle_event_sim.restype = _L
    for name in ("oracle_router_logits", "oracle_route_f64", "oracle_route_f32",
                 "oracle_dispatch", "oracle_expert_ffn", "oracle_moe_layer", "oracle_chain",
                 "oracle_chain_routed", "oracle_splitk"):
        getattr(L, name).restype = _I


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(t):
    """bf16 torch tensor or uint16 numpy array -> contiguous uint16 numpy array."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16, t.dtype
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _f32(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return np.ascontiguousarray(t, dtype=np.float32)
    return t.detach().cpu().contiguous().float().numpy()


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(lib().oracle_get_threads())


def router_logits(x, gate_w, bias=None):
    """fp64 logits [T, E] = x @ gate_w (+ bias)."""
    xb, wb, bb = _u16(x), _u16(gate_w), _f32(bias)
    T, H = xb.shape
    E = wb.shape[1]
    out = np.empty((T, E), dtype=np.float64)
    _check(lib().oracle_router_logits(_ptr(xb), _ptr(wb), _ptr(bb), T, H, E, _ptr(out)), "router")
    return out


def route(logits: np.ndarray, k: int):
    """Top-k ids (ties -> lower id) and renormalised softmax weights from fp64 logits."""
    L = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = L.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    _check(lib().oracle_route_f64(_ptr(L), T, E, k, _ptr(ids), _ptr(w)), "route")
    return ids, w


def route_f32(logits: np.ndarray, k: int):
    """The same routing rule applied to fp32 logits (compared exactly)."""
    L = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = L.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    _check(lib().oracle_route_f32(_ptr(L), T, E, k, _ptr(ids), _ptr(w)), "route_f32")
    return ids, w


def dispatch(ids: np.ndarray, n_experts: int):
    """counts [E], exp_indptr [E+1], pos [T,k], row_token [T*k] of the stable permutation."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    counts = np.empty(n_experts, dtype=np.int32)
    indptr = np.empty(n_experts + 1, dtype=np.int32)
    pos = np.empty((T, k), dtype=np.int32)
    row_token = np.empty(T * k, dtype=np.int32)
    _check(lib().oracle_dispatch(_ptr(ids), T, n_experts, k, _ptr(counts), _ptr(indptr),
                                 _ptr(pos), _ptr(row_token)), "dispatch")
    return counts, indptr, pos, row_token


def expert_ffn(x_row, w_gate_up_e, w_down_e):
    """y = (silu(x Wg^T) * (x Wu^T)) Wd^T for one bf16 row and one expert."""
    xb, a, b = _u16(x_row).reshape(-1), _u16(w_gate_up_e), _u16(w_down_e)
    H = xb.shape[0]
    I = a.shape[0] // 2
    y = np.empty(H, dtype=np.float64)
    _check(lib().oracle_expert_ffn(_ptr(xb), _ptr(a), _ptr(b), H, I, _ptr(y)), "expert_ffn")
    return y


def mlp(x, w_gate_up, w_down, rows=None):
    """fp64 dense MLP (silu(x Wg^T) * (x Wu^T)) Wd^T on rows of x [T, H] (all rows if None)."""
    xb, a, b = _u16(x), _u16(w_gate_up), _u16(w_down)
    T, H = xb.shape
    I = a.shape[0] // 2
    if rows is None:
        n, rp = T, None
    else:
        rp = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = rp.shape[0]
    out = np.empty((n, H), dtype=np.float64)
    _check(lib().oracle_mlp(_ptr(xb), _ptr(a), _ptr(b), T, H, I,
                            None if rp is None else _ptr(rp), n, _ptr(out)), "mlp")
    return out


def moe_layer(x, gate_w, w_gate_up, w_down, top_k: int, bias=None, want_routing=False):
    """fp64 MoE layer output [T, H]; with want_routing also (logits, ids, weights)."""
    xb, wg, wgu, wd, bb = _u16(x), _u16(gate_w), _u16(w_gate_up), _u16(w_down), _f32(bias)
    T, H = xb.shape
    E = wg.shape[1]
    I = wgu.shape[1] // 2
    out = np.empty((T, H), dtype=np.float64)
    logits = np.empty((T, E), dtype=np.float64)
    ids = np.empty((T, top_k), dtype=np.int32)
    w = np.empty((T, top_k), dtype=np.float64)
    _check(lib().oracle_moe_layer(_ptr(xb), _ptr(wg), _ptr(bb), _ptr(wgu), _ptr(wd), T, H, E,
                                  top_k, I, _ptr(out), _ptr(logits), _ptr(ids), _ptr(w)),
           "moe_layer")
    return (out, logits, ids, w) if want_routing else out


def chain(x, blocks, eps: float = 1e-6, want_routing=False, ids_in=None):
    """fp64 chain x <- x + MoE_b(RMSNorm_b(x)) over the given blocks (MoEWeights-like).

    ids_in (optional int [n_blocks, T, k]): the experts of every token in every
    block, given instead of selected; each block still weights them by the
    softmax of its own fp64 logits over the given experts."""
    xb = _u16(x)
    T, H = xb.shape
    nb = len(blocks)
    keep = []

    def arr_ptrs(arrs):
        keep.extend(arrs)
        P = (ctypes.c_void_p * nb)(*[a.ctypes.data for a in arrs])
        keep.append(P)
        return P

    norm = arr_ptrs([_u16(b.norm_w) for b in blocks])
    wg = arr_ptrs([_u16(b.gate_w) for b in blocks])
    wgu = arr_ptrs([_u16(b.w_gate_up) for b in blocks])
    wd = arr_ptrs([_u16(b.w_down) for b in blocks])
    if any(b.router_bias is not None for b in blocks):
        bias = arr_ptrs([_f32(b.router_bias) for b in blocks])
    else:
        bias = None
    E = blocks[0].n_experts
    k = blocks[0].top_k
    I = blocks[0].inter
    out = np.empty((T, H), dtype=np.float64)
    ids = np.empty((nb, T, k), dtype=np.int32)
    logits = np.empty((nb, T, E), dtype=np.float64)
    if ids_in is None:
        _check(lib().oracle_chain(_ptr(xb), nb, norm, wg, bias, wgu, wd, T, H, E, k, I, float(eps),
                                  _ptr(out), _ptr(ids), _ptr(logits)), "chain")
    else:
        given = np.ascontiguousarray(ids_in, dtype=np.int32)
        assert given.shape == (nb, T, k), given.shape
        _check(lib().oracle_chain_routed(_ptr(xb), nb, norm, wg, bias, wgu, wd, T, H, E, k, I,
                                         float(eps), _ptr(out), _ptr(ids), _ptr(logits),
                                         _ptr(given)), "chain")
    return (out, ids, logits) if want_routing else out


def splitk(A, n_split: int):
    """(B [n_rows, n_split], C [n_rows]) in fp64 for the split-K row sum."""
    a = _f32(A)
    n_rows, n_cols = a.shape
    B = np.empty((n_rows, n_split), dtype=np.float64)
    C = np.empty(n_rows, dtype=np.float64)
    _check(lib().oracle_splitk(_ptr(a), n_rows, n_cols, n_split, _ptr(B), _ptr(C)), "splitk")
    return B, C


def event_sim(part_val: np.ndarray, wait_count: int, out_map: str = "ij->i",
              in_map: str = "i->i", seed: int = 0):
    """Run the split-K event graph in a random ready order.

    Returns (C, notifies_per_event, early_consumer_starts, executed_order).
    """
    pv = np.ascontiguousarray(part_val, dtype=np.float64)
    n_rows, n_split = pv.shape
    C = np.full(n_rows, np.nan)
    notes = np.zeros(n_rows, dtype=np.int32)
    early = np.zeros(1, dtype=np.int32)
    order = np.zeros(n_rows * n_split + n_rows, dtype=np.int64)
    ran = lib().oracle_event_sim(n_rows, n_split, wait_count, out_map.encode(), in_map.encode(),
                                 seed, _ptr(pv), _ptr(C), _ptr(notes), _ptr(early), _ptr(order))
    if ran < 0:
        raise ValueError("bad index map")
    return C, notes, int(early[0]), order[:ran]
