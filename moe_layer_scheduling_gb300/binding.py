"""Thin ctypes binding of libetc_moe.so: argument marshalling only.

Every function here has the name of the C entry point it calls
(``include/etc_moe.h``) and passes torch tensors as raw device pointers and the
current torch stream as the cudaStream_t.  All computation happens in the
library's CUDA kernels; there is no fallback.  Loading fails loudly if the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

ETC_OK = 0
ETC_ERR_INVALID = -1
ETC_ERR_CUDA = -2
ETC_ERR_TIMEOUT = -3
ETC_ERR_UNIMPLEMENTED = -4
ETC_ERR_STATE = -5
ETC_SCHED_STATIC = 0
ETC_SCHED_DYNAMIC = 1
ETC_SCHED_MIXED = 2
ETC_DEBUG_FAULT_EXTRA_WAIT = 0x1
ETC_DEBUG_POISON = 0x2
ETC_DEBUG_NO_PAIR = 0x8
ETC_DEBUG_PAIR_MOE = 0x10
ETC_DEBUG_NO_HEAVY = 0x20
ETC_DEBUG_WIDE_SWAP_AB = 0x40
ETC_OUT_F32 = 0
ETC_OUT_BF16 = 1
ETC_COMBINE_FUSED = 0
ETC_COMBINE_ORDERED = 1

EXPORTED = [
    "etc_moe_plan", "etc_moe_forward", "etc_moe_forward_unfused", "etc_moe_route_from_logits",
    "etc_moe_debug_routing", "etc_moe_debug_buffer", "etc_moe_debug_trace", "etc_chain_forward",
    "etc_plan_check", "etc_plan_reset",
    "etc_plan_stats", "etc_plan_destroy", "etc_splitk_rowsum", "etc_splitk_rowsum_ex",
    "etc_splitk_check", "etc_splitk_rowsum_noalloc", "etc_launch_count", "etc_last_error",
    "etc_mlp_plan", "etc_mlp_forward", "etc_mlp_forward_unfused", "etc_chain_plan",
]


class EtcError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"etc error {code}: {msg}")
        self.code = code


class etc_moe_opts(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
        ("inter", ctypes.c_int), ("t_max", ctypes.c_int), ("sched", ctypes.c_int),
        ("n_blocks", ctypes.c_int), ("rms_eps", ctypes.c_float),
        ("router_bias", ctypes.c_void_p), ("wait_timeout_ns", ctypes.c_ulonglong),
        ("debug_flags", ctypes.c_uint), ("debug_arg", ctypes.c_int),
        ("out_dtype", ctypes.c_int), ("combine", ctypes.c_int),
    ]


class etc_mlp_opts(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int), ("inter", ctypes.c_int), ("t_max", ctypes.c_int),
        ("sched", ctypes.c_int), ("wait_timeout_ns", ctypes.c_ulonglong),
        ("debug_flags", ctypes.c_uint), ("out_dtype", ctypes.c_int), ("debug_arg", ctypes.c_int),
    ]


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libetc_moe.so (building it first when asked and needed)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build_if_missing else _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"libetc_moe.so not built at {path}; run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    P, I, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
    L.etc_moe_plan.argtypes = [ctypes.POINTER(P), ctypes.POINTER(etc_moe_opts)]
    L.etc_moe_forward.argtypes = [P, P, P, P, P, P, I, P]
    L.etc_moe_forward_unfused.argtypes = [P, P, P, P, P, P, I, P]
    L.etc_moe_route_from_logits.argtypes = [P, P, P, P, I]
    L.etc_moe_debug_routing.argtypes = [P, P, I, P, P, P, P, P, P]
    L.etc_moe_debug_buffer.argtypes = [P, P, I, P, ctypes.c_ulonglong]
    L.etc_moe_debug_trace.argtypes = [P, P, P, I]
    L.etc_chain_forward.argtypes = [P, P, P, P, P, P, P, P, I, P]
    L.etc_mlp_plan.argtypes = [ctypes.POINTER(P), ctypes.POINTER(etc_mlp_opts)]
    L.etc_chain_plan.argtypes = [ctypes.POINTER(P), ctypes.POINTER(etc_moe_opts), I]
    L.etc_mlp_forward.argtypes = [P, P, P, P, P, I, P]
    L.etc_mlp_forward_unfused.argtypes = [P, P, P, P, P, I, P]
    L.etc_plan_check.argtypes = [P]
    L.etc_plan_reset.argtypes = [P, P]
    L.etc_plan_stats.argtypes = [P, ctypes.POINTER(LL), I]
    L.etc_plan_destroy.argtypes = [P]
    L.etc_plan_destroy.restype = None
    L.etc_splitk_rowsum.argtypes = [P, P, LL, LL, I, P, I]
    L.etc_splitk_rowsum_ex.argtypes = [P, P, LL, LL, I, P, I, ctypes.c_ulonglong, ctypes.c_uint, LL]
    L.etc_splitk_check.argtypes = []
    L.etc_splitk_rowsum_noalloc.argtypes = [P, P, LL, LL, I, P, I]
    L.etc_launch_count.restype = LL
    L.etc_last_error.restype = ctypes.c_char_p
    for name in EXPORTED:
        if name not in ("etc_plan_destroy", "etc_launch_count", "etc_last_error"):
            getattr(L, name).restype = I
    _lib = L
    return L


def _check(rc: int):
    if rc != ETC_OK:
        raise EtcError(rc, load().etc_last_error().decode())
    return rc


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensor must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owns an etc_plan_t; destroyed with the object."""

    def __init__(self, handle: int, opts: etc_moe_opts, keep=None):
        self.handle = handle
        self.opts = opts
        self._keep = keep

    @property
    def out_dtype(self):
        import torch
        return torch.bfloat16 if self.opts.out_dtype == ETC_OUT_BF16 else torch.float32

    def close(self):
        if self.handle:
            load().etc_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def etc_moe_plan(hidden, n_experts, top_k, inter, t_max, sched=ETC_SCHED_STATIC, n_blocks=1,
                 rms_eps=1e-6, router_bias=None, wait_timeout_ns=0, debug_flags=0,
                 debug_arg=0, out_dtype=ETC_OUT_F32, combine=ETC_COMBINE_FUSED) -> Plan:
    o = etc_moe_opts(hidden, n_experts, top_k, inter, t_max, sched, n_blocks, rms_eps,
                     _ptr(router_bias), wait_timeout_ns, debug_flags, debug_arg, out_dtype, combine)
    h = ctypes.c_void_p()
    _check(load().etc_moe_plan(ctypes.byref(h), ctypes.byref(o)))
    return Plan(h.value, o, keep=router_bias)


def etc_moe_forward(plan: Plan, x, gate_w, w_gate_up, w_down, T, out, stream=None):
    return _check(load().etc_moe_forward(plan.handle, _stream(stream), _ptr(x), _ptr(gate_w),
                                         _ptr(w_gate_up), _ptr(w_down), int(T), _ptr(out)))


def etc_moe_forward_unfused(plan: Plan, x, gate_w, w_gate_up, w_down, T, out, stream=None):
    return _check(load().etc_moe_forward_unfused(plan.handle, _stream(stream), _ptr(x),
                                                 _ptr(gate_w), _ptr(w_gate_up), _ptr(w_down),
                                                 int(T), _ptr(out)))


def etc_chain_plan(n_blocks, hidden, n_experts, top_k, inter, t_max, sched=ETC_SCHED_STATIC,
                   rms_eps=1e-6, wait_timeout_ns=0, debug_flags=0, debug_arg=0,
                   out_dtype=ETC_OUT_F32, combine=ETC_COMBINE_FUSED) -> Plan:
    o = etc_moe_opts(hidden, n_experts, top_k, inter, t_max, sched, 1, rms_eps, None,
                     wait_timeout_ns, debug_flags, debug_arg, out_dtype, combine)
    h = ctypes.c_void_p()
    _check(load().etc_chain_plan(ctypes.byref(h), ctypes.byref(o), int(n_blocks)))
    o.n_blocks = int(n_blocks)
    return Plan(h.value, o)


def etc_mlp_plan(hidden, inter, t_max, sched=ETC_SCHED_STATIC, wait_timeout_ns=0, debug_flags=0,
                 out_dtype=ETC_OUT_F32, debug_arg=0) -> Plan:
    o = etc_mlp_opts(hidden, inter, t_max, sched, wait_timeout_ns, debug_flags, out_dtype, debug_arg)
    h = ctypes.c_void_p()
    _check(load().etc_mlp_plan(ctypes.byref(h), ctypes.byref(o)))
    return Plan(h.value, o)


def etc_mlp_forward(plan: Plan, x, w_gate_up, w_down, T, out, stream=None):
    return _check(load().etc_mlp_forward(plan.handle, _stream(stream), _ptr(x), _ptr(w_gate_up),
                                         _ptr(w_down), int(T), _ptr(out)))


def etc_mlp_forward_unfused(plan: Plan, x, w_gate_up, w_down, T, out, stream=None):
    return _check(load().etc_mlp_forward_unfused(plan.handle, _stream(stream), _ptr(x),
                                                 _ptr(w_gate_up), _ptr(w_down), int(T), _ptr(out)))


def etc_moe_route_from_logits(plan: Plan, logits, x, T, stream=None):
    return _check(load().etc_moe_route_from_logits(plan.handle, _stream(stream), _ptr(logits),
                                                   _ptr(x), int(T)))


def etc_moe_debug_routing(plan: Plan, block=0, logits=None, topk_ids=None, topk_w=None,
                          counts=None, exp_indptr=None, pos=None, stream=None):
    return _check(load().etc_moe_debug_routing(plan.handle, _stream(stream), int(block),
                                               _ptr(logits), _ptr(topk_ids), _ptr(topk_w),
                                               _ptr(counts), _ptr(exp_indptr), _ptr(pos)))


def etc_moe_debug_buffer(plan: Plan, which: int, dst, stream=None):
    """which: 0 x_perm, 1 act, 2 y_perm; fills all of `dst` (a CUDA tensor)."""
    return _check(load().etc_moe_debug_buffer(plan.handle, _stream(stream), int(which), _ptr(dst),
                                              dst.numel() * dst.element_size()))


def etc_chain_forward(plan: Plan, x, norm_w, gate_w, router_bias, w_gate_up, w_down, T, out,
                      stream=None):
    n = plan.opts.n_blocks
    for name, ts in (("norm_w", norm_w), ("gate_w", gate_w), ("w_gate_up", w_gate_up),
                     ("w_down", w_down), ("router_bias", router_bias)):
        if ts is not None and len(ts) != n:
            raise ValueError(f"{name}: the plan has {n} blocks, got {len(ts)} tensors")
    arr = ctypes.c_void_p * n

    def ptrs(ts):
        return arr(*[_ptr(t) for t in ts])

    nw, gw, gu, dw = ptrs(norm_w), ptrs(gate_w), ptrs(w_gate_up), ptrs(w_down)
    bias = ptrs(router_bias) if router_bias is not None else None
    return _check(load().etc_chain_forward(plan.handle, _stream(stream), _ptr(x), nw, gw, bias,
                                           gu, dw, int(T), _ptr(out)))


def etc_plan_check(plan: Plan) -> int:
    rc = load().etc_plan_check(plan.handle)
    return rc


def etc_plan_reset(plan: Plan, stream=None):
    return _check(load().etc_plan_reset(plan.handle, _stream(stream)))


def etc_plan_stats(plan: Plan) -> dict:
    out = (ctypes.c_longlong * 8)()
    _check(load().etc_plan_stats(plan.handle, out, 8))
    keys = ["launches", "grid", "smem_bytes", "epoch", "token_block", "max_chunk_rows",
            "queue_capacity", "max_chunks"]
    return dict(zip(keys, list(out)))


def etc_splitk_rowsum(A, n_split, C, sched=ETC_SCHED_STATIC, stream=None):
    n_rows, n_cols = A.shape
    return _check(load().etc_splitk_rowsum(_stream(stream), _ptr(A), n_rows, n_cols, int(n_split),
                                           _ptr(C), int(sched)))


def etc_splitk_rowsum_ex(A, n_split, C, sched=ETC_SCHED_STATIC, wait_timeout_ns=0,
                         debug_flags=0, debug_arg=-1, stream=None):
    n_rows, n_cols = A.shape
    return load().etc_splitk_rowsum_ex(_stream(stream), _ptr(A), n_rows, n_cols, int(n_split),
                                       _ptr(C), int(sched), int(wait_timeout_ns),
                                       int(debug_flags), int(debug_arg))


def etc_splitk_check() -> int:
    return load().etc_splitk_check()


def etc_launch_count() -> int:
    return int(load().etc_launch_count())


def etc_last_error() -> str:
    return load().etc_last_error().decode()


def etc_plan_destroy(plan: Plan):
    plan.close()


def etc_splitk_rowsum_noalloc(A, n_split, C, sched=ETC_SCHED_STATIC, stream=None):
    """Split-K row sum whose scratch is a fixed array inside the library (no allocation)."""
    n_rows, n_cols = A.shape
    return _check(load().etc_splitk_rowsum_noalloc(_stream(stream), _ptr(A), n_rows, n_cols,
                                                   int(n_split), _ptr(C), int(sched)))


ETC_DEBUG_TRACE = 0x4
TASK_NAMES = {1: "norm", 2: "router", 3: "topk", 4: "scan", 5: "perm", 6: "gate_up", 7: "down",
              8: "combine"}


def etc_moe_debug_trace(plan: Plan, max_records: int = 65536, stream=None):
    """Task trace of the last call as a list of dicts (type, block, sm, a, b, times in ns)."""
    import torch
    buf = torch.zeros(1 + 4 * max_records, dtype=torch.int64, device="cuda")
    _check(load().etc_moe_debug_trace(plan.handle, _stream(stream), _ptr(buf), int(max_records)))
    torch.cuda.synchronize()
    return decode_trace(buf.cpu().numpy().astype("uint64"), max_records)


def decode_trace(v, max_records: int) -> list[dict]:
    """Records of a trace buffer (uint64 [1 + 4n]): v[0] = count, then per task the
    word (type<<56 | block<<48 | sm<<32 | a<<8 | b), dispatch, start and end times."""
    n = int(min(int(v[0]), max_records))
    recs = []
    for i in range(n):
        w0, t_disp, t0, t1 = (int(x) for x in v[1 + 4 * i: 5 + 4 * i])
        recs.append(dict(type=TASK_NAMES.get(w0 >> 56, str(w0 >> 56)), block=(w0 >> 48) & 0xFF,
                         sm=(w0 >> 32) & 0xFFFF, a=(w0 >> 8) & 0xFFFFFF, b=w0 & 0xFF,
                         t_dispatch=t_disp, t_start=t0, t_end=t1))
    return recs
