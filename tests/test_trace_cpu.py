"""CPU checks of the task-trace decoding and summary (host logic of the profiling aid)."""
import numpy as np
import pytest

from moe_layer_scheduling_gb300 import binding as B
from moe_layer_scheduling_gb300.trace import summarize


def _word(ty, blk, sm, a, b):
    # the kernel's packing: type<<56 | block<<48 | sm<<32 | a<<8 | (b & 0xFF)
    return (ty << 56) | (blk << 48) | (sm << 32) | (a << 8) | (b & 0xFF)


def test_decode_trace_unpacks_the_kernel_word():
    recs_in = [(6, 0, 151, 331, 5, 1000, 1100, 5100), (7, 3, 0, 131071, 255, 0, 2000, 2500),
               (2, 1, 17, 0, 0, 900, 900, 1900)]
    v = np.zeros(1 + 4 * 4, dtype=np.uint64)
    v[0] = len(recs_in)
    for i, (ty, blk, sm, a, b, td, ts, te) in enumerate(recs_in):
        v[1 + 4 * i: 5 + 4 * i] = [_word(ty, blk, sm, a, b), td, ts, te]
    out = B.decode_trace(v, max_records=4)
    assert [r["type"] for r in out] == ["gate_up", "down", "router"]
    assert [(r["block"], r["sm"], r["a"], r["b"]) for r in out] == \
        [(0, 151, 331, 5), (3, 0, 131071, 255), (1, 17, 0, 0)]
    assert [(r["t_dispatch"], r["t_start"], r["t_end"]) for r in out] == \
        [(1000, 1100, 5100), (0, 2000, 2500), (900, 900, 1900)]
    # a count above the buffer's records is clamped to what the caller asked for
    v[0] = 99
    assert len(B.decode_trace(v, max_records=2)) == 2


def test_summarize_spans_and_busy_fractions():
    # two SMs; times in ns from t0 = 1000 (the earliest dispatch)
    recs = [dict(type="router", block=0, sm=0, a=0, b=0, t_dispatch=1000, t_start=1000, t_end=3000),
            dict(type="router", block=0, sm=1, a=1, b=0, t_dispatch=1000, t_start=1500, t_end=3500),
            dict(type="down", block=0, sm=0, a=0, b=0, t_dispatch=0, t_start=4000, t_end=5000)]
    s = summarize(recs)
    assert s["span_us"] == pytest.approx(4.0)
    assert s["sms"] == 2
    assert s["worker_busy_frac"] == pytest.approx((2000 + 2000 + 1000) / (4000 * 2))
    r = s["stages"]["router"]
    assert r["tasks"] == 2 and r["busy_us_mean"] == pytest.approx(2.0)
    assert r["queue_us_mean"] == pytest.approx(0.25) and r["first_start_us"] == pytest.approx(0.0)
    d = s["stages"]["down"]
    assert d["queue_us_mean"] is None  # no dispatch time recorded
    assert d["last_end_us"] == pytest.approx(4.0)
    assert summarize([]) == {}


def test_summarize_busy_fraction_per_window():
    # two SMs, 20 us windows: [0, 20) holds 20 + 10 us of task time, [20, 40)
    # 10 + 20 us, [40, 60) 10 us (of 2 x 20 us each)
    recs = [dict(type="router", block=0, sm=0, a=0, b=0, t_dispatch=0, t_start=0, t_end=30000),
            dict(type="gate_up", block=0, sm=1, a=0, b=0, t_dispatch=0, t_start=10000, t_end=50000)]
    w = summarize(recs)["busy_frac_per_window"]
    assert w["window_us"] == pytest.approx(20.0)
    assert w["values"] == [0.75, 0.75, 0.25]
    # a call shorter than one window: one window of its own length
    w = summarize(recs[:1], window_ns=100000)["busy_frac_per_window"]
    assert w["window_us"] == pytest.approx(30.0) and w["values"] == [1.0]
