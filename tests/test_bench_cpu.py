"""bench.py's host-side bookkeeping on CPU: stage times from the event marks
of one or two streams."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def elapsed(a, b):
    return b - a


def test_serial_stages_run_mark_to_mark(bench):
    marks = [("step_start", 0.0), ("reorder", 1.0), ("select", 1.5), ("kv_demand", 2.5), ("attn_fwd", 12.5),
             ("reorder_out", 13.0)] * 1
    st = bench.stage_times(marks, (), elapsed, 1)
    assert st == {"reorder": 1.0, "select": 0.5, "kv_demand": 1.0, "attn_fwd": 10.0, "reorder_out": 0.5}


def test_overlapped_stages_use_their_begin_marks(bench):
    # gather (side stream) 1.5 -> 4.0 beside attention 1.5 -> 11.5; the caller's stream
    # joins both at 11.6; the inverse reorder follows the join, not the side marks
    one = [("step_start", 0.0), ("select", 1.4), ("kv_demand", 1.5), ("overlap:begin", 1.5),
           ("attn_fwd:begin", 1.5), ("attn_fwd", 11.5), ("kv_gather:begin", 1.5), ("kv_gather", 4.0),
           ("overlap", 11.6), ("reorder_out", 12.1)]
    two = [(n, t + 20.0) for n, t in one]
    st = bench.stage_times(one + two, ("attn_fwd", "kv_gather"), elapsed, 2)
    assert st["attn_fwd"] == pytest.approx(10.0)
    assert st["kv_gather"] == pytest.approx(2.5)
    assert st["overlap"] == pytest.approx(10.1)
    assert st["reorder_out"] == pytest.approx(0.5)
    assert st["select"] == pytest.approx(1.4)
    assert st["kv_demand"] == pytest.approx(0.1)
