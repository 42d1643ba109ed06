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


def test_stage_bytes_and_l2_resident_stages(bench):
    """Algorithmic bytes of the Wan-layer step's memory-bound stages, and the
    rule that a stage whose bytes fit in L2 gets no fraction of the HBM peak."""
    import synth
    wl = synth.WORKLOADS["wan"]

    class Shape:
        B, H, N, d, nb, Bt = wl.B, wl.H, wl.N, wl.d, wl.nb, wl.Bt

    nnz, demanded = 2_076_448, 5_000_000_000
    tensor = 40 * 30720 * 128 * 2
    b = bench.stage_bytes(Shape, wl, nnz, demanded, fused=True, overlapped=True)
    assert b["reorder"] == 6 * tensor + 2 * 40 * 240 * 128 * 4
    assert b["select"] == 4 * 40 * 240 * 240 + 4 * (nnz + 40 * 240 + 1)
    assert b["kv_gather"] == demanded + 2 * tensor
    serial = bench.stage_bytes(Shape, wl, nnz, demanded, fused=True, overlapped=False)
    assert "kv_gather" not in serial and serial["kv_demand"] == b["kv_demand"] + b["kv_gather"]
    h = bench.hbm_fractions({"reorder": 0.3, "select": 0.05, "missing": 1.0}, b, 6700.0)
    assert h["reorder"]["frac"] == pytest.approx(b["reorder"] / 0.3e-3 / 1e9 / 6700.0)
    assert h["select"]["frac"] is None and h["select"]["l2_resident"]
    assert "scores" not in h
