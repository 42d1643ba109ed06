"""Steps from pinned host memory to pinned host memory, overlapped.

HostPipeline.step() enqueues one whole forward step for inputs that live in
pinned host buffers and writes O back to a pinned host buffer;
HostPipeline.train_step() does the same for a forward + backward step (Q, K, V
and dO in; O, dQ, dK and dV out). The device input and output buffers are
double-buffered and the copies run on their own streams, so the host-to-device
copy of step n+1 and the device-to-host copy of step n-1 overlap the kernels
of step n; each input has its own copy event, so a step's kernels start on an
input as soon as it has landed, and in a training step O goes back while the
backward runs. Every step still copies its own inputs in and its own results
out; events order each buffer's reuse.
"""
from __future__ import annotations

import torch

from .pipeline import Pipeline


class HostPipeline:
    def __init__(self, pipe: Pipeline):
        self.pipe = pipe
        s = pipe.shape
        dt = s.torch_dtype
        raster = (s.B, s.N, s.H, s.d)
        self.inp = [[torch.empty(raster, dtype=dt, device="cuda") for _ in range(3)] for _ in range(2)]
        self.out = [torch.empty(raster, dtype=dt, device="cuda") for _ in range(2)]
        self.h2d = torch.cuda.Stream()
        self.d2h = torch.cuda.Stream()
        cur = torch.cuda.current_stream()
        mk = lambda: [torch.cuda.Event() for _ in range(2)]
        self.in_free, self.out_ready, self.out_free = mk(), mk(), mk()
        # one event per input copy, so that a step's kernels start on each input as soon as
        # it has landed rather than after all of them
        self.in_ready = [{x: torch.cuda.Event() for x in ("q", "k", "v", "do")} for _ in range(2)]
        self.o_ready = mk()
        for evs in (self.in_free, self.out_ready, self.out_free, self.o_ready):
            for e in evs:
                e.record(cur)
        self.n = 0
        self.t_inp = self.t_out = None

    def _copy_in(self, b, dsts, srcs, names):
        """Host-to-device copies of step buffers b on the copy stream, one event each."""
        with torch.cuda.stream(self.h2d):
            self.h2d.wait_event(self.in_free[b])          # step n-2 has consumed these buffers
            for dst, src, x in zip(dsts, srcs, names):
                dst.copy_(src, non_blocking=True)
                self.in_ready[b][x].record(self.h2d)

    def _waiter(self, b, cur):
        return lambda name: cur.wait_event(self.in_ready[b][name])

    def step(self, hq, hk, hv, ho, wq=None, wk=None):
        """One forward step: pinned host q, k, v (raster) in, pinned host O out."""
        b = self.n & 1
        cur = torch.cuda.current_stream()
        self._copy_in(b, self.inp[b], (hq, hk, hv), ("q", "k", "v"))
        cur.wait_event(self.out_free[b])                   # step n-2's O has left the device

        def mark(name, stream=None):
            if name == self.pipe.inputs_read_mark:         # raster inputs are no longer read
                self.in_free[b].record(cur)

        self.pipe.forward(*self.inp[b], wq=wq, wk=wk, mark=mark, out=self.out[b], before=self._waiter(b, cur))
        self.out_ready[b].record(cur)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.out_ready[b])
            ho.copy_(self.out[b], non_blocking=True)
            self.out_free[b].record(self.d2h)
        self.n += 1
        return ho

    def train_step(self, hq, hk, hv, hdo, ho, hdq, hdk, hdv, wq=None, wk=None):
        """One forward + backward step: pinned host q, k, v, dO (raster) in;
        pinned host O, dQ, dK, dV out. Needs a Pipeline built with backward=True."""
        if self.t_inp is None:
            s = self.pipe.shape
            raster = (s.B, s.N, s.H, s.d)
            mk = lambda n: [[torch.empty(raster, dtype=s.torch_dtype, device="cuda") for _ in range(n)]
                            for _ in range(2)]
            self.t_inp, self.t_out = mk(4), mk(4)
        b = self.n & 1
        cur = torch.cuda.current_stream()
        self._copy_in(b, self.t_inp[b], (hq, hk, hv, hdo), ("q", "k", "v", "do"))
        cur.wait_event(self.out_free[b])                   # step n-2's results have left the device

        def mark(name, stream=None):
            if name == "reorder_dout":                     # every raster input has been read
                self.in_free[b].record(cur)

        q, k, v, do = self.t_inp[b]
        o, dq, dk, dv = self.t_out[b]
        waiter = self._waiter(b, cur)
        self.pipe.forward(q, k, v, wq=wq, wk=wk, out=o, before=waiter)
        # O goes back while the backward runs (the backward only reads it)
        self.o_ready[b].record(cur)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.o_ready[b])
            ho.copy_(o, non_blocking=True)
        self.pipe.backward(do, mark=mark, outs=(dq, dk, dv), before=waiter)
        self.out_ready[b].record(cur)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.out_ready[b])
            for dst, src in zip((hdq, hdk, hdv), (dq, dk, dv)):
                dst.copy_(src, non_blocking=True)
            self.out_free[b].record(self.d2h)
        self.n += 1
        return ho, hdq, hdk, hdv

    def synchronize(self):
        self.d2h.synchronize()
