"""The whole hot path as one object with preallocated device buffers.

forward(): reorder Q, K, V into tiles -> block scores -> Top-p/Top-k selection
-> (optional) head balancing over P virtual ranks and slack-aware augmentation
of the CSR -> (optional) dependency-aware placement of blocks on the P
partitions -> KV demand of P partitions (+ gather) -> block-sparse attention
-> O in raster order (written there by attention itself where the tcgen05
kernel runs, else by an inverse reorder). backward(): dO into tiles ->
attention backward -> dQ, dK, dV in raster order (likewise). Every step is one
or more libsparsp kernels on the current stream, except that by default the
KV demand gather runs on a side
stream beside attention (the caller's stream waits for both); nothing here
allocates after construction. capture() records forward() (and, with a
backward, forward() + backward()) as one CUDA graph, for shapes where the
host's launches, not the kernels, set the pace.
"""
from __future__ import annotations

import dataclasses

import torch

from . import (EST_LOWRANK, EST_MEAN, PROF_SLOTS, Shape, attn_bwd, attn_fwd, attn_workspace_size, augment,
               augment_workspace_size, balance_heads, Balance, predictor_fit,
               block_scores, block_scores_pooled, block_scores_workspace_size, kv_demand, kv_gather, lib, placement,
               placement_workspace_size, reorder, reorder_pool, select, select_workspace_size, DemandOut,
               OUT_RASTER, IN_RASTER, pool_means)


class Pipeline:
    def kernels_per_forward(self) -> int:
        """Kernels forward() launches: reorder x3, pool + product, select x3 (count,
        scan, fill), predictor fitting x7 when enabled, balancing (1) and augmentation x14 (keys, slack, four
        histogram + digit passes, row counts, ties, scan, fill) when enabled, placement x2 (affinity, greedy) when
        enabled, demand x5 (counter reset, bitmap, scan, list, gather), schedule (1, or 2 in
        flat order) + attention, inverse reorder (none when attention writes raster O)."""
        lpt = 2 if self.flags & 1 else 1
        gather = 1 if self.demand.kg is not None else 0
        scores = (2 if self.est == EST_LOWRANK else 1) if self.fused else 2
        place = 2 if self.owner is not None else 0
        bal = (1 if self.migrations is not None else 0) + (14 if self.augment else 0)
        # projection, two score products, gradient products, loss (partials, sum), weight gradients
        pred = 7 if self.predictor_lr is not None else 0
        return 3 + scores + pred + 3 + bal + place + 4 + gather + lpt + 1 + (0 if self.raster_out else 1)

    def kernels_per_backward(self) -> int:
        """reorder dO, rowdot, CSR transpose, schedule, dQ, schedule, dK + dV (one
        kernel, two with BWD_SPLIT_KV), 3 inverse reorders (none when the
        backward writes raster gradients)."""
        lpt = 2 if self.flags & 1 else 1
        kv = 2 if self.flags & 4 else 1
        return 1 + 1 + 1 + lpt + 1 + lpt + kv + (0 if self.raster_out else 3)

    def __init__(self, shape: Shape, estimator: str, top_p: float, k_floor: int, P: int, rank: int = 16,
                 gather: bool = True, flags: int = 0, backward: bool = False, device="cuda",
                 fused_estimation: bool = True, placement: bool = False, migrations: int | None = None,
                 augment: bool = False, predictor_lr: float | None = None, overlap_demand: bool = True,
                 raster_inputs: bool = False):
        """overlap_demand: after the KV demand lists (bitmap, offsets, indices),
        run the demand gather on a low-priority side stream while attention runs
        on a high-priority one; the two only read the same K/V, and the
        gather's CTAs (no shared memory) fit beside the persistent attention
        CTAs. forward() returns after both on the caller's stream. migrations: balance heads over P virtual ranks with at most this many
        migrations (None: no balancing). augment: fill each rank's slack with
        extra blocks (on the balanced ranks, or the contiguous head split);
        attention then runs on the augmented CSR. predictor_lr: with the
        low-rank estimator, after the scores are taken, one fitting step of the
        predictor weights (updated in place) against the real block scores.
        raster_inputs (forward-only, tcgen05 shapes, fused estimation): no
        reorder pass; the tile means come from a pooling read of raster Q and
        K, and the demand gather and attention read the raster tensors
        themselves (each block one 5-D TMA box), so forward()'s inputs stay
        in use until attention and the gather have finished."""
        self.shape, self.top_p, self.k_floor, self.P, self.rank, self.flags = shape, top_p, k_floor, P, rank, flags
        self.est = EST_LOWRANK if estimator == "lowrank" else EST_MEAN
        self.fused = fused_estimation
        s = shape
        dt = s.torch_dtype
        dev = torch.device(device)
        blocked = (s.B, s.H, s.N, s.d)
        self.raster_in = raster_inputs
        self.qb = self.kb = self.vb = None
        if not raster_inputs:
            self.qb, self.kb, self.vb = (torch.empty(blocked, dtype=dt, device=dev) for _ in range(3))
        self.o = torch.empty((s.B, s.N, s.H, s.d), dtype=dt, device=dev)
        self.lse = torch.empty((s.B, s.H, s.N), dtype=torch.float32, device=dev)
        self.scores = torch.empty((s.B, s.H, s.nb, s.nb), dtype=torch.float32, device=dev)
        self.ws_scores = torch.empty(max(block_scores_workspace_size(s, self.est, rank), 16), dtype=torch.uint8,
                                     device=dev)
        self.qmeans, self.kmeans = (torch.empty((s.B, s.H, s.nb, s.d), dtype=torch.float32, device=dev)
                                    for _ in range(2))
        import ctypes
        n = lib().sparsp_block_scores_pooled_workspace_size(ctypes.byref(s), self.est, rank)
        self.ws_pooled = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
        self.row_ptr = torch.empty(s.rows + 1, dtype=torch.int32, device=dev)
        self.col_idx = torch.empty(s.rows * s.nb, dtype=torch.int32, device=dev)
        self.ws_sel = torch.empty(max(select_workspace_size(s), 16), dtype=torch.uint8, device=dev)
        W = (s.nb + 31) // 32
        parts = s.B * s.H * P
        kg = vg = None
        if gather:
            kg = torch.empty((parts * s.nb, s.Bt, s.d), dtype=dt, device=dev)
            vg = torch.empty_like(kg)
        self.demand = DemandOut(torch.empty((s.B, s.H, P, W), dtype=torch.int32, device=dev),
                                torch.empty(parts + 1, dtype=torch.int32, device=dev),
                                torch.empty(parts * s.nb, dtype=torch.int32, device=dev), kg, vg,
                                torch.empty(4, dtype=torch.int64, device=dev))
        self.migrations, self.augment = migrations, augment
        self.predictor_lr = predictor_lr
        if predictor_lr is not None:
            if self.est != EST_LOWRANK or not fused_estimation:
                raise ValueError("predictor fitting needs the low-rank estimator with fused estimation")
            self.predictor_loss = torch.empty(s.H, dtype=torch.float32, device=dev)
            self.gwq, self.gwk = (torch.empty((s.H, s.d, rank), dtype=torch.float32, device=dev) for _ in range(2))
            self.ws_pred = torch.empty(max(lib().sparsp_predictor_workspace_size(ctypes.byref(s), rank), 16),
                                       dtype=torch.uint8, device=dev)
        # the tcgen05 forward takes O straight into raster order (64-token blocks with
        # d = 128 beyond 1,024 blocks run the portable kernel, which writes block
        # order only); the tcgen05 backward (the same shapes) also reads raster O
        # and writes raster dQ, dK, dV
        fwd_raster = (s.torch_dtype == torch.bfloat16 and not (flags & 2) and s.Bt in (64, 128)
                      and s.d in (64, 128) and not (s.Bt == 64 and s.d == 128 and s.nb > 1024))
        self.raster_out = fwd_raster
        if raster_inputs and (backward or not fwd_raster or not fused_estimation):
            raise ValueError("raster inputs need a forward-only step on the tcgen05 kernel with fused estimation")
        # the stage after which forward()'s raster inputs are no longer read
        self.inputs_read_mark = ("overlap" if overlap_demand and gather else "attn_fwd") if raster_inputs \
            else "reorder"
        self._o_fwd = None   # the buffer forward() last wrote O to (read by backward() when raster)
        # block-order O (and gradients) only where attention does not write raster rows
        self.ob = None if self.raster_out else torch.empty(blocked, dtype=dt, device=dev)
        self.overlap_demand = overlap_demand
        if overlap_demand:
            lo, hi = torch.cuda.Stream.priority_range()   # least, greatest
            self._attn_stream = torch.cuda.Stream(device=dev, priority=hi)
            self._demand_stream = torch.cuda.Stream(device=dev, priority=lo)
            self._selected = torch.cuda.Event()
        self.balance = None
        if migrations is not None or augment:
            if migrations is None:
                self.migrations = 0
            self.balance = Balance(
                torch.empty((s.B, s.H), dtype=torch.int32, device=dev),
                torch.empty((s.B, 2, P), dtype=torch.int64, device=dev),
                torch.empty(max(s.B, 4), dtype=torch.int32, device=dev))
        if augment:
            self.row_ptr_aug = torch.empty(s.rows + 1, dtype=torch.int32, device=dev)
            self.col_idx_aug = torch.empty(s.rows * s.nb, dtype=torch.int32, device=dev)
            self.added = torch.empty((s.B, P), dtype=torch.int64, device=dev)
            self.ws_aug = torch.empty(max(augment_workspace_size(s, P), 16), dtype=torch.uint8, device=dev)
        self.csr = (self.row_ptr, self.col_idx)
        self.owner = self.ws_place = None
        if placement:
            self.owner = torch.empty((s.B, s.nb), dtype=torch.int32, device=dev)
            self.ws_place = torch.empty(max(placement_workspace_size(s), 16), dtype=torch.uint8, device=dev)
        self.ws_attn = torch.empty(max(attn_workspace_size(s, backward), 16), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.prof = torch.zeros(PROF_SLOTS, dtype=torch.int64, device=dev)
        if backward:
            self.dob = torch.empty(blocked, dtype=dt, device=dev)
            self.dqb = self.dkb = self.dvb = None
            if not self.raster_out:
                self.dqb, self.dkb, self.dvb = (torch.empty(blocked, dtype=dt, device=dev) for _ in range(3))
            self.dq, self.dk, self.dv = (torch.empty((s.B, s.N, s.H, s.d), dtype=dt, device=dev)
                                         for _ in range(3))

    def forward(self, q, k, v, wq=None, wk=None, prof: bool = False, mark=None, out=None, before=None):
        """mark: optional callable(stage_name, stream=None) invoked after each
        stage is enqueued (used to record CUDA events; stream None is the
        current stream). With overlap_demand the overlapped stages are marked on
        their own streams, each preceded by a "<stage>:begin" mark, and the
        region they share by "overlap". out: optional raster output buffer
        (default: self.o). before: optional callable(name) invoked just before
        input "q", "k" or "v" is first read (e.g. to wait for its copy)."""
        s = self.shape
        mark = mark or (lambda name, stream=None: None)
        before = before or (lambda name: None)
        if self.raster_in:   # the tile means alone: attention and the gather read the raster tensors
            before("q")
            pool_means(s, q, self.qmeans)
            before("k")
            pool_means(s, k, self.kmeans)
            mark("reorder")
            block_scores_pooled(s, self.qmeans, self.kmeans, self.est, wq, wk, self.rank, out=self.scores,
                                ws=self.ws_pooled)
        elif self.fused:   # the tile means come out of the reorder pass itself
            before("q")
            reorder_pool(s, q, self.qb, self.qmeans)
            before("k")
            reorder_pool(s, k, self.kb, self.kmeans)
            before("v")
            reorder(s, v, self.vb)
            mark("reorder")
            block_scores_pooled(s, self.qmeans, self.kmeans, self.est, wq, wk, self.rank, out=self.scores,
                                ws=self.ws_pooled)
        else:
            before("q")
            reorder(s, q, self.qb)
            before("k")
            reorder(s, k, self.kb)
            before("v")
            reorder(s, v, self.vb)
            mark("reorder")
            block_scores(s, self.qb, self.kb, self.est, wq, wk, self.rank, out=self.scores, ws=self.ws_scores)
        mark("scores")
        if self.predictor_lr is not None:
            predictor_fit(s, self.qmeans, self.kmeans, wq, wk, self.predictor_lr, self.rank, self.predictor_loss,
                          self.gwq, self.gwk, self.ws_pred)
            mark("predictor")
        select(s, self.scores, self.top_p, self.k_floor, self.row_ptr, self.col_idx, self.ws_sel, self.status)
        mark("select")
        rp, ci = self.row_ptr, self.col_idx
        if self.balance is not None:
            balance_heads(s, self.P, self.row_ptr, self.migrations, out=self.balance)
            mark("balance")
        if self.augment:
            rp, ci, _ = augment(s, self.P, self.scores, self.row_ptr, self.col_idx, self.balance.head_rank,
                                self.row_ptr_aug, self.col_idx_aug, self.added, self.ws_aug, self.status)
            mark("augment")
        self.csr = (rp, ci)
        if self.owner is not None:
            placement(s, self.P, rp, ci, self.owner, self.ws_place, self.status)
            mark("placement")
        o = self.o if out is None else out
        # attention output: raster O directly, or block order and an inverse reorder
        o_attn, aflags = (o, self.flags | OUT_RASTER) if self.raster_out else (self.ob, self.flags)
        if self.raster_in:
            before("v")
            aq, ak, av, aflags = q, k, v, aflags | IN_RASTER
        else:
            aq, ak, av = self.qb, self.kb, self.vb
        if self.overlap_demand and self.demand.kg is not None:
            # the lists (bitmap, offsets, indices) first, on this stream: they need a
            # little shared memory, which attention leaves none of; then the gather
            # (no shared memory) beside attention
            main = torch.cuda.current_stream()
            lists = dataclasses.replace(self.demand, kg=None, vg=None)
            kv_demand(s, self.P, rp, ci, out=lists, status=self.status, owner=self.owner)
            mark("kv_demand")
            hi, lo = self._attn_stream, self._demand_stream
            mark("overlap:begin")
            self._selected.record(main)
            hi.wait_event(self._selected)
            lo.wait_event(self._selected)
            with torch.cuda.stream(hi):   # enqueued first: the persistent CTAs take their SMs first
                mark("attn_fwd:begin", hi)
                attn_fwd(s, aq, ak, av, rp, ci, 0.0, o_attn, self.lse, self.ws_attn,
                         aflags, self.prof if prof else None, self.status, stream=hi)
                mark("attn_fwd", hi)
            with torch.cuda.stream(lo):
                mark("kv_gather:begin", lo)
                kv_gather(s, self.P, self.demand, ak, av, status=self.status, stream=lo, raster=self.raster_in)
                mark("kv_gather", lo)
            main.wait_stream(hi)
            main.wait_stream(lo)
            mark("overlap")
        else:
            if self.raster_in and self.demand.kg is not None:
                lists = dataclasses.replace(self.demand, kg=None, vg=None)
                kv_demand(s, self.P, rp, ci, out=lists, status=self.status, owner=self.owner)
                kv_gather(s, self.P, self.demand, ak, av, status=self.status, raster=True)
            else:
                kv_demand(s, self.P, rp, ci, self.kb, self.vb, out=self.demand, status=self.status,
                          owner=self.owner)
            mark("kv_demand")
            attn_fwd(s, aq, ak, av, rp, ci, 0.0, o_attn, self.lse, self.ws_attn,
                     aflags, self.prof if prof else None, self.status)
            mark("attn_fwd")
        if not self.raster_out:
            reorder(s, self.ob, o, inverse=True)
            mark("reorder_out")
        self._o_fwd = o
        return o, self.lse

    def backward(self, dout, prof: bool = False, mark=None, outs=None, before=None):
        """outs: optional raster (dQ, dK, dV) output buffers (default: self.dq, self.dk, self.dv);
        before: optional callable("do") invoked just before dout is first read.
        With raster_out the backward reads O from the buffer the last forward()
        wrote it to, which must still hold it, and writes the gradients' raster
        rows itself."""
        s = self.shape
        mark = mark or (lambda name: None)
        if before is not None:   # e.g. to wait for dout's copy
            before("do")
        reorder(s, dout, self.dob)
        mark("reorder_dout")
        rp, ci = self.csr
        dq, dk, dv = (self.dq, self.dk, self.dv) if outs is None else outs
        if self.raster_out:
            if self._o_fwd is None:
                raise RuntimeError("backward() needs a forward() first")
            attn_bwd(s, self.qb, self.kb, self.vb, self._o_fwd, self.lse, self.dob, rp, ci, 0.0, dq, dk, dv,
                     self.ws_attn, self.flags | OUT_RASTER, self.prof if prof else None, self.status)
            mark("attn_bwd")
            return dq, dk, dv
        attn_bwd(s, self.qb, self.kb, self.vb, self.ob, self.lse, self.dob, rp, ci, 0.0,
                 self.dqb, self.dkb, self.dvb, self.ws_attn, self.flags, self.prof if prof else None, self.status)
        mark("attn_bwd")
        reorder(s, self.dqb, dq, inverse=True)
        reorder(s, self.dkb, dk, inverse=True)
        reorder(s, self.dvb, dv, inverse=True)
        mark("reorder_grads")
        return dq, dk, dv

    def capture(self, q, k, v, wq=None, wk=None, dout=None) -> "GraphedStep":
        """A CUDA graph of one step on these device buffers: forward(q, k, v),
        and backward(dout) too when dout is given. replay() reruns the whole
        step with one launch on whatever the buffers hold at that moment (the
        caller refills them in place) and returns what the step returns. The
        step runs once eagerly on a side stream first, as graph capture wants;
        the buffers stay bound to the graph. The captured step runs the KV
        demand gather before attention on one stream: a graph does not keep the
        side streams' priorities, without which the gather beside attention
        takes the SMs attention needs."""
        def step():
            out = self.forward(q, k, v, wq=wq, wk=wk)
            return out if dout is None else out + self.backward(dout)
        overlap, self.overlap_demand = self.overlap_demand, False
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                step()
            torch.cuda.current_stream().wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                outs = step()
        finally:
            self.overlap_demand = overlap
        return GraphedStep(graph, outs)


class GraphedStep:
    """A captured Pipeline step (Pipeline.capture)."""

    def __init__(self, graph, outs):
        self.graph = graph
        self.outs = outs

    def replay(self):
        """Runs the step on the current stream; returns the step's outputs
        (O, LSE[, dQ, dK, dV]) in the buffers the capture bound."""
        self.graph.replay()
        return self.outs

