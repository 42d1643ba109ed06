#!/usr/bin/env python3
"""Benchmark of the whole block-sparse attention hot path on GB300.

One step = reorder Q, K, V into video tiles -> mean-pooled (or low-rank) block
scores -> Top-p/Top-k selection into a per-head CSR -> KV demand of P query
partitions with the gather -> block-sparse attention forward (and, for the
training workload, the backward) -> outputs back to raster order.

Default workload: the Wan-14B attention-layer shape (B=1, H=40, d=128,
30,720 tokens in 2x8x8 tiles, Top-p 0.95, floor 8, P = 8), bf16, synthetic
seeded inputs. Prints one JSON line (rank 0). On one GPU the line also
carries a compact "workloads" object with the other four seeded workloads
(skewed per-head sparsity, the 65,536-token training step, the medium and
the tiny case), each timed over its own short run.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload wan|skewed|training|medium|tiny]
  python bench.py --impl reference ...   # the CPU oracle on the host cores, same metric
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "block-sparse attn effective TFLOP/s at 32K video tokens; % of bf16 TC peak"
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def stage_times(marks, side, elapsed, steps):
    """Per-step stage times (ms) from [(name, event)] in enqueue order. A stage
    runs from its "<name>:begin" mark if it has one (a stage overlapped on its
    own stream), else from the mark before it; marks of the names in `side`
    (recorded on side streams) do not start the next stage. elapsed(a, b) is
    the time from event a to event b; "step_start" opens each step."""
    out = {}
    prev = None
    begins = {}
    for name, ev in marks:
        if name.endswith(":begin"):
            begins[name[:-len(":begin")]] = ev
            continue
        if name != "step_start":
            first = begins.pop(name, prev)
            out[name] = out.get(name, 0.0) + elapsed(first, ev)
        if name not in side:
            prev = ev
    return {k: v / steps for k, v in out.items()}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


L2_BYTES = 129e6          # GB300 L2; a stage whose bytes fit was fed from L2, not HBM
# fp32 FFMA peak, derived (not measured): 152 SMs x 128 fp32 lanes x 2 flop per FMA x 2,070 MHz
FP32_FFMA_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12
EXTRA_WORKLOADS = ("skewed", "training", "medium", "tiny")

# DRAM bytes (read + write) per launch of the tcgen05 forward kernel, from an ncu capture of the
# Wan-layer shape with 8 of its 40 heads (237.3 MB: Q, K, V read once, O written), scaled by the
# heads a full launch processes; the traffic grows with the heads, each head's tiles being
# independent. The algorithmic bytes are Q + K + V + O + LSE = 1,263 MB.
ATTN_TRAFFIC = {"wan14b-layer-30k-bf16": 237.3e6 * 40 / 8}


def attn_flops(nnz: int, wl) -> float:
    """Algorithmic forward flops over the selected blocks: QK^T and PV, 2 flops per MAC."""
    return 4.0 * nnz * wl.Bt * wl.Bt * wl.d


def bwd_flops(nnz: int, wl) -> float:
    """FlashAttention convention for the backward: 2.5x the forward (recompute counted)."""
    return 10.0 * nnz * wl.Bt * wl.Bt * wl.d


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names[1:], parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def cpu_baseline(wl, data, budget_s: float = 12.0) -> dict:
    """The oracle, as it stands, on a bounded sample of the same workload: the
    whole forward chain for head 0 (reorder, scores, selection, demand) and
    attention for that head's query blocks in longest-first order until the
    time budget is spent. Value = attention flops done / total time."""
    from oracle import sparsp_oracle as orc
    g = orc.grid_of(wl)
    g1 = orc.Grid(1, 1, g.T, g.Y, g.X, g.d, g.ta, g.tb, g.tc)
    sub = {x: np.ascontiguousarray(data[x][:1, :, :1, :]) for x in ("q", "k", "v")}
    t0 = time.perf_counter()
    qb, kb, vb = (orc.reorder(sub[x], g1) for x in ("q", "k", "v"))
    if wl.estimator == "lowrank":
        S = orc.scores_lowrank(qb, kb, data["wq"][:1], data["wk"][:1], g.Bt)
    else:
        S = orc.scores_mean(qb, kb, g.Bt)
    sel = orc.select(S.astype(np.float32).reshape(-1, g.nb), wl.top_p, wl.k_floor)
    orc.kv_demand(sel.row_ptr, sel.col_idx, 1, 1, g.nb, wl.P, g.Bt, g.d, wl.elem_bytes, kb, vb)
    order = orc.lpt_order(sel.row_ptr, 1, 1, g.nb)
    flops = 0.0
    done = 0
    scale = 1.0 / math.sqrt(g.d)
    for it in order:
        orc.attn_fwd_row(qb, kb, vb, sel.row_ptr, sel.col_idx, g.Bt, scale, 0, 0, int(it))
        flops += attn_flops(int(sel.row_ptr[it + 1] - sel.row_ptr[it]), wl)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    threads = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            threads = max(int(x.get("num_threads", 1)) for x in info)
    except Exception:
        pass
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"head 0 of {wl.name}: reorder, scores, selection, demand+gather, then attention for "
                      f"{done}/{g.nb} query blocks in longest-first order; {dt:.1f} s",
            "seconds": dt}


def static_config(wl) -> dict:
    """The workload's own keys, shared by both arms' config."""
    return {"workload": wl.name, "B": wl.B, "H": wl.H, "N": wl.N, "d": wl.d, "tile": [wl.ta, wl.tb, wl.tc],
            "nb": wl.nb, "estimator": wl.estimator, "top_p": wl.top_p, "k_floor": wl.k_floor, "P": wl.P,
            "backward": wl.backward}


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    data = synth.make(wl)
    per_step = []
    cb = None
    for _ in range(args.warmup + args.steps):
        cb = cpu_baseline(wl, data, budget_s=max(2.0, min(20.0, 150.0 / max(1, args.warmup + args.steps))))
        per_step.append(cb)
    timed = per_step[args.warmup:]
    val = statistics.median(x["value"] for x in timed)
    secs = sum(x["seconds"] for x in timed)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / len(timed),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {**static_config(wl), "parallelism": "host cores"},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cb["cores"], "kind": "oracle",
                             "sample": cb["sample"]},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def stage_bytes(shape, wl, nnz: int, demanded: int, fused: bool, overlapped: bool) -> dict:
    """Algorithmic HBM bytes of the memory-bound stages of one step: what each
    stage must read and write at least (the roofline's numerator)."""
    el = 2 if wl.dtype == "bf16" else 4
    BH = shape.B * shape.H
    tensor = BH * shape.N * shape.d * el
    means = BH * shape.nb * shape.d * 4
    rows = BH * shape.nb
    out = {
        "reorder": 6 * tensor + (2 * means if fused else 0),
        "scores": (2 * means if fused else 2 * tensor) + 4 * BH * shape.nb * shape.nb,
        "select": 4 * BH * shape.nb * shape.nb + 4 * (nnz + rows + 1),
        "reorder_out": 2 * tensor,
    }
    # demand lists: the CSR read, the bitmap and the index lists written; the gather: the
    # gathered copy written once, each source K/V tile read from HBM once (its P-fold reuse
    # across partitions hits in L2)
    lists = 4 * nnz + BH * wl.P * ((shape.nb + 31) // 32) * 4 + 4 * (demanded // (2 * shape.Bt * shape.d * el))
    gather = demanded + 2 * tensor
    if overlapped:
        out["kv_demand"] = lists
        out["kv_gather"] = gather
    else:
        out["kv_demand"] = lists + gather
    return out


def hbm_fractions(stage_ms: dict, nbytes: dict, hbm_gbs: float) -> dict:
    """GB/s of each memory-bound stage against the measured copy peak. A stage
    whose bytes fit in L2 (its inputs were written just before by the previous
    stage) is fed from L2: it gets its GB/s but no fraction of the HBM peak."""
    out = {}
    for name, b in nbytes.items():
        ms = stage_ms.get(name)
        if not ms or ms <= 0:
            continue
        gbs = b / (ms * 1e-3) / 1e9
        if b <= L2_BYTES:
            out[name] = {"bytes": int(b), "gbs": gbs, "frac": None, "l2_resident": True}
        else:
            out[name] = {"bytes": int(b), "gbs": gbs, "frac": gbs / hbm_gbs}
    return out


class Run:
    """One workload on the device: inputs resident in HBM, a Pipeline in the
    benchmark's configuration, and timed steps."""

    def __init__(self, sp, wl, args, flags=0, overlap=True):
        import torch
        self.torch, self.sp, self.wl = torch, sp, wl
        self.data = synth.make(wl)
        self.shape = sp.shape_of(wl)
        self.pipe = sp.Pipeline(self.shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, backward=wl.backward,
                                flags=flags, fused_estimation=not args.unfused, placement=args.placement,
                                migrations=wl.P if args.augment else None, augment=args.augment,
                                overlap_demand=overlap,
                                raster_inputs=getattr(args, "raster_inputs", False) and not wl.backward)
        tdt = self.shape.torch_dtype
        self.host_in = {x: torch.from_numpy(self.data[x]).to(tdt).pin_memory() for x in ("q", "k", "v")}
        self.dev_in = {x: self.host_in[x].cuda() for x in self.host_in}
        self.kw = {}
        if wl.estimator == "lowrank":
            self.kw = {"wq": torch.from_numpy(self.data["wq"]).cuda(), "wk": torch.from_numpy(self.data["wk"]).cuda()}
        self.dout = None
        if wl.backward:
            self.host_in["do"] = torch.from_numpy(self.data["do"]).to(tdt).pin_memory()
            self.dout = self.host_in["do"].cuda()
        self.stream = torch.cuda.current_stream()

    def step(self, mark=None, prof=False):
        self.pipe.forward(self.dev_in["q"], self.dev_in["k"], self.dev_in["v"], prof=prof, mark=mark, **self.kw)
        if self.wl.backward:
            self.pipe.backward(self.dout, prof=prof, mark=mark)

    def warm(self, n):
        for _ in range(n):
            self.step()
        self.torch.cuda.synchronize()
        st = self.pipe.status.item()
        if st != 0:
            raise SystemExit(f"{self.wl.name}: device status {self.sp.status_string(st)}")
        self.nnz = int(self.pipe.csr[0][-1].item())     # the CSR attention ran on
        self.kv_bytes = [int(x) for x in self.pipe.demand.bytes.tolist()]

    def timed(self, steps, before=None):
        """K steps between two events on the launching stream, with an event
        after every stage; returns (ms per step, {stage: ms per step})."""
        torch = self.torch
        marks = []

        def mark(name, on=None):
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(on if on is not None else self.stream)
            marks.append((name, ev))

        if before is not None:
            before()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(self.stream)
        for _ in range(steps):
            mark("step_start")
            self.step(mark=mark)
        end.record(self.stream)
        torch.cuda.synchronize()
        side = ("attn_fwd", "kv_gather") if self.pipe.overlap_demand else ()
        return start.elapsed_time(end) / steps, stage_times(marks, side, lambda a, b: a.elapsed_time(b), steps)

    def graph_ms(self, steps):
        """The same step captured as one CUDA graph (Pipeline.capture) and
        replayed: ms per step, with the host's per-kernel launches gone."""
        torch = self.torch
        graphed = self.pipe.capture(self.dev_in["q"], self.dev_in["k"], self.dev_in["v"],
                                    dout=self.dout if self.wl.backward else None, **self.kw)
        for _ in range(3):
            graphed.replay()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(self.stream)
        for _ in range(steps):
            graphed.replay()
        end.record(self.stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / steps

    def attn_alone_ms(self, calls=5):
        """The forward attention kernel with nothing beside it (in the step it
        may share its SMs with the KV gather)."""
        torch, sp, pipe = self.torch, self.sp, self.pipe
        rp, ci = pipe.csr
        flags = pipe.flags | (sp.OUT_RASTER if pipe.raster_out else 0)
        o = pipe.o if pipe.raster_out else pipe.ob
        q, k, v = pipe.qb, pipe.kb, pipe.vb
        if pipe.raster_in:
            q, k, v, flags = self.dev_in["q"], self.dev_in["k"], self.dev_in["v"], flags | sp.IN_RASTER
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        b0.record(self.stream)
        for _ in range(calls):
            sp.attn_fwd(self.shape, q, k, v, rp, ci, 0.0, o, pipe.lse, pipe.ws_attn, flags, None, pipe.status)
        b1.record(self.stream)
        torch.cuda.synchronize()
        return b0.elapsed_time(b1) / calls

    def sm_imbalance(self):
        """Per-SM busy time of the attention kernel, max over mean (one profiled step)."""
        torch = self.torch
        self.pipe.prof.zero_()
        self.pipe.forward(self.dev_in["q"], self.dev_in["k"], self.dev_in["v"], prof=True, **self.kw)
        torch.cuda.synchronize()
        busy = self.pipe.prof.cpu().numpy().astype(np.float64)
        busy = busy[busy > 0]
        return float(busy.max() / busy.mean()) if len(busy) else None


def end_to_end(sp, run, steps, work, world=1, barrier=None, replicas=None) -> dict:
    """The same steps through sp.HostPipeline: every step copies its inputs in
    from pinned host memory and its outputs (O; and dQ, dK, dV with a
    backward) back, overlapped with the neighbouring steps' kernels. The timed
    window includes the first step's uncovered input copy and the last step's
    output copy."""
    import torch
    wl, pipe, host_in, kw = run.wl, run.pipe, run.host_in, run.kw
    tdt = run.shape.torch_dtype
    host_out = torch.empty(pipe.o.shape, dtype=tdt).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out.numel() * host_out.element_size()
    if wl.backward:
        host_grads = [torch.empty(pipe.o.shape, dtype=tdt).pin_memory() for _ in range(3)]
        d2h += 3 * host_out.numel() * host_out.element_size()
    hp = sp.HostPipeline(pipe)
    if wl.backward:
        def e2e_step():
            hp.train_step(host_in["q"], host_in["k"], host_in["v"], host_in["do"], host_out, *host_grads, **kw)
    else:
        def e2e_step():
            hp.step(host_in["q"], host_in["k"], host_in["v"], host_out, **kw)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    if barrier is not None:
        barrier()
    stream = run.stream
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        e2e_step()
    stream.wait_stream(hp.d2h)         # the last result has reached the host
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    if replicas is not None:
        ms = replicas.max_over_ranks(ms)
    rate = (replicas.whole_job_rate(work, ms, world) if replicas is not None else work / (ms * 1e-3)) / 1e12
    return {"value": rate, "unit": "TFLOP/s", "ms_per_step": ms, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "copies": "overlapped with neighbouring steps (HostPipeline)"}


def workload_summary(sp, name, args, pk) -> dict:
    """One of the other seeded workloads, in the default configuration: its own
    short timed run (3 warm-ups, min(K, 10) steps), no CPU baseline."""
    import torch
    wl = synth.WORKLOADS[name]
    run = Run(sp, wl, args)
    run.warm(3)
    ms, st = run.timed(min(args.steps, 10))
    shape = run.shape
    f_fwd = attn_flops(run.nnz, wl)
    f_step = f_fwd + (bwd_flops(run.nnz, wl) if wl.backward else 0.0)
    alone = run.attn_alone_ms()
    tensor = wl.dtype == "bf16"
    peak = pk["bf16_tflops"]
    out = {"workload": wl.name, "ms_per_step": ms, "tflops": f_step / (ms * 1e-3) / 1e12,
           "tokens_per_s": wl.B * wl.N / (ms * 1e-3), "nnz_blocks": run.nnz,
           "density": run.nnz / (shape.rows * shape.nb),
           "attn_fwd_ms": st["attn_fwd"], "attn_fwd_tflops": f_fwd / (st["attn_fwd"] * 1e-3) / 1e12,
           "attn_fwd_alone_ms": alone, "attn_fwd_alone_tflops": f_fwd / (alone * 1e-3) / 1e12}
    if tensor:
        out["attn_fwd_frac_of_burst"] = out["attn_fwd_tflops"] / peak
        out["attn_fwd_alone_frac_of_burst"] = out["attn_fwd_alone_tflops"] / peak
    else:
        out["attn_fwd_bound"] = "alu (fp32 FFMA kernel; peak derived: 152 SMs x 128 lanes x 2 x 2,070 MHz)"
        out["attn_fwd_frac_of_fp32_peak"] = out["attn_fwd_tflops"] / FP32_FFMA_TFLOPS
        out["attn_fwd_alone_frac_of_fp32_peak"] = out["attn_fwd_alone_tflops"] / FP32_FFMA_TFLOPS
    if wl.backward:
        fb = bwd_flops(run.nnz, wl)
        out["attn_bwd_ms"] = st["attn_bwd"]
        out["attn_bwd_tflops"] = fb / (st["attn_bwd"] * 1e-3) / 1e12
        out["attn_bwd_frac_of_burst"] = out["attn_bwd_tflops"] / peak
    nbytes = stage_bytes(shape, wl, run.nnz, run.kv_bytes[0], not args.unfused, run.pipe.overlap_demand)
    out["hbm_stages"] = {k: (round(v["frac"], 4) if v["frac"] is not None else "l2-resident")
                         for k, v in hbm_fractions(st, nbytes, pk["hbm_gbs"]).items()}
    out["stages_ms"] = {k: round(v, 5) for k, v in st.items()}
    if wl.skew:
        out["attn_sm_imbalance"] = run.sm_imbalance()
    gms = run.graph_ms(min(args.steps, 10))
    out["graph_ms_per_step"] = gms
    out["graph_tflops"] = f_step / (gms * 1e-3) / 1e12
    if not args.no_e2e:
        e = end_to_end(sp, run, min(args.steps, 10), f_step)
        out["e2e_ms_per_step"] = e["ms_per_step"]
        out["e2e_tflops"] = e["value"]
        out["e2e_copies_gb_per_step"] = [round(e["h2d_bytes_per_step"] / 1e9, 3), round(e["d2h_bytes_per_step"] / 1e9, 3)]
    del run
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="wan", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--flat", action="store_true", help="flat (cross-head) longest-first order")
    ap.add_argument("--portable", action="store_true", help="mma.sync attention kernel")
    ap.add_argument("--bwd-split-kv", action="store_true",
                    help="backward: dK and dV by two tcgen05 kernels instead of one")
    ap.add_argument("--unfused", action="store_true", help="separate pooling pass instead of reorder+pool")
    ap.add_argument("--placement", action="store_true",
                    help="dependency-aware block placement inside the step (default: contiguous partitions)")
    ap.add_argument("--augment", action="store_true",
                    help="head balancing over P virtual ranks + slack-aware augmentation inside the step")
    ap.add_argument("--serial-demand", action="store_true",
                    help="time the step with the KV demand stage before attention on one stream (default: the "
                         "gather beside attention on a side stream)")
    ap.add_argument("--raster-inputs", action="store_true",
                    help="forward-only steps: no reorder pass; pooling, the gather and attention read raster Q, K, V")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the other seeded workloads")
    ap.add_argument("--heads", type=int, default=0, help="override the head count (smaller profiling case)")
    ap.add_argument("--head-dim", type=int, default=0, choices=[0, 64, 128],
                    help="override the head dimension (profiling the d = 64 kernels on a workload's shape)")
    ap.add_argument("--tile-frames", type=int, default=0, choices=[0, 1, 2],
                    help="override the tile's frame count (1: 64-token blocks on a 2x8x8 workload)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wl = synth.WORKLOADS[args.workload]
    if args.heads or args.head_dim or args.tile_frames:
        import dataclasses
        if args.heads:
            wl = dataclasses.replace(wl, H=args.heads, name=f"{wl.name}-h{args.heads}")
        if args.head_dim:
            wl = dataclasses.replace(wl, d=args.head_dim, name=f"{wl.name}-d{args.head_dim}")
        if args.tile_frames:
            wl = dataclasses.replace(wl, ta=args.tile_frames, name=f"{wl.name}-ta{args.tile_frames}")
    if args.impl == "reference":
        return run_reference(args, wl)

    import torch
    import torch.distributed as dist

    import block_sparse_attention_token_gb300 as sp
    from block_sparse_attention_token_gb300 import replicas

    rank, local, world = replicas.rank_world()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    barrier = replicas.barrier
    flags = ((sp.SCHED_FLAT if args.flat else 0) | (sp.KERNEL_PORTABLE if args.portable else 0)
             | (sp.BWD_SPLIT_KV if args.bwd_split_kv else 0))
    run = Run(sp, wl, args, flags=flags, overlap=True)
    pipe, shape, stream = run.pipe, run.shape, run.stream
    run.warm(args.warmup)
    nnz = run.nnz
    demanded, all_bytes, remote_dem, remote_all = run.kv_bytes
    default_overlap = not args.serial_demand

    # ---- the other order of the KV demand gather, untimed warm-up then its own timed steps
    # (A/B in one process; the headline takes the default order)
    pipe.overlap_demand = not default_overlap
    run.warm(2)
    other_ms, other_stages = run.timed(args.steps)
    pipe.overlap_demand = default_overlap
    run.warm(2)

    # ---- timed region: K steps, events around every stage, clocks sampled meanwhile
    clocks = ClockSampler(local)
    time.sleep(0.5)
    ms_step, stage_ms = run.timed(args.steps, before=barrier)
    barrier()
    clk = clocks.stop()
    ms_step = replicas.max_over_ranks(ms_step)
    overlap_ms, serial_ms = (ms_step, other_ms) if default_overlap else (other_ms, ms_step)

    pk = peaks()
    f_fwd = attn_flops(nnz, wl)
    f_step = f_fwd + (bwd_flops(nnz, wl) if wl.backward else 0.0)
    value = replicas.whole_job_rate(f_step, ms_step, world) / 1e12
    attn_ms = stage_ms["attn_fwd"]
    achieved = f_fwd / (attn_ms * 1e-3) / 1e12
    if wl.dtype == "bf16":
        peak = pk["bf16_tflops"]
        roofline = {"bound": "tensor", "kernel": "attn_fwd", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "peak_kind": f"bf16 burst ({pk['source']}; the kernel runs at full "
                                                          f"clock inside a sub-second timed region)",
                    "frac_of_sustained": achieved / pk["bf16_tflops_sustained"]}
    else:
        peak = FP32_FFMA_TFLOPS
        roofline = {"bound": "alu", "kernel": "attn_fwd", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak,
                    "peak_kind": "fp32 FFMA, derived: 152 SMs x 128 lanes x 2 flop x 2,070 MHz"}
    roofline.update({"traffic": ATTN_TRAFFIC.get(wl.name) if not args.portable else None,
                     "work": f"4*nnz*Bt^2*d = {f_fwd:.4g} flop per launch (nnz={nnz})"})
    if wl.backward:
        roofline["bwd_achieved"] = bwd_flops(nnz, wl) / (stage_ms["attn_bwd"] * 1e-3) / 1e12
        roofline["bwd_frac"] = roofline["bwd_achieved"] / peak
    if not args.portable:
        alone = f_fwd / (run.attn_alone_ms() * 1e-3) / 1e12
        roofline["achieved_alone"] = alone
        roofline["frac_alone"] = alone / peak
        if default_overlap:
            roofline["in_step"] = "shares its SMs with the KV demand gather (side stream)"

    nbytes = stage_bytes(shape, wl, nnz, demanded, not args.unfused, default_overlap)
    hbm = hbm_fractions(stage_ms, nbytes, pk["hbm_gbs"])
    if "kv_gather" in hbm:
        hbm["kv_gather"]["note"] = "runs beside attention, sharing its SMs: not a standalone rate"
    other_bytes = stage_bytes(shape, wl, nnz, demanded, not args.unfused, not default_overlap)
    demand_order = {"overlapped_ms_per_step": overlap_ms, "serial_ms_per_step": serial_ms,
                    "default": "overlapped" if default_overlap else "serial",
                    ("serial" if default_overlap else "overlapped") + "_stages_ms": other_stages,
                    ("serial" if default_overlap else "overlapped") + "_hbm_stages":
                        hbm_fractions(other_stages, other_bytes, pk["hbm_gbs"])}

    # ---- end to end through the public API: pinned host -> device, step, O -> pinned host
    # (right after the device-timed steps, before the dense context line's heavy kernels)
    tdt = shape.torch_dtype
    e2e = None if args.no_e2e else end_to_end(sp, run, args.steps, f_step, world, barrier, replicas)

    # ---- context only: dense attention (PyTorch SDPA) over the same tensors
    BH = shape.B * shape.H
    dense = None
    try:
        import torch.nn.functional as F
        qd, kd, vd = pipe.qb, pipe.kb, pipe.vb
        for _ in range(2):
            F.scaled_dot_product_attention(qd, kd, vd)
        d0 = torch.cuda.Event(enable_timing=True)
        d1 = torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(3):
            F.scaled_dot_product_attention(qd, kd, vd)
        d1.record(stream)
        torch.cuda.synchronize()
        dms = d0.elapsed_time(d1) / 3
        dense = {"sdpa_ms": dms, "sdpa_tflops": 4.0 * BH * shape.N * shape.N * shape.d / (dms * 1e-3) / 1e12,
                 "sparse_attn_speedup": dms / stage_ms["attn_fwd"],
                 "kind": "torch SDPA, dense, same Q/K/V (a library baseline of unknown tuning: context only)"}
    except Exception as exc:   # context only: never fails the bench
        dense = {"unavailable": str(exc)[:120]}

    imbalance = run.sm_imbalance()

    # dependency-aware placement against the contiguous split on this step's CSR
    # (untimed by the step; its own kernels timed here)
    ws_pl = torch.empty(max(sp.placement_workspace_size(shape), 16), dtype=torch.uint8, device="cuda")
    owner = torch.empty((shape.B, shape.nb), dtype=torch.int32, device="cuda")
    contiguous = sp.kv_demand(shape, wl.P, pipe.row_ptr, pipe.col_idx)
    placed = sp.kv_demand(shape, wl.P, pipe.row_ptr, pipe.col_idx, owner=sp.placement(
        shape, wl.P, pipe.row_ptr, pipe.col_idx, owner, ws_pl))
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(5):
        sp.placement(shape, wl.P, pipe.row_ptr, pipe.col_idx, owner, ws_pl)
    p1.record(stream)
    torch.cuda.synchronize()
    cb, pb = contiguous.bytes.tolist(), placed.bytes.tolist()
    placement_info = {"remote_demanded_contiguous": int(cb[2]), "remote_demanded_placed": int(pb[2]),
                      "demanded_contiguous": int(cb[0]), "demanded_placed": int(pb[0]),
                      "remote_reduction": 1.0 - pb[2] / cb[2] if cb[2] else None,
                      "placement_ms": p0.elapsed_time(p1) / 5, "in_step": bool(args.placement)}

    # virtual-rank balancing and slack-aware augmentation on this step's selection
    # (ranks hold whole heads, so there are at most H of them)
    R = min(wl.P, shape.H)
    bal = sp.balance_heads(shape, R, pipe.row_ptr, R)
    bal0 = sp.balance_heads(shape, R, pipe.row_ptr, 0)
    ws_aug = torch.empty(max(sp.augment_workspace_size(shape, R), 16), dtype=torch.uint8, device="cuda")
    rp_aug = torch.empty(shape.rows + 1, dtype=torch.int32, device="cuda")
    ci_aug = torch.empty(shape.rows * shape.nb, dtype=torch.int32, device="cuda")
    added = torch.empty((shape.B, R), dtype=torch.int64, device="cuda")
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(5):
        sp.balance_heads(shape, R, pipe.row_ptr, R, out=bal)
        sp.augment(shape, R, pipe.scores, pipe.row_ptr, pipe.col_idx, bal.head_rank, rp_aug, ci_aug, added,
                   ws_aug)
    a1.record(stream)
    torch.cuda.synchronize()
    L = bal.loads.cpu().numpy()
    L0 = bal0.loads.cpu().numpy()

    def _imb(x):
        return float(x.max() * x.shape[-1] / x.sum()) if x.sum() else 1.0

    balance_info = {"ranks": R, "imbalance_contiguous": _imb(L0[0, 0]), "imbalance_balanced": _imb(L[0, 1]),
                    "migrations": int(bal.migrations[0].item()), "blocks_added": int(added.sum().item()),
                    "nnz_after_augment": int(rp_aug[-1].item()),
                    "balance_augment_ms": a0.elapsed_time(a1) / 5, "in_step": bool(args.augment)}

    # predictor fitting on this step's tile means (low-rank workloads), outside the step
    predictor_info = None
    if wl.estimator == "lowrank" and not args.unfused:
        kw = run.kw
        wq_f, wk_f = kw["wq"].clone(), kw["wk"].clone()
        ploss, _, _ = sp.predictor_fit(shape, pipe.qmeans, pipe.kmeans, wq_f, wk_f, lr=0.0)
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(5):
            sp.predictor_fit(shape, pipe.qmeans, pipe.kmeans, wq_f, wk_f, lr=1e-3)
        f1.record(stream)
        torch.cuda.synchronize()
        predictor_info = {"loss_mean": float(ploss.mean().item()), "fit_step_ms": f0.elapsed_time(f1) / 5}

    launches = args.steps * (pipe.kernels_per_forward() + (pipe.kernels_per_backward() if wl.backward else 0))
    counts = np.diff(pipe.csr[0].cpu().numpy())
    data = run.data
    del run, pipe, contiguous, placed, owner, ws_pl, ws_aug, rp_aug, ci_aug
    torch.cuda.empty_cache()

    # the other seeded workloads, each its own short run (one GPU only; rank 0 prints)
    workloads = None
    if world == 1 and not args.no_workloads and not args.heads:
        workloads = {}
        for name in EXTRA_WORKLOADS:
            if synth.WORKLOADS[name].name == wl.name:
                continue
            workloads[name] = workload_summary(sp, name, args, pk)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(wl, data)
        cpu.pop("seconds", None)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic",
        "pct_of_peak": 100.0 * value / world / peak,
        "tokens_per_s": world * wl.B * wl.N / (ms_step * 1e-3),
        "config": {**static_config(wl), "nnz_blocks": nnz, "density": nnz / (shape.rows * shape.nb),
                   "row_len_min_max": [int(counts.min()), int(counts.max())],
                   "schedule": "flat" if args.flat else "head-grouped longest-first",
                   **({"backward_kernels": "dQ; dK and dV split" if args.bwd_split_kv else "dQ; dK + dV fused"}
                      if wl.backward else {}),
                   "kernel": "portable mma.sync" if args.portable else "default",
                   "estimation": "separate pooling pass" if args.unfused else "fused with the reorder",
                   "partitions": "dependency-aware placement" if args.placement else "contiguous",
                   "augmentation": "balanced heads + slack fill" if args.augment else "none",
                   "kv_demand": "lists and gather serial, before attention" if not default_overlap else
                                "lists before attention; gather beside it on a low-priority side stream",
                   "l2": f"inputs larger than L2 ({shape.B * shape.H * shape.N * shape.d * 2 / 1e6:.0f} MB per tensor)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "stages_ms": stage_ms,
        "hbm_stages": hbm,
        "demand_order": demand_order,
        "dense_context": dense,
        "kv_bytes": {"demanded": demanded, "all": all_bytes, "remote_demanded": remote_dem,
                     "remote_all": remote_all},
        "placement": placement_info,
        "balance": balance_info,
        "predictor": predictor_info,
        "attn_sm_imbalance": imbalance,
        "workloads": workloads,
        "clocks": clk, "e2e": e2e, "gpu_launches": launches, "roofline": roofline, "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
