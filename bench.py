"""Benchmark: masked attention forward + backward on one GB300 per rank.

Workload (one step = the whole hot path once): the 32K causal-document
configuration, B=1, H=32, S=32768, d=128, bf16 Q/K/V/dO ~ N(0,1) seed 0,
documents U[256, 2048], scale 1/sqrt(d).  A step runs fm_fwd (bound summary,
tile classification, longest-first order, forward kernel) and fm_bwd (the
same analysis over k-tiles, D / LSE preprocessing, backward kernel, dQ
conversion) on inputs already resident in HBM.

Metric: effective fwd+bwd TFLOP/s counting only visible score entries:
14 * d * N_u per (batch, head), N_u = number of visible (row, key) pairs.

    python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (it is the baseline: there is no other implementation to run).
Under torchrun every rank runs its own replica of the workload (the heads of
independent problems; no data-path collective) and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = dict(name="suite_32k/causal_document", B=1, H=32, S=32768, d=128, mask="causal_document")
METRIC = "effective fwd+bwd TFLOP/s on visible score entries (causal-document mask, 32K, hd128)"


# Every (workload, mask) point of the metric, measured after the headline step:
# (name, B, H, S, d, masks, mask parameters).  The localised 64K point runs
# four simulated ranks, one after another, each with its local query rows
# (two chunks of 8192, dual-chunk order) against the full keys.
PER_MASK_POINTS = (
    ("sweep_4k", 4, 16, 4096, 128,
     ("full", "causal", "sliding_window", "causal_document", "prefix_lm"), {}),
    ("suite_32k", 1, 32, 32768, 128,
     ("causal", "sliding_window", "causal_document", "bidirectional_document", "prefix_lm",
      "prefix_document", "share_question", "causal_blockwise", "random_eviction",
      "global_sliding", "qk_sparse", "block_sparse"), {}),
    ("long_128k", 1, 8, 131072, 128, ("causal_document_window",), {"window": 8192}),
    ("localize_64k", 1, 16, 65536, 128, ("causal_document",), {}),
    ("long_128k_gqa", 1, 8, 131072, 128, ("causal_document_window",), {"window": 8192}),
    # packed variable-length batches of 16K tokens (sequence lengths drawn
    # U[512, 4096], the last one cut), hidden size 2048: the FlashAttention-2
    # page's benchmark shape, with d 128 and 64
    ("varlen_16k_d128", 1, 16, 16384, 128, ("varlen_causal", "varlen_full"), {}),
    ("varlen_16k_d64", 1, 32, 16384, 64, ("varlen_causal", "varlen_full"), {}),
)


def _point_bounds(fm, mask, B, S, params):
    """Bounds of one per-mask point: a named mask (fm_inputs), or a packed
    batch built through fm_varlen_bounds from seeded sequence lengths."""
    import numpy as np
    import torch

    from fm_inputs.tensors import mask_bounds
    if not mask.startswith("varlen_"):
        return mask_bounds(mask, B, S, device="cuda", **params)
    rng = np.random.default_rng(0)
    cu = [0]
    while cu[-1] < S:
        cu.append(min(S, cu[-1] + int(rng.integers(512, 4097))))
    return fm.varlen_bounds(torch.tensor(cu, dtype=torch.int32, device="cuda"),
                            causal=mask == "varlen_causal")
# points run with fewer K/V heads than query heads (grouped-query attention):
# the 128K workload's 8 query heads over 2 K/V heads
GQA_POINTS = {"long_128k_gqa": ("long_128k", 2)}


# GEMMs of 2 * d flop per visible entry in each attention kernel: the
# forward S and P V; the dK/dV pass S^T, dP^T, dV, dK; the dQ pass S, dP, dQ
# (S and dP are computed in both backward passes)
KERNEL_GEMMS = {"fwd_kernel": 2, "bwd_kv_kernel": 4, "bwd_dq_kernel": 3}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return j, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        sm = [float(r[1]) for r in self.rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            if len(r) >= 9:
                for n, v in zip(names, r[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _visible_entries(bounds_np, S, H):
    from oracle import masks as om  # exact integer count of the visible pairs (not timed)
    return om.visible_count_all(bounds_np, S, H)


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _config(W, n_vis: int, world: int) -> dict:
    """The workload as both arms report it."""
    return {"workload": W["name"], "B": W["B"], "H": W["H"], "S": W["S"], "d": W["d"],
            "mask": W["mask"], "visible_entries_per_rank": n_vis,
            "l2": "inputs larger than L2 (Q, K, V, dO 256 MiB each); no flush between steps",
            "parallelism": f"replicas x{world} (no collective on the data path)"}


def _max_over_ranks(ms: float, world: int, device) -> float:
    """Step time of the whole job: the slowest rank's (all ranks hold the
    result).  One rank: the time itself."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_value(flop_per_rank_step: float, ms: float, world: int) -> float:
    """Whole-job throughput in TFLOP/s: the work of all ranks in one step
    (each rank runs its own replica of the workload) over the step time."""
    return world * flop_per_rank_step / (ms * 1e-3) / 1e12


def run_ours(args):
    import torch
    import torch.distributed as dist

    import masked_attention_bound_gb300 as fm
    from fm_inputs.tensors import mask_bounds, qkv_do

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    W = dict(WORKLOAD)
    if args.heads:
        W["H"] = args.heads
    B, H, S, d = W["B"], W["H"], W["S"], W["d"]
    scale = d ** -0.5
    q, k, v, do = qkv_do(B, S, S, H, d, seed=0, device="cuda")
    bounds = mask_bounds(W["mask"], B, S, device="cuda")
    n_vis = _visible_entries(bounds.cpu().numpy(), S, H)
    flop_fwd, flop_bwd = 4.0 * d * n_vis, 10.0 * d * n_vis
    flop_step = flop_fwd + flop_bwd

    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    desc = fm.make_desc(q, k, v, o)
    # one step workspace: the mask analysis runs once per step, for both passes
    ws = fm.workspace(desc, fm.WS_STEP)
    stream = torch.cuda.current_stream()

    def step(st=None):
        st = stream if st is None else st
        fm.plan(q, k, bounds, ws=ws, for_bwd=fm.WS_STEP, stream=st)
        fm.forward(q, k, v, bounds, scale, o=o, lse=lse, ws=ws, stream=st, planned=True)
        fm.backward(q, k, v, o, lse, do, bounds, scale, dq=dq, dk=dk, dv=dv, ws=ws, stream=st,
                    planned=True)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fm.device_status(ws) != 0:
        raise RuntimeError("device status not OK after warm-up")

    def timed(run, n):
        """ms per call of run() over n calls, events on the launching stream,
        barrier and synchronize on both sides, max over ranks."""
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(n):
            run()
        ev1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        return _max_over_ranks(ev0.elapsed_time(ev1) / n, world, "cuda")

    # ---- timed regions: K steps each, inputs (1 GiB of Q/K/V/dO) larger
    # than L2.  The headline has no per-kernel events (they add about 2 % to
    # a step); the same K steps are then run with the library's per-kernel
    # events for the breakdown and the roofline, and replayed once more as a
    # CUDA graph of the step.
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms = timed(step, args.steps)
    fm.profile_enable(True)
    prof_ms = timed(step, args.steps)
    fm.profile_enable(False)
    prof = fm.profile_read()
    clk = clocks.stop()
    graph_ms = None
    if not args.no_graph:
        # captured on a side stream (capture needs a non-default stream),
        # replayed on the timing stream
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            step(side)
        stream.wait_stream(side)
        graph.replay()
        graph_ms = timed(graph.replay, args.steps)
    # the mask analysis alone (latency-bound kernels of a few MB): captured
    # once as a CUDA graph and replayed 100 times
    plan_ms = None
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        pgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(pgraph, stream=side):
            fm.plan(q, k, bounds, ws=ws, for_bwd=fm.WS_STEP, stream=side)
        stream.wait_stream(side)
        pgraph.replay()
        plan_ms = timed(pgraph.replay, 100)
    if fm.device_status(ws) != 0:
        raise RuntimeError("device status not OK after the timed steps")

    if args.no_e2e:
        e2e_ms, h2d, d2h = float("nan"), 0, 0
    else:
        e2e_ms, h2d, d2h = run_e2e(args, fm, q, k, v, do, bounds, scale, o, lse, dq, dk, dv,
                                   ws, stream, world)
    # the secondary (exp2) ceiling, measured outside the timed regions
    exp2_rate = fm.measure_exp2_rate(stream) if rank == 0 else None
    per_mask = fp8_points = None
    if not args.no_per_mask and rank == 0:
        del q, k, v, do, o, lse, dq, dk, dv, ws
        torch.cuda.empty_cache()
        per_mask = run_per_mask(args, fm)
        fp8_points = run_fp8_points(args, fm)
    if world > 1:
        dist.barrier()
    report(args, W, world, rank, ms, prof, flop_fwd, flop_bwd, n_vis, e2e_ms, h2d, d2h, clk,
           per_mask, exp2_rate, fp8_points, prof_ms=prof_ms, graph_ms=graph_ms, plan_ms=plan_ms)
    if world > 1:
        dist.destroy_process_group()


def run_e2e(args, fm, q, k, v, do, bounds, scale, o, lse, dq, dk, dv, ws, stream, world):
    """Same step through the public API with pinned HOST inputs and outputs:
    every step copies Q, K, V, dO and the bounds host-to-device and O, LSE,
    dQ, dK, dV device-to-host, all inside the timed region.  The copies run
    on their own streams with two device buffer sets, so step i+1's inputs
    and step i-1's outputs move while step i computes (the two copy
    directions also overlap each other)."""
    import torch
    import torch.distributed as dist
    hq, hk, hv, hdo = (x.cpu().pin_memory() for x in (q, k, v, do))
    hb = bounds.cpu().pin_memory()
    ho, hdq, hdk, hdv = (torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in (o, dq, dk, dv))
    hlse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    # two sets of device inputs and outputs (set 0 reuses the bench's outputs)
    sets = []
    for n in range(2):
        ins = tuple(torch.empty_like(x) for x in (q, k, v, do, bounds))
        outs = (o, lse, dq, dk, dv) if n == 0 else tuple(torch.empty_like(x) for x in (o, lse, dq, dk, dv))
        sets.append((ins, outs))
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    issued = [0]  # steps issued so far (their buffer-set events are recorded)

    def e2e_step():
        i = issued[0]
        n = i & 1
        (dq_in, dk_in, dv_in, ddo_in, db), (o_n, lse_n, dq_n, dk_n, dv_n) = sets[n]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(comp_done[n])  # step i-2 is done reading this set's inputs
            for d_, h_ in ((dq_in, hq), (dk_in, hk), (dv_in, hv), (ddo_in, hdo), (db, hb)):
                d_.copy_(h_, non_blocking=True)
            in_done[n].record(s_in)
        stream.wait_event(in_done[n])
        if i >= 2:
            stream.wait_event(out_done[n])  # step i-2's outputs have left this set
        fm.plan(dq_in, dk_in, db, ws=ws, for_bwd=fm.WS_STEP, stream=stream)
        fm.forward(dq_in, dk_in, dv_in, db, scale, o=o_n, lse=lse_n, ws=ws, stream=stream,
                   planned=True)
        fm.backward(dq_in, dk_in, dv_in, o_n, lse_n, ddo_in, db, scale, dq=dq_n, dk=dk_n, dv=dv_n,
                    ws=ws, stream=stream, planned=True)
        comp_done[n].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[n])
            for h_, d_ in ((ho, o_n), (hlse, lse_n), (hdq, dq_n), (hdk, dk_n), (hdv, dv_n)):
                h_.copy_(d_, non_blocking=True)
            out_done[n].record(s_out)
        issued[0] += 1

    e2e_step()
    e2e_step()
    torch.cuda.synchronize()
    e_steps = max(1, min(args.steps, 10))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0.record(s_in)
    for _ in range(e_steps):
        e2e_step()
    # the end of the timed region: the last step's outputs are on the host
    s_in.wait_event(out_done[(issued[0] - 1) & 1])
    ev1.record(s_in)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e2e_ms = _max_over_ranks(ev0.elapsed_time(ev1) / e_steps, world, "cuda")
    if fm.device_status(ws) != 0:
        raise RuntimeError("device status not OK after the end-to-end steps")
    # the forward is deterministic: the last step's host copies of O and LSE
    # equal the outputs the device-timed leg left in buffer set 0
    if not (torch.equal(ho, o.cpu()) and torch.equal(hlse, lse.cpu())):
        raise RuntimeError("end-to-end outputs differ from the device-timed outputs")
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hdo, hb))
    d2h = sum(x.numel() * x.element_size() for x in (ho, hlse, hdq, hdk, hdv))
    return e2e_ms, h2d, d2h


# FP8 (e4m3) forward points: (workload, B, H, S, mask, params)
FP8_POINTS = (
    ("suite_32k", 1, 32, 32768, "causal", {}),
    ("suite_32k", 1, 32, 32768, "causal_document", {}),
    ("long_128k", 1, 8, 131072, "causal_document_window", {"window": 8192}),
)


def run_fp8_points(args, fm):
    """FP8 forward throughput on pre-quantised inputs (fm_quantize_fp8 timed
    apart), beside the bf16 forward on the same inputs; effective TFLOP/s on
    the visible entries (4 * d flop each) against the fp8 peak taken as the
    measured bf16 peak times 2 (the nominal dense fp8 / bf16 ratio)."""
    import torch

    from fm_inputs.tensors import qkv_do
    peak = float(_peaks()[0]["bf16_tflops"])
    stream = torch.cuda.current_stream()
    out = []
    for name, B, H, S, mask, params in FP8_POINTS:
        q, k, v, _ = qkv_do(B, S, S, H, 128, seed=0, device="cuda")
        bounds = _point_bounds(fm, mask, B, S, params)
        n_vis = _visible_entries(bounds.cpu().numpy(), S, H)
        scale = 128 ** -0.5
        o = torch.empty_like(q)
        lse = torch.empty(B, H, S, dtype=torch.float32, device="cuda")
        desc = fm.make_desc(q, k, v, o)
        ws = fm.workspace(desc, fm.WS_FWD)
        f = fm.quantize_fp8(q, k, v, stream=stream)
        n = args.mask_steps
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        for i in range(2 + n):
            if i == 2:
                ev[0].record(stream)
            fm.quantize_fp8(q, k, v, stream=stream)
            if i == 2:
                ev[1].record(stream)
        ev[2].record(stream)
        for i in range(n):
            fm.forward_fp8(f, bounds, scale, o=o, lse=lse, ws=ws, stream=stream)
        ev[3].record(stream)
        for i in range(n):
            fm.forward(q, k, v, bounds, scale, o=o, lse=lse, ws=ws, stream=stream)
        ev[4].record(stream)
        torch.cuda.synchronize()
        if fm.device_status(ws) != 0:
            raise RuntimeError(f"device status not OK for fp8 {name}/{mask}")
        f8_ms = ev[2].elapsed_time(ev[3]) / n
        bf_ms = ev[3].elapsed_time(ev[4]) / n
        flop = 4.0 * 128 * n_vis
        t8 = flop / (f8_ms * 1e-3) / 1e12
        out.append({"workload": name, "mask": mask, "B": B, "H": H, "S": S, "d": 128,
                    "visible_entries": n_vis, "fwd_fp8_ms": round(f8_ms, 4),
                    "fwd_fp8_tflops": round(t8, 1),
                    "pct_fp8_peak": round(100.0 * t8 / (2 * peak), 1),
                    "fwd_bf16_ms": round(bf_ms, 4),
                    "fwd_bf16_tflops": round(flop / (bf_ms * 1e-3) / 1e12, 1),
                    "quantize_ms": round(ev[0].elapsed_time(ev[1]), 4),
                    "peak": "fp8 = 2 x bf16_tflops (burst) of measured"})
        del q, k, v, o, f, ws
        torch.cuda.empty_cache()
    return out


def run_per_mask(args, fm):
    """Forward, backward and step throughput of every (workload, mask) point,
    with the fp64 oracle timed beside each on a bounded sample.  Inputs are
    resident in HBM; each point does 2 untimed and ``args.mask_steps`` timed
    steps (CUDA events on the launch stream around fm_fwd and fm_bwd)."""
    import torch

    from fm_inputs.configs import LOCALIZE_RANKS, dual_chunk_map
    from fm_inputs.tensors import qkv_do
    peak = float(_peaks()[0]["bf16_tflops"])
    stream = torch.cuda.current_stream()
    out = []
    for name, B, H, S, d, masks, params in PER_MASK_POINTS:
        if args.mask_points and name not in args.mask_points:
            continue
        scale = d ** -0.5
        q, k, v, do = qkv_do(B, S, S, H, d, seed=0, device="cuda")
        Hkv = GQA_POINTS[name][1] if name in GQA_POINTS else H
        if Hkv != H:
            k, v = k[:, :, :Hkv].contiguous(), v[:, :, :Hkv].contiguous()
        for mask in masks:
            bounds = _point_bounds(fm, mask, B, S, params)
            bounds_np = bounds.cpu().numpy()
            n_vis = _visible_entries(bounds_np, S, H)
            if name == "localize_64k":
                # simulated ranks: local Q / dO rows, localised bounds, full K / V
                ranks = []
                for chunks in dual_chunk_map(S, LOCALIZE_RANKS):
                    rows = torch.cat([torch.arange(g, g + c, device="cuda") for g, c in chunks])
                    ranks.append((q[:, rows].contiguous(), do[:, rows].contiguous(),
                                  fm.localize(bounds, chunks)))
            else:
                ranks = [(q, do, bounds)]
            bufs = []
            for ql, dol, bl in ranks:
                o = torch.empty_like(ql)
                lse = torch.empty(B, H, ql.shape[1], dtype=torch.float32, device="cuda")
                desc = fm.make_desc(ql, k, v, o)
                bufs.append((ql, dol, bl, o, lse, torch.empty_like(ql), torch.empty_like(k),
                             torch.empty_like(v), fm.workspace(desc, fm.WS_STEP)))
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4 * args.mask_steps)]
            for i in range(2 + args.mask_steps):
                timed = i >= 2
                j = (i - 2) * 4
                if timed:
                    ev[j].record(stream)
                # the forward's time includes the step's one mask analysis
                for ql, dol, bl, o, lse, dq, dk, dv, w in bufs:
                    fm.plan(ql, k, bl, ws=w, for_bwd=fm.WS_STEP, stream=stream)
                    fm.forward(ql, k, v, bl, scale, o=o, lse=lse, ws=w, stream=stream, planned=True)
                if timed:
                    ev[j + 1].record(stream)
                for ql, dol, bl, o, lse, dq, dk, dv, w in bufs:
                    fm.backward(ql, k, v, o, lse, dol, bl, scale, dq=dq, dk=dk, dv=dv, ws=w,
                                stream=stream, planned=True)
                if timed:
                    ev[j + 2].record(stream)
            torch.cuda.synchronize()
            for b_ in bufs:
                if fm.device_status(b_[8]) != 0:
                    raise RuntimeError(f"device status not OK for {name}/{mask}")
            n = args.mask_steps
            fwd_ms = sum(ev[4 * i].elapsed_time(ev[4 * i + 1]) for i in range(n)) / n
            bwd_ms = sum(ev[4 * i + 1].elapsed_time(ev[4 * i + 2]) for i in range(n)) / n
            ff, fb = 4.0 * d * n_vis, 10.0 * d * n_vis
            tot = (ff + fb) / ((fwd_ms + bwd_ms) * 1e-3) / 1e12
            row = {"workload": name, "mask": mask, "B": B, "H": H, "Hkv": Hkv, "S": S, "d": d,
                   "visible_entries": n_vis,
                   "fwd_ms": round(fwd_ms, 4), "bwd_ms": round(bwd_ms, 4),
                   "fwd_tflops": round(ff / (fwd_ms * 1e-3) / 1e12, 1),
                   "bwd_tflops": round(fb / (bwd_ms * 1e-3) / 1e12, 1),
                   "tflops": round(tot, 1), "pct_bf16_peak": round(100.0 * tot / peak, 1)}
            if name == "localize_64k":
                row["note"] = (f"{LOCALIZE_RANKS} simulated ranks one after another on one GPU, "
                               "each fm_localize'd bounds, local Q/dO x full K/V")
            if not args.no_cpu_baseline:
                row["oracle"] = oracle_point(bounds_np, S, d, args.mask_oracle_seconds)
            out.append(row)
            del bufs, ranks
        del q, k, v, do
        torch.cuda.empty_cache()
    return out


def oracle_point(bounds_np, S, d, seconds):
    """The fp64 oracle, as it stands, on a bounded sample of one point: the
    backward pass (with its forward) of query rows [S/2, S/2 + R) of one head,
    R doubled from 64 until about ``seconds`` pass.  Those rows see the full
    key axis through bounds localised to them (oracle.masks.localize_bounds),
    so the sample is the same computation as in the full problem; the value
    is per visible entry of the sample."""
    import numpy as np

    from oracle import attention as oa
    from oracle import masks as om
    rng = np.random.default_rng(1)
    q, k, v, do = (rng.standard_normal((S, d)).astype(np.float32).astype(np.float64) for _ in range(4))
    R, el, work = 64, 0.0, 0
    while True:
        r0 = S // 2
        R = min(R, S - r0)
        lb = om.localize_bounds(bounds_np[:, :1, :1], [(r0, R)])
        mvec = tuple(lb[t, 0, 0] for t in range(4))
        t0 = time.perf_counter()
        oa.backward_head(q[r0:r0 + R], k, v, do[r0:r0 + R], mvec, d ** -0.5, slice_rows=256,
                         skip_hidden=True)
        el = time.perf_counter() - t0
        work = om.visible_count(*mvec, R)
        if el >= seconds or R >= S - S // 2:
            break
        R *= 2
    return {"value": round(14.0 * d * work / max(el, 1e-9) / 1e12, 6), "unit": "TFLOP/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"backward of query rows [{S // 2}, {S // 2 + R}) of one head, {work} visible "
                      f"entries in {el:.2f} s"}


def _traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu record, or None
    when the kernel's sources have changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    try:
        rec = json.load(open(path))[kernel]
    except (OSError, KeyError, ValueError):
        return None
    m = hashlib.sha256()
    for f in rec["sources"]:
        try:
            m.update(open(os.path.join(ROOT, "masked_attention_bound_gb300", "csrc", f), "rb").read())
        except OSError:
            return None
    return int(rec["bytes_per_launch"]) if m.hexdigest() == rec["sources_sha256"] else None


def exp2_ceiling(rate, d):
    """Effective-TFLOP/s ceilings set by a measured exp2 rate (evaluations per
    second): one exp2 per visible entry in the forward (4 * d flop), two in
    the backward (its dK/dV and dQ kernels each recompute P; 10 * d flop),
    three per step (14 * d flop)."""
    if not rate:
        return None
    return {"exp2_per_s": float(f"{rate:.4g}"),
            "fwd_tflops": round(rate * 4 * d / 1e12, 1),
            "bwd_tflops": round(rate * 10 * d / 2 / 1e12, 1),
            "step_tflops": round(rate * 14 * d / 3 / 1e12, 1),
            "how": "fm_measure_exp2_rate: one 1024-thread block per SM, eight independent "
                   "ex2.approx.f32 chains per thread, CUDA events"}


def report(args, W, world, rank, ms, prof, flop_fwd, flop_bwd, n_vis, e2e_ms, h2d, d2h, clk,
           per_mask=None, exp2_rate=None, fp8_points=None, prof_ms=None, graph_ms=None,
           plan_ms=None):
    B, H, S, d = W["B"], W["H"], W["S"], W["d"]
    flop_step = flop_fwd + flop_bwd
    if rank == 0:
        peaks, peak_src = _peaks()
        avg = {k: prof[k][0] / max(prof[k][1], 1) for k in KERNEL_GEMMS if k in prof}
        fwd_avg = avg["fwd_kernel"]
        bwd_avg = avg["bwd_kv_kernel"] + avg["bwd_dq_kernel"]
        # each attention kernel's own tensor work on the visible entries:
        # 2 * d flop per entry and GEMM (the step's metric counts 14 * d)
        flop_unit = flop_fwd / 4.0  # d * visible entries
        kernel_tflops = {k: round(2 * g * flop_unit / (avg[k] * 1e-3) / 1e12, 2)
                         for k, g in KERNEL_GEMMS.items()}
        # the dominant kernel is the one with the largest share of device time
        dom = max(KERNEL_GEMMS, key=lambda k: prof[k][0])
        achieved = kernel_tflops[dom]
        # the timed loop lasts well under a second: compare with the burst figure
        peak = float(peaks["bf16_tflops"])
        value = _job_value(flop_step, ms, world)
        launches = sum(n for _, n in prof.values())
        total_kernel_ms = sum(t for t, _ in prof.values())
        out = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 4),
            "profiled_ms_per_step": None if prof_ms is None else round(prof_ms, 4),
            "graph_ms_per_step": None if graph_ms is None else round(graph_ms, 4),
            "analysis_graph_ms": None if plan_ms is None else round(plan_ms, 4),
            "timing": "ms_per_step: the step through the public API, no per-kernel events; "
                      "profiled_ms_per_step: the same K steps with per-kernel CUDA events "
                      "(kernel_ms_per_step, roofline); graph_ms_per_step: the step captured "
                      "once as a CUDA graph and replayed K times; analysis_graph_ms: the "
                      "step's mask analysis (fm_plan) alone, as a CUDA graph replayed 100 times",
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) Q/K/V/dO, seeded document lengths)",
            "config": _config(W, n_vis, world),
            "fwd_tflops": round(flop_fwd / (fwd_avg * 1e-3) / 1e12, 2),
            "bwd_tflops": round(flop_bwd / (bwd_avg * 1e-3) / 1e12, 2),
            "kernel_tflops": kernel_tflops,
            "pct_bf16_peak": round(100.0 * value / world / peak, 1),
            "roofline": {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 2),
                         "algorithmic_flop": f"{2 * KERNEL_GEMMS[dom]} * d * visible entries "
                                             f"per launch",
                         "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                         "peak_source": f"bf16_tflops (burst) of {peak_src}",
                         "traffic": _traffic(dom) if (W["H"] == 32 and world >= 1) else None,
                         "traffic_unit": "bytes per launch (ncu dram read + write)",
                         "exp2_ceiling": exp2_ceiling(exp2_rate, d)},
            "kernel_ms_per_step": {n: round(t / args.steps, 4) for n, (t, c) in prof.items() if c},
            "kernel_launches_per_step": {n: c // args.steps for n, (t, c) in prof.items() if c},
            "kernel_time_share": {n: round(t / total_kernel_ms, 4) for n, (t, c) in prof.items() if c},
            "gpu_launches": launches,
            "e2e": None if e2e_ms != e2e_ms else {
                "value": round(_job_value(flop_step, e2e_ms, world), 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "overlap": "host-to-device and device-to-host copies on their own streams, "
                           "two device buffer sets: step i+1's inputs and step i-1's outputs "
                           "move while step i computes"},
            "clocks": clk,
        }
        if per_mask is not None:
            out["per_mask"] = per_mask
        if fp8_points is not None:
            out["fp8_forward"] = fp8_points
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
        print(json.dumps(out), flush=True)


def _oracle_sample_inputs(S, d, mask):
    import numpy as np

    from fm_inputs.tensors import mask_bounds
    bounds_np = mask_bounds(mask, 1, S).numpy()
    mvec = tuple(bounds_np[t, 0, 0] for t in range(4))
    rng = np.random.default_rng(0)
    q, k, v, do = (rng.standard_normal((S, d)).astype(np.float32).astype(np.float64)
                   for _ in range(4))
    return mvec, q, k, v, do


def cpu_baseline(seconds: float = 15.0):
    """The fp64 oracle, as it stands, on a bounded sample of the workload: the
    full backward pass (which recomputes the forward) of one head at a time,
    each head with its own seeded inputs, until about ``seconds`` have passed."""
    import numpy as np

    from oracle import attention as oa
    from oracle import masks as om

    W = WORKLOAD
    S, d = W["S"], W["d"]
    mvec, _, _, _, _ = _oracle_sample_inputs(S, d, W["mask"])
    per_head = om.visible_count(*mvec, S)
    heads, el = 0, 0.0
    rng = np.random.default_rng(0)
    while el < seconds and heads < W["H"]:
        q, k, v, do = (rng.standard_normal((S, d)).astype(np.float32).astype(np.float64)
                       for _ in range(4))
        t0 = time.perf_counter()
        oa.backward_head(q, k, v, do, mvec, d ** -0.5, slice_rows=1024, skip_hidden=True)
        el += time.perf_counter() - t0
        heads += 1
    work = heads * per_head
    return {"value": round(14.0 * d * work / el / 1e12, 6), "unit": "TFLOP/s",
            "cores": len(os.sched_getaffinity(0)), "threads": "numpy/BLAS default", "kind": "oracle",
            "sample": f"fp64 oracle backward (with its forward) of {heads} of the {W['H']} heads of "
                      f"{W['name']}: {work} visible entries in {el:.1f} s"}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    import numpy as np

    from oracle import attention as oa
    from oracle import masks as om

    W = WORKLOAD
    S, d = W["S"], W["d"]
    mvec, q, k, v, do = _oracle_sample_inputs(S, d, W["mask"])
    rows = 2048  # one bounded sample per step: the backward of 2048 query rows of one head
    n_vis = int((~om.dense_mask(*mvec, S, rows=np.arange(rows))).sum())

    def one():
        oa.backward_head(q[:rows], k, v, do[:rows], mvec, d ** -0.5, slice_rows=1024, skip_hidden=True)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = (time.perf_counter() - t0) / args.steps
    value = 14.0 * d * n_vis / el / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = (f"fp64 oracle backward (with its forward) of query rows [0, {rows}) of one head of "
              f"{W['name']} per step, {n_vis} visible entries")
    # the whole workload's count, as the device arm reports it
    from fm_inputs.tensors import mask_bounds
    n_vis_job = _visible_entries(mask_bounds(W["mask"], W["B"], S, device="cpu").numpy(), S, W["H"])
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(W, n_vis_job, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--no-per-mask", action="store_true",
                    help="skip the per-(workload, mask) measurements after the headline step")
    ap.add_argument("--mask-steps", type=int, default=5, help="timed steps per (workload, mask)")
    ap.add_argument("--mask-oracle-seconds", type=float, default=0.6,
                    help="CPU seconds of oracle sample per (workload, mask)")
    ap.add_argument("--mask-points", nargs="*", default=None,
                    help="only these workloads of the per-mask sweep")
    ap.add_argument("--heads", type=int, default=0,
                    help="override H (smaller cases for profiler captures; not a bench line)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
