"""Benchmark of the balanced expert-parallel dispatch hot path on one GB300.

One step = one pass of the whole path over one batch at the bench-shaped
training workload (R=8 virtual ranks, S=8192 tokens/rank, E=384, K=8,
H=7168, H'=2048, B=48):
    plan -> prefetch_weight -> dispatch -> grouped GEMM -> combine
    -> combine backward (dY) -> reduce_grad (replica grads into home rows).
The K timed steps cycle through four routings tuned to maxvio 0.2 / 1 / 10 / 20
(all resident in HBM), so the job spans the skew range; per-maxvio times are
reported under "sweep". Inputs (tens of GB) are far larger than L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl bep|reference]

--impl reference times the CPU oracle (the slow plain restatement) on a bounded
sample of the same workload. Under torchrun (N > 1) every rank runs an
independent replica of the job on its own GPU (the path has no cross-GPU
exchange on one GPU: replicas only); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "bench_r8_e384"
TARGETS = (0.2, 1.0, 10.0, 20.0)
METRIC = "dispatch+combine tokens/s and HBM GB/s vs peak, maxvio 0.2-20, 1 GB300"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per forward grouped GEMM call
# (its two launches: the segments of 768 rows or more with two m-tiles per unit, then
# the others), from one ncu capture of this bench at full size (mean over the four
# routings). Must be reset to None whenever that kernel changes.
GEMM_DRAM_BYTES_PER_LAUNCH = {"bench_r8_e384": 23.20e9}

# Input sets the end-to-end loop keeps on the device: uploads run up to this many steps
# ahead of compute (1.5 GB per set at the S=8192, E=384 workload, 18 GB in all).
E2E_DEPTH = 12

# Steps the end-to-end loop times at least (about 1.5 s at the S=8192, E=384 workload).
# Host-to-device copies on this platform stall for 40-90 ms now and then; the look-ahead
# hides a stall in mid-run, and a longer run keeps one that falls on the first uploads,
# which nothing can overlap, from weighing as much as it does in a 0.5 s run.
E2E_MIN_STEPS = 120


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"bep_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    s, m = float(parts[0]), float(parts[1])
                except ValueError:
                    continue
                sm.append(s)
                mx.append(m)
                for n, v in zip(names, parts[4:8]):
                    if v.lower() == "active":
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def flat_dev(xs):
    """max_i |x_i - mean| / mean, or None for no values."""
    if not xs:
        return None
    m = statistics.mean(xs)
    return max(abs(x - m) for x in xs) / m


def run_inference(bep, synth, w_home, stream, dev, reps):
    """Plan, prefetch, dispatch, grouped GEMM and combine at the inference workload (S=512,
    B=4, hot experts on one home group), timing the GEMM per maxvio target. Algorithmic GEMM
    bytes: receive rows read once, Y written once, and one weight row per non-empty segment."""
    import torch
    name = "infer_r8_e384_b4"
    wl = synth.WORKLOADS[name]
    R, S, K, E, B, H, Hp = wl.R, wl.S, wl.K, wl.E, wl.B, wl.H, wl.Hp
    cfg = bep.Config(R, E, B, K, S, H, Hp, wl.mode)
    ctx = bep.Context(cfg)
    buf = bep.Buffers(cfg, dev)
    x = synth.tokens_device((R, S, H), 11, device=dev)
    gates = torch.from_numpy(synth.gates_host(R, S, K, 11)).to(dev)
    w_slots = torch.zeros((R, B, H, Hp), dtype=torch.bfloat16, device=dev)
    res = {"workload": f"{name} (R={R}, S={S}/rank, E={E}, K={K}, H={H}, H'={Hp}, B={B}, inference)"}
    pk = peaks()
    for target in synth.MAXVIO_TARGETS[name]:
        topk = torch.from_numpy(synth.routing(wl, target, 0)).to(dev)
        # events around each call: plan | prefetch | dispatch | GEMM | combine
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(reps)]
        for i in range(reps + 1):
            e = ev[i - 1] if i > 0 else None
            if e:
                e[0].record(stream)
            bep.bep_plan(ctx, topk, buf.cu_seqlens, buf.slot_expert, buf.dest, buf.maxvio, stream)
            if e:
                e[1].record(stream)
            bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots, stream)
            if e:
                e[2].record(stream)
            bep.bep_dispatch(ctx, x, buf.dest, buf.recv, stream)
            if e:
                e[3].record(stream)
            bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_home, w_slots, buf.y, stream)
            if e:
                e[4].record(stream)
            bep.bep_combine(ctx, buf.y, buf.dest, gates, buf.out, stream)
            if e:
                e[5].record(stream)
        torch.cuda.synchronize()
        st = bep.bep_status(ctx, stream)
        if st:
            raise RuntimeError(f"device status {st}: {bep.strerror(st)}")
        cu = buf.cu_seqlens
        nseg = int((cu[:, 1:] > cu[:, :-1]).sum().item())
        # overflow segments: non-empty rows of [0, E) outside the rank's own home group
        nonempty = (cu[:, 1:E + 1] > cu[:, :E]).cpu()
        home = (torch.arange(E) // (E // R))[None, :] == torch.arange(R)[:, None]
        overflow = int((nonempty & ~home).sum().item())
        st_ms = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev) for j in range(5)]
        ms = st_ms[3]
        byts = nseg * H * Hp * 2 + R * S * K * (H + Hp) * 2
        used = int((buf.slot_expert >= 0).sum().item())
        moved = {"prefetch": used * 2 * H * Hp * 2,
                 "dispatch": R * S * H * 2 + R * S * K * H * 2 + R * S * K * 4,
                 "combine": R * S * K * Hp * 2 + R * S * Hp * 2 + R * S * K * 8}
        stage = {}
        for j, nm in ((1, "prefetch"), (2, "dispatch"), (4, "combine")):
            gbs = moved[nm] / (st_ms[j] * 1e-3) / 1e9
            stage[nm] = {"ms": round(st_ms[j], 4), "gbs": round(gbs, 1),
                         "frac_hbm": round(gbs / pk["hbm"], 3)}
        res[str(target)] = {"maxvio": round(float(buf.maxvio.item()), 4), "segments": nseg,
                            "gemm_ms": ms, "gemm_gbs": byts / (ms * 1e-3) / 1e9,
                            "frac_hbm": byts / (ms * 1e-3) / 1e9 / pk["hbm"],
                            "tflops": 2.0 * R * S * K * H * Hp / (ms * 1e-3) / 1e12,
                            "overflow_segments": overflow, "plan_ms": round(st_ms[0], 4),
                            "replicas": used, **stage}
    del ctx, buf, x, w_slots
    torch.cuda.empty_cache()
    return res


def run_small_configs(bep, synth, stream, dev, reps):
    """Latency of every stage at the small workloads, whose inputs fit in L2: the tiny
    one (R=2, E=8), the E=64 training workload at each of its maxvio targets, and the
    reduce_grad workload (H=2048, H'=1024, replica gradients N(0, 1e-3) in the used
    slots, then combine backward on H-wide rows). A 256 MiB buffer is written before
    every repeat so that no stage starts with its inputs in L2. Median microseconds."""
    import torch
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {"l2_flush": "256 MiB written before every repeat (L2 is 126 MiB)", "unit": "us"}

    def timed(fns, n):
        times = {k: [] for k in fns}
        for _ in range(n + 1):
            for k, fn in fns.items():
                with torch.cuda.stream(stream):
                    flush.fill_(1)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                times[k].append((a, b))
        torch.cuda.synchronize()
        return {k: round(statistics.median(a.elapsed_time(b) for a, b in v[1:]) * 1e3, 1)
                for k, v in times.items()}

    for name in ("tiny_r2_e8", "train_r8_e64", "grad_r8_e64"):
        wl = synth.WORKLOADS[name]
        R, S, K, E, B, H, Hp = wl.R, wl.S, wl.K, wl.E, wl.B, wl.H, wl.Hp
        cfg = bep.Config(R, E, B, K, S, H, Hp, wl.mode)
        ctx = bep.Context(cfg)
        buf = bep.Buffers(cfg, dev, with_grad=True)
        x = synth.tokens_device((R, S, H), 21, device=dev)
        gates = torch.from_numpy(synth.gates_host(R, S, K, 21)).to(dev)
        dout = synth.tokens_device((R, S, Hp), 22, device=dev)
        w_home = synth.weights_device((E, H, Hp), 23, device=dev)
        w_slots = torch.zeros((R, B, H, Hp), dtype=torch.bfloat16, device=dev)
        res = {"workload": f"{name} (R={R}, S={S}/rank, E={E}, K={K}, H={H}, H'={Hp}, B={B})"}
        for target in synth.MAXVIO_TARGETS[name]:
            topk = torch.from_numpy(synth.routing(wl, target, 0)).to(dev)
            key = "zipf1.2" if target is None else f"{target:g}"
            if name == "grad_r8_e64":
                # the backward fold: reduce_grad on the replica gradients, combine backward on
                # the [S*K, H] receive rows
                bep.bep_plan(ctx, topk, buf.cu_seqlens, buf.slot_expert, buf.dest, buf.maxvio, stream)
                g = torch.zeros((E, H, Hp), dtype=torch.float32, device=dev)
                red = torch.empty((R, B, H, Hp), dtype=torch.float32, device=dev).normal_(0, 1e-3)
                dout_h = synth.tokens_device((R, S, H), 24, device=dev)
                dy_h = torch.empty((R * S * K, H), dtype=torch.bfloat16, device=dev)
                fns = {"reduce_grad": lambda: bep.bep_reduce_grad(ctx, buf.slot_expert, g, red, stream),
                       "combine_bwd_d_h": lambda: bep.bep_combine_bwd(ctx, dout_h, buf.dest, gates, dy_h,
                                                                      stream)}
                res[key] = timed(fns, reps)
                res[key]["replicas"] = int((buf.slot_expert >= 0).sum().item())
                del g, red, dout_h, dy_h
                continue
            fns = {
                "plan": lambda: bep.bep_plan(ctx, topk, buf.cu_seqlens, buf.slot_expert, buf.dest,
                                             buf.maxvio, stream),
                "prefetch": lambda: bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots, stream),
                "dispatch": lambda: bep.bep_dispatch(ctx, x, buf.dest, buf.recv, stream),
                "gemm": lambda: bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_home, w_slots,
                                                     buf.y, stream),
                "combine": lambda: bep.bep_combine(ctx, buf.y, buf.dest, gates, buf.out, stream),
                "combine_bwd": lambda: bep.bep_combine_bwd(ctx, dout, buf.dest, gates, buf.dy, stream),
            }
            res[key] = timed(fns, reps)
            res[key]["maxvio"] = round(float(buf.maxvio.item()), 4)
        st = bep.bep_status(ctx, stream)
        if st:
            raise RuntimeError(f"device status {st}: {bep.strerror(st)}")
        out[name] = res
        del ctx, buf, x, gates, dout, w_home, w_slots
    del flush
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- GPU arm
def run_gpu(args, rank, world, local_rank):
    import numpy as np
    import torch

    import moe_expert_dispatch_online_gb300 as bep
    import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = synth.WORKLOADS[args.workload]
    R, S, K, E, B, H, Hp = wl.R, wl.S, wl.K, wl.E, wl.B, wl.H, wl.Hp
    cfg = bep.Config(R, E, B, K, S, H, Hp, wl.mode)
    ctx = bep.Context(cfg)
    buf = bep.Buffers(cfg, dev, with_grad=True)

    targets = TARGETS if args.workload == WORKLOAD else synth.MAXVIO_TARGETS[args.workload]
    topks = [torch.from_numpy(synth.routing(wl, t, 0)).to(dev) for t in targets]
    x = synth.tokens_device((R, S, H), 1, device=dev)
    gates = torch.from_numpy(synth.gates_host(R, S, K, 1)).to(dev)
    dout = synth.tokens_device((R, S, Hp), 2, device=dev)
    w_home = synth.weights_device((E, H, Hp), 3, device=dev)
    w_slots = torch.zeros((R, B, H, Hp), dtype=torch.bfloat16, device=dev)
    g_home = torch.zeros((E, H, Hp), dtype=torch.float32, device=dev)
    red = torch.empty((R, B, H, Hp), dtype=torch.float32, device=dev)
    red.normal_(0.0, 1e-3)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    stages = ("plan", "prefetch", "dispatch", "gemm", "combine", "combine_bwd", "reduce_grad")

    def step(i, ev=None):
        topk = topks[i % len(topks)]
        if ev is not None:
            ev[0].record(stream)
        bep.bep_plan(ctx, topk, buf.cu_seqlens, buf.slot_expert, buf.dest, buf.maxvio, stream)
        if ev is not None:
            ev[1].record(stream)
        bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots, stream)
        if ev is not None:
            ev[2].record(stream)
        bep.bep_dispatch(ctx, x, buf.dest, buf.recv, stream)
        if ev is not None:
            ev[3].record(stream)
        bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_home, w_slots, buf.y, stream)
        if ev is not None:
            ev[4].record(stream)
        bep.bep_combine(ctx, buf.y, buf.dest, gates, buf.out, stream)
        if ev is not None:
            ev[5].record(stream)
        bep.bep_combine_bwd(ctx, dout, buf.dest, gates, buf.dy, stream)
        if ev is not None:
            ev[6].record(stream)
        bep.bep_reduce_grad(ctx, buf.slot_expert, g_home, red, stream)
        if ev is not None:
            ev[7].record(stream)

    # per-step statistics that do not depend on timing
    maxvios, nrep = [], []
    for i in range(len(topks)):
        step(i)
        torch.cuda.synchronize()
        maxvios.append(float(buf.maxvio.item()))
        nrep.append(int((buf.slot_expert >= 0).sum().item()))
    st = bep.bep_status(ctx, stream)
    if st:
        raise RuntimeError(f"device status {st}: {bep.strerror(st)}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        time.sleep(1.0)   # nvidia-smi's first sample lands before the work starts
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        dist_barrier(world)
        t_start.record(stream)
        for i in range(args.steps):
            step(i, evs[i])
        t_end.record(stream)
        torch.cuda.synchronize()
    dist_barrier(world)
    total_ms = t_start.elapsed_time(t_end)
    stage_ms = {s: [evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)]
                for j, s in enumerate(stages)}
    st = bep.bep_status(ctx, stream)
    if st:
        raise RuntimeError(f"device status {st}: {bep.strerror(st)}")

    # ---- backward GEMMs and dispatch backward (rows beyond the step: measured apart)
    bwd = None
    if not args.no_backward:
        drecv = torch.empty((R * S * K, H), dtype=torch.bfloat16, device=dev)
        dx = torch.empty((R, S, H), dtype=torch.bfloat16, device=dev)
        nb = min(args.steps, 2 * len(topks))
        bev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(nb)]
        nseg, nwrite = [], []
        for i in range(nb + 1):
            ev = bev[i - 1] if i > 0 else None
            if ev is not None:
                ev[5].record(stream)
            step(i)            # plan, dispatch, GEMM, combine, combine_bwd for routing i
            if ev is not None:
                ev[0].record(stream)
            bep.bep_grouped_gemm_dx(ctx, buf.cu_seqlens, buf.dy, w_home, w_slots, drecv, stream)
            if ev is not None:
                ev[1].record(stream)
            bep.bep_dispatch_bwd(ctx, drecv, buf.dest, dx, stream)
            if ev is not None:
                ev[2].record(stream)
            # the weight gradient written (a step's first micro-batch), then added (a later one)
            bep.bep_grouped_gemm_dw_overwrite(ctx, buf.cu_seqlens, buf.recv, buf.dy, g_home, red,
                                              stream)
            if ev is not None:
                ev[3].record(stream)
            bep.bep_grouped_gemm_dw(ctx, buf.cu_seqlens, buf.recv, buf.dy, g_home, red, stream)
            if ev is not None:
                ev[4].record(stream)
                nseg.append(int((buf.cu_seqlens[:, 1:] > buf.cu_seqlens[:, :-1]).sum().item()))
                nwrite.append(E + int((buf.slot_expert >= 0).sum().item()))
        torch.cuda.synchronize()
        st = bep.bep_status(ctx, stream)
        if st:
            raise RuntimeError(f"device status {st}: {bep.strerror(st)}")
        dx_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in bev)
        db_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in bev)
        dwo_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in bev)
        dw_ms = statistics.mean(e[3].elapsed_time(e[4]) for e in bev)
        # one layer's forward and backward: the step's rows, dX, dispatch backward, dW
        layer_ms = statistics.mean(e[5].elapsed_time(e[3]) for e in bev)
        flops = 2.0 * R * S * K * H * Hp
        dw_bytes = statistics.mean(nseg) * H * Hp * 4 * 2 + R * S * K * (H + Hp) * 2
        dwo_bytes = statistics.mean(nwrite) * H * Hp * 4 + R * S * K * (H + Hp) * 2
        db_bytes = R * S * K * H * 2 + R * S * H * 2 + R * S * K * 4
        bwd = {
            "grouped_gemm_dx": {"ms": dx_ms, "tflops": flops / (dx_ms * 1e-3) / 1e12,
                                "frac_bf16_sustained": flops / (dx_ms * 1e-3) / 1e12 / peaks()["bf16_sus"]},
            "dispatch_bwd": {"ms": db_ms, "gbs": db_bytes / (db_ms * 1e-3) / 1e9,
                             "frac_hbm": db_bytes / (db_ms * 1e-3) / 1e9 / peaks()["hbm"]},
            "grouped_gemm_dw": {"ms": dw_ms, "tflops": flops / (dw_ms * 1e-3) / 1e12,
                                "frac_bf16_sustained": flops / (dw_ms * 1e-3) / 1e12 / peaks()["bf16_sus"],
                                "fp32_rmw_gbs": dw_bytes / (dw_ms * 1e-3) / 1e9,
                                "segments": statistics.mean(nseg)},
            "grouped_gemm_dw_overwrite": {
                "ms": dwo_ms, "tflops": flops / (dwo_ms * 1e-3) / 1e12,
                "frac_bf16_sustained": flops / (dwo_ms * 1e-3) / 1e12 / peaks()["bf16_sus"],
                "fp32_write_gbs": dwo_bytes / (dwo_ms * 1e-3) / 1e9,
                "rows_written": statistics.mean(nwrite)},
            "layer_fwd_bwd": {"ms": layer_ms, "tokens_per_s": R * S / (layer_ms * 1e-3),
                              "kernels": "plan, prefetch, dispatch, GEMM, combine, combine_bwd, "
                                         "reduce_grad, dX GEMM, dispatch_bwd, dW GEMM (overwriting)"},
            "launches": nb,
        }
        del drecv, dx
        torch.cuda.empty_cache()

    # ---- the forward with prefetch_weight on a side stream beside the dispatch: the slots
    # must be filled before the GEMM only, and the dispatch does not touch them. Both
    # chains are timed back to back per routing (plan -> prefetch | dispatch -> GEMM ->
    # combine), L2 holding no inputs (tens of GB move per chain).
    overlap = None
    if not args.no_backward:
        side = torch.cuda.Stream(device=dev)
        n_ov = max(2, min(args.steps, 8))
        ser, ovl = {}, {}
        for j, topk in enumerate(topks):
            key = "zipf1.2" if targets[j] is None else f"{targets[j]:g}"
            ts_s, ts_o = [], []
            for i in range(n_ov + 1):
                for mode, ts in (("serial", ts_s), ("overlap", ts_o)):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    planned = torch.cuda.Event()
                    filled = torch.cuda.Event()
                    a.record(stream)
                    bep.bep_plan(ctx, topk, buf.cu_seqlens, buf.slot_expert, buf.dest, buf.maxvio,
                                 stream)
                    if mode == "serial":
                        bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots, stream)
                        bep.bep_dispatch(ctx, x, buf.dest, buf.recv, stream)
                    else:
                        planned.record(stream)
                        side.wait_event(planned)
                        bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots, side)
                        filled.record(side)
                        bep.bep_dispatch(ctx, x, buf.dest, buf.recv, stream)
                        stream.wait_event(filled)
                    bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_home, w_slots, buf.y,
                                         stream)
                    bep.bep_combine(ctx, buf.y, buf.dest, gates, buf.out, stream)
                    b.record(stream)
                    if i > 0:
                        ts.append((a, b))
            torch.cuda.synchronize()
            ser[key] = statistics.mean(a.elapsed_time(b) for a, b in ts_s)
            ovl[key] = statistics.mean(a.elapsed_time(b) for a, b in ts_o)
        st = bep.bep_status(ctx, stream)
        if st:
            raise RuntimeError(f"device status {st}: {bep.strerror(st)}")
        overlap = {"forward_ms_serial": {k: round(v, 4) for k, v in ser.items()},
                   "forward_ms_prefetch_on_side_stream": {k: round(v, 4) for k, v in ovl.items()},
                   "saving_ms_mean": round(statistics.mean(ser[k] - ovl[k] for k in ser), 4),
                   "repeats": n_ov}

    # ---- dispatch + combine under a 32-SM budget (the pages' comm-SM setting)
    comm32 = None
    if not args.no_backward:
        bep.bep_set_comm_sms(ctx, 32)
        nb = min(args.steps, 2 * len(topks))
        cev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nb)]
        for i in range(nb + 1):
            bep.bep_plan(ctx, topks[i % len(topks)], buf.cu_seqlens, buf.slot_expert, buf.dest,
                         buf.maxvio, stream)
            ev = cev[i - 1] if i > 0 else None
            if ev is not None:
                ev[0].record(stream)
            bep.bep_dispatch(ctx, x, buf.dest, buf.recv, stream)
            if ev is not None:
                ev[1].record(stream)
            bep.bep_combine(ctx, buf.y, buf.dest, gates, buf.out, stream)
            if ev is not None:
                ev[2].record(stream)
        torch.cuda.synchronize()
        bep.bep_set_comm_sms(ctx, 0)
        d32 = statistics.mean(e[0].elapsed_time(e[1]) for e in cev)
        c32 = statistics.mean(e[1].elapsed_time(e[2]) for e in cev)
        rh, rhp = H * 2, Hp * 2
        db = R * S * rh + R * S * K * rh + R * S * K * 4
        cb = R * S * K * rhp + R * S * rhp + R * S * K * 8
        comm32 = {"sms": 32, "dispatch_ms": d32, "combine_ms": c32,
                  "tokens_per_s": R * S / ((d32 + c32) * 1e-3),
                  "dispatch_gbs": db / (d32 * 1e-3) / 1e9, "combine_gbs": cb / (c32 * 1e-3) / 1e9}

    # ---- the weighted combine on H-wide rows (the down projection's output, the EP payload)
    comb_h = None
    if not args.no_backward:
        out_h_dev = torch.empty((R, S, H), dtype=torch.bfloat16, device=dev)
        nb = min(args.steps, 2 * len(topks))
        hev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(nb)]
        for i in range(nb + 1):
            bep.bep_plan(ctx, topks[i % len(topks)], buf.cu_seqlens, buf.slot_expert, buf.dest,
                         buf.maxvio, stream)
            bep.bep_dispatch(ctx, x, buf.dest, buf.recv, stream)
            if i > 0:
                hev[i - 1][0].record(stream)
            bep.bep_combine(ctx, buf.recv, buf.dest, gates, out_h_dev, stream)
            if i > 0:
                hev[i - 1][1].record(stream)
        torch.cuda.synchronize()
        ch_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in hev)
        chb = R * S * K * H * 2 + R * S * H * 2 + R * S * K * 8
        comb_h = {"D": H, "ms": ch_ms, "gbs": chb / (ch_ms * 1e-3) / 1e9,
                  "frac_hbm": chb / (ch_ms * 1e-3) / 1e9 / peaks()["hbm"]}
        del out_h_dev
        torch.cuda.empty_cache()

    # ---- inference mode with overflow (B = 4 < E/R, S = 512): the grouped GEMM reads each
    # active weight row once and is bound by HBM, not by the tensor cores
    infer = None
    if not args.no_backward and args.workload == WORKLOAD:
        infer = run_inference(bep, synth, w_home, stream, dev, min(args.steps, 8))

    # ---- the ceiling of dispatch's access pattern: the same kernel with each token's K
    # copies going to K consecutive receive rows (dest[t, k] = t*K + k, no scatter), so the
    # time is the read-once / write-K-times pattern itself; likewise for combine backward
    fan = None
    if not args.no_backward and args.workload == WORKLOAD:
        dest_seq = torch.arange(R * S * K, dtype=torch.int32, device=dev).view(R, S, K)
        fev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(6)]
        for i in range(7):
            if i > 0:
                fev[i - 1][0].record(stream)
            bep.bep_dispatch(ctx, x, dest_seq, buf.recv, stream)
            if i > 0:
                fev[i - 1][1].record(stream)
        torch.cuda.synchronize()
        fan_ms = statistics.median(e[0].elapsed_time(e[1]) for e in fev)
        # combine backward has the same shape of traffic on H'-wide rows
        for i in range(7):
            if i > 0:
                fev[i - 1][0].record(stream)
            bep.bep_combine_bwd(ctx, dout, dest_seq, gates, buf.dy, stream)
            if i > 0:
                fev[i - 1][1].record(stream)
        torch.cuda.synchronize()
        cb_ms = statistics.median(e[0].elapsed_time(e[1]) for e in fev)
        fan_bytes = R * S * H * 2 * (1 + K) + R * S * K * 4
        cb_bytes = R * S * Hp * 2 * (1 + K) + R * S * K * 8
        fan = {"dispatch_contiguous_dest_ms": fan_ms,
               "dispatch_contiguous_dest_gbs": fan_bytes / (fan_ms * 1e-3) / 1e9,
               "planned_over_contiguous": statistics.mean(stage_ms["dispatch"]) / fan_ms,
               "combine_bwd_contiguous_dest_ms": cb_ms,
               "combine_bwd_contiguous_dest_gbs": cb_bytes / (cb_ms * 1e-3) / 1e9,
               "combine_bwd_planned_over_contiguous": statistics.mean(stage_ms["combine_bwd"]) / cb_ms}
        del dest_seq

    # ---- the small workloads (inputs fit in L2): per-stage latency with L2 flushed
    small = None
    if not args.no_backward and args.workload == WORKLOAD:
        small = run_small_configs(bep, synth, stream, dev, 9)

    # ---- the second projection: the down projection [E+B, H', H] on the same plan (a second
    # context with H and H' swapped), fed by the first projection's output rows
    proj2 = None
    if not args.no_backward:
        ctx2 = bep.Context(bep.Config(R, E, B, K, S, Hp, H, wl.mode))
        w_dn = synth.weights_device((E, Hp, H), 13, device=dev)
        dn_slots = torch.zeros((R, B, Hp, H), dtype=torch.bfloat16, device=dev)
        y2 = torch.empty((R * S * K, H), dtype=torch.bfloat16, device=dev)
        nb = min(args.steps, 2 * len(topks))
        pev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(nb)]
        for i in range(nb + 1):
            step(i)            # plan, prefetch, dispatch, up projection, combine, ...
            bep.bep_prefetch_weight(ctx2, buf.slot_expert, w_dn, dn_slots, stream)
            if i > 0:
                pev[i - 1][0].record(stream)
            bep.bep_grouped_gemm(ctx2, buf.cu_seqlens, buf.y, w_dn, dn_slots, y2, stream)
            if i > 0:
                pev[i - 1][1].record(stream)
        torch.cuda.synchronize()
        st = bep.bep_status(ctx2, stream)
        if st:
            raise RuntimeError(f"device status {st}: {bep.strerror(st)}")
        p2_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in pev)
        fl = 2.0 * R * S * K * H * Hp
        proj2 = {"ms": p2_ms, "tflops": fl / (p2_ms * 1e-3) / 1e12,
                 "frac_bf16_sustained": fl / (p2_ms * 1e-3) / 1e12 / peaks()["bf16_sus"]}
        del ctx2, w_dn, dn_slots, y2
        torch.cuda.empty_cache()

    # ---- the VM group GEMM through the weight store's aliased [E+B, H, H'] views
    vmg = None
    if not args.no_backward:
        try:
            store = bep.WeightStore(cfg, layers=1)
        except bep.BepError as exc:
            vmg = {"unavailable": str(exc)}
            store = None
        if store is not None:
            s_home, s_slots, s_views = store.home(0), store.slots(), store.views(0)
            s_home.copy_(w_home)
            nb = min(args.steps, 2 * len(topks))
            vev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(nb)]
            for i in range(nb + 1):
                bep.bep_plan(ctx, topks[i % len(topks)], buf.cu_seqlens, buf.slot_expert,
                             buf.dest, buf.maxvio, stream)
                bep.bep_prefetch_weight(ctx, buf.slot_expert, s_home, s_slots, stream)
                bep.bep_dispatch(ctx, x, buf.dest, buf.recv, stream)
                if i > 0:
                    vev[i - 1][0].record(stream)
                bep.bep_grouped_gemm_vm(ctx, buf.cu_seqlens, buf.recv, s_views, buf.y, stream)
                if i > 0:
                    vev[i - 1][1].record(stream)
            torch.cuda.synchronize()
            st = bep.bep_status(ctx, stream)
            if st:
                raise RuntimeError(f"device status {st}: {bep.strerror(st)}")
            vm_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in vev)
            fl = 2.0 * R * S * K * H * Hp
            vmg = {"ms": vm_ms, "tflops": fl / (vm_ms * 1e-3) / 1e12,
                   "frac_bf16_sustained": fl / (vm_ms * 1e-3) / 1e12 / peaks()["bf16_sus"]}
            del s_home, s_slots, s_views
            store.close()
            torch.cuda.empty_cache()

    # ---- end to end through the public API with host buffers. Every step uploads its
    # inputs (topk, x, gates, dOut) from pinned host memory and downloads its output.
    # The uploads run on their own stream up to E2E_DEPTH steps ahead of compute, into
    # E2E_DEPTH device input sets; the downloads run on a third stream. Host-to-device
    # copies on this platform now and then stall for tens of milliseconds (one copy in
    # 20-40 took 60-90 ms instead of 5.7 ms); the look-ahead absorbs such a stall the way
    # an input pipeline does, and every step's inputs are still copied inside the timed
    # region.
    x_h = x.cpu().pin_memory()
    dout_h = dout.cpu().pin_memory()
    gates_h = gates.cpu().pin_memory()
    topks_h = [t.cpu().pin_memory() for t in topks]
    out_h = [torch.empty(buf.out.shape, dtype=buf.out.dtype).pin_memory() for _ in range(2)]
    depth = E2E_DEPTH
    sets = [dict(topk=torch.empty_like(topks[0]), x=torch.empty_like(x), g=torch.empty_like(gates),
                 dout=torch.empty_like(dout), out=torch.empty_like(buf.out)) for _ in range(depth)]
    h2d = x_h.numel() * 2 + dout_h.numel() * 2 + gates_h.numel() * 4 + topks_h[0].numel() * 4
    d2h = out_h[0].numel() * 2
    up_stream = torch.cuda.Stream(device=dev)
    down_stream = torch.cuda.Stream(device=dev)
    loaded = [torch.cuda.Event() for _ in range(depth)]
    released = [torch.cuda.Event() for _ in range(depth)]

    def upload(i):
        b = sets[i % depth]
        with torch.cuda.stream(up_stream):
            if i >= depth:   # step i - depth has consumed this set and its output is read back
                up_stream.wait_event(released[i % depth])
            b["topk"].copy_(topks_h[i % len(topks_h)], non_blocking=True)
            b["x"].copy_(x_h, non_blocking=True)
            b["g"].copy_(gates_h, non_blocking=True)
            b["dout"].copy_(dout_h, non_blocking=True)
            loaded[i % depth].record(up_stream)

    def e2e_run(n):
        for i in range(min(n, depth)):
            upload(i)
        for i in range(n):
            b = sets[i % depth]
            stream.wait_event(loaded[i % depth])
            bep.bep_plan(ctx, b["topk"], buf.cu_seqlens, buf.slot_expert, buf.dest, buf.maxvio,
                         stream)
            bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots, stream)
            bep.bep_dispatch(ctx, b["x"], buf.dest, buf.recv, stream)
            bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_home, w_slots, buf.y, stream)
            bep.bep_combine(ctx, buf.y, buf.dest, b["g"], b["out"], stream)
            bep.bep_combine_bwd(ctx, b["dout"], buf.dest, b["g"], buf.dy, stream)
            bep.bep_reduce_grad(ctx, buf.slot_expert, g_home, red, stream)
            down_stream.wait_stream(stream)
            with torch.cuda.stream(down_stream):
                out_h[i % 2].copy_(b["out"], non_blocking=True)
                released[i % depth].record(down_stream)
            if i + depth < n:
                upload(i + depth)
        stream.wait_stream(up_stream)
        stream.wait_stream(down_stream)

    e2e_run(max(args.warmup, depth))   # every input set used once before the timer starts
    torch.cuda.synchronize()
    dist_barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up_stream.wait_event(e0)
    down_stream.wait_event(e0)
    e2e_steps = max(args.steps, E2E_MIN_STEPS)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    dist_barrier(world)

    total_ms = dist_max(world, total_ms)
    e2e_ms = dist_max(world, e2e_ms)
    tokens_per_step = R * S
    pk = peaks()
    gemm_ms = statistics.mean(stage_ms["gemm"])
    gemm_flops = 2.0 * R * S * K * H * Hp
    gemm_tflops = gemm_flops / (gemm_ms * 1e-3) / 1e12
    # algorithmic HBM bytes of the memory-bound stages
    row_h, row_hp = H * 2, Hp * 2
    disp_bytes = R * S * row_h + R * S * K * row_h + R * S * K * 4
    comb_bytes = R * S * K * row_hp + R * S * row_hp + R * S * K * 8
    disp_ms = statistics.mean(stage_ms["dispatch"])
    comb_ms = statistics.mean(stage_ms["combine"])
    per_target = {}
    for j, t in enumerate(targets):
        idx = [i for i in range(args.steps) if i % len(targets) == j]
        if not idx:
            continue
        step_ms = [sum(stage_ms[s][i] for s in stages) for i in idx]
        fwd = ("plan", "prefetch", "dispatch", "gemm", "combine")
        fwd_ms = [sum(stage_ms[s][i] for s in fwd) for i in idx]
        fwd_np_ms = [sum(stage_ms[s][i] for s in fwd if s != "prefetch") for i in idx]
        per_target["zipf1.2" if t is None else f"{t:g}"] = {
            "maxvio": round(maxvios[j], 4), "replicas": nrep[j],
            "step_ms": round(statistics.mean(step_ms), 4),
            # the forward alone (plan ... combine), with and without the prefetch of replicas
            "forward_ms": round(statistics.mean(fwd_ms), 4),
            "forward_ms_without_prefetch": round(statistics.mean(fwd_np_ms), 4),
            **{f"{s}_ms": round(statistics.mean(stage_ms[s][i] for i in idx), 4) for s in stages},
        }
    traffic = GEMM_DRAM_BYTES_PER_LAUNCH.get(args.workload)
    clocks = clk.summary()
    result = {
        "metric": METRIC,
        "value": world * tokens_per_step * args.steps / (total_ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded Dirichlet-popularity Gumbel-top-K routing; bf16 U[-1,1] tokens, "
                "N(0,0.02) weights, softmax gates)",
        "config": {"workload": f"{args.workload} (R={R} virtual ranks, S={S}/rank, E={E}, K={K}, "
                               f"H={H}, H'={Hp}, B={B}, training)",
                   "maxvio_targets": list(targets), "global_batch_tokens": R * S,
                   "l2": "inputs larger than L2 (tens of GB per step)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU, R virtual ranks"},
        "stages_ms": {s: round(statistics.mean(v), 4) for s, v in stage_ms.items()},
        "dispatch_combine": {
            "tokens_per_s": tokens_per_step / ((disp_ms + comb_ms) * 1e-3),
            "dispatch_gbs": disp_bytes / (disp_ms * 1e-3) / 1e9,
            "combine_gbs": comb_bytes / (comb_ms * 1e-3) / 1e9,
            "dispatch_frac_hbm": disp_bytes / (disp_ms * 1e-3) / 1e9 / pk["hbm"],
            "combine_frac_hbm": comb_bytes / (comb_ms * 1e-3) / 1e9 / pk["hbm"],
            "frac_vs_8000gbs": (disp_bytes + comb_bytes) / ((disp_ms + comb_ms) * 1e-3) / 1e9 / 8000.0,
        },
        "sweep": per_target,
        "flatness_max_over_min": (max(v["step_ms"] for v in per_target.values()) /
                                  min(v["step_ms"] for v in per_target.values())) if per_target else None,
        # largest deviation of one maxvio target's step time from the mean over the targets
        # (the +-10% flatness criterion), for the whole step and for dispatch+combine alone
        "flatness_dev_from_mean": flat_dev([v["step_ms"] for v in per_target.values()]),
        "dispatch_combine_dev_from_mean": flat_dev(
            [v["dispatch_ms"] + v["combine_ms"] for v in per_target.values()]),
        "forward_dev_from_mean": flat_dev([v["forward_ms"] for v in per_target.values()]),
        # The timed region is K steps of about 12 ms (a fraction of a second), not a seconds-long
        # loop, so the burst peak is the one that applies; the sustained figure rides along.
        "roofline": {"kernel": "grouped_gemm", "bound": "tensor", "achieved": gemm_tflops,
                     "peak": pk["bf16"], "unit": "TFLOP/s", "frac": gemm_tflops / pk["bf16"],
                     "peak_source": f"{pk['src']} bf16 burst (the timed region lasts under a second)",
                     "frac_of_sustained": gemm_tflops / pk["bf16_sus"],
                     "traffic": traffic},
        "e2e": {"value": world * tokens_per_step * e2e_steps / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        # our kernels per step: plan 4, prefetch 1, dispatch 1, GEMM 2 (work list, GEMM) or 4
        # (the library's two-launch forward: H >= 2048, 256 | H', at least 512 receive rows
        # per expert), combine 1, combine backward 1, reduce_grad 2
        "gpu_launches": (12 + (2 if (H >= 2048 and Hp % 256 == 0 and R * S * K >= 512 * E) else 0))
                        * args.steps,
        "clocks": clocks,
        "backward": bwd,
        "prefetch_overlap": overlap,
        "comm_sms_32": comm32,
        "vm_group_gemm": vmg,
        "combine_d_h": comb_h,
        "second_projection": proj2,
        "inference": infer,
        "small_configs": small,
        "dispatch_pattern_ceiling": fan,
    }
    dc = result["dispatch_combine"]
    disp_gbs, comb_gbs = dc["dispatch_gbs"], dc["combine_gbs"]
    result["summary"] = {
        "step_tokens_per_s": round(result["value"]),
        "e2e_tokens_per_s": round(result["e2e"]["value"]),
        "dispatch_combine_tokens_per_s": round(dc["tokens_per_s"]),
        "dispatch": {"ms": round(disp_ms, 4), "gbs": round(disp_gbs, 1),
                     "frac_of_measured_hbm": round(disp_gbs / pk["hbm"], 3),
                     "frac_of_8000": round(disp_gbs / 8000.0, 3)},
        "combine": {"ms": round(comb_ms, 4), "gbs": round(comb_gbs, 1),
                    "frac_of_measured_hbm": round(comb_gbs / pk["hbm"], 3),
                    "frac_of_8000": round(comb_gbs / 8000.0, 3)},
        "hbm_peak_gbs": pk["hbm"],
        "gemm": {"ms": round(gemm_ms, 4), "tflops": round(gemm_tflops, 1),
                 "frac_of_burst": round(gemm_tflops / pk["bf16"], 3),
                 "frac_of_sustained": round(gemm_tflops / pk["bf16_sus"], 3)},
        "step_ms_per_maxvio": {k: v["step_ms"] for k, v in per_target.items()},
        "dispatch_combine_ms_per_maxvio": {k: round(v["dispatch_ms"] + v["combine_ms"], 4)
                                           for k, v in per_target.items()},
        "flatness_dev_from_mean": {"step": result["flatness_dev_from_mean"],
                                   "forward": result["forward_dev_from_mean"],
                                   "dispatch_combine": result["dispatch_combine_dev_from_mean"],
                                   "criterion": 0.10},
        "dw_ms": (round(bwd["grouped_gemm_dw"]["ms"], 3)
                  if isinstance(bwd, dict) and "grouped_gemm_dw" in bwd else None),
    }
    return result


# ----------------------------------------------------------------------------- CPU oracle
class CpuSample:
    """The oracle, as it stands, on a bounded sample of the bench workload; each
    stage's cost is scaled to one whole step. Inputs are drawn once; step() times
    the oracle's work only. Runs single-threaded (BLAS threads pinned to 1).

    Two sizes: "baseline" (the GPU arm's cpu_baseline, one sample of several seconds
    of CPU work) and "step" (the reference arm, one smaller sample per timed step)."""

    SIZES = {  # (tokens for dispatch / combine, GEMM receive rows, prefetch / reduce_grad 1/FRAC slot)
        "baseline": (16384, 8192, 1),
        "step": (2048, 256, 4),
    }

    def __init__(self, size: str = "baseline"):
        self.N_TOK, self.M_ROWS, self.FRAC = self.SIZES[size]
        import numpy as np

        import synth
        self.np = np
        wl = synth.WORKLOADS[WORKLOAD]
        self.wl = wl
        R, S, K, E, B, H, Hp = wl.R, wl.S, wl.K, wl.E, wl.B, wl.H, wl.Hp
        n = self.N_TOK
        self.topk = synth.routing(wl, 10.0, 0)
        self.x = synth.tokens_host((1, n, H), 1)
        self.dest = np.arange(n * K, dtype=np.int32).reshape(1, n, K)
        self.g = synth.gates_host(1, n, K, 1)
        self.y = synth.tokens_host((n * K, Hp), 2)
        self.dout = synth.tokens_host((1, n, Hp), 3)
        self.w = synth.weights_host((H, Hp), 4)
        gsz = (H * Hp) // self.FRAC
        self.G1 = np.zeros((1, gsz), np.float32)
        self.red1 = np.ones((1, 1, gsz), np.float32)
        self.w_home1 = synth.weights_host((1, gsz), 5)
        self.slots1 = np.zeros((1, 1, gsz), np.uint16)
        self.zero_map = np.zeros((1, 1), np.int32)

    def step(self):
        import oracle
        np = self.np
        wl = self.wl
        R, S, K, E, B, H, Hp = wl.R, wl.S, wl.K, wl.E, wl.B, wl.H, wl.Hp
        C, n, m = S * K, self.N_TOK, self.M_ROWS
        tok_scale = R * S / n
        raw = {}

        def timed(name, fn):
            t0 = time.perf_counter()
            out = fn()
            raw[name] = time.perf_counter() - t0
            return out

        p = timed("plan", lambda: oracle.plan(self.topk, E, B, wl.mode))
        recv = timed("dispatch", lambda: oracle.dispatch(self.x, self.dest))
        timed("combine", lambda: oracle.combine(self.y, self.dest, self.g))
        timed("combine_bwd", lambda: oracle.combine_bwd(self.dout, self.dest, self.g))
        timed("gemm_rows", lambda: oracle.gemm_rows(recv[:m], self.w))
        timed("weight_conversion", lambda: oracle.bf16_to_f32(self.w).astype(np.float64))
        timed("reduce_grad", lambda: oracle.reduce_grad(self.G1, self.red1, self.zero_map))
        timed("prefetch", lambda: oracle.prefetch(self.w_home1, self.zero_map, self.slots1))
        nseg = int(sum((np.diff(p.cu[u]) > 0).sum() for u in range(R)))
        used = int((p.slot_expert >= 0).sum())
        # each stage's sample time scaled to one whole step of R*S tokens
        t_gemm = (max(raw["gemm_rows"] - raw["weight_conversion"], 0.0) * (R * C / m) +
                  raw["weight_conversion"] * nseg)
        stages = {"plan": raw["plan"], "prefetch": raw["prefetch"] * self.FRAC * used,
                  "dispatch": raw["dispatch"] * tok_scale, "gemm": t_gemm,
                  "combine": raw["combine"] * tok_scale, "combine_bwd": raw["combine_bwd"] * tok_scale,
                  "reduce_grad": raw["reduce_grad"] * self.FRAC * used}
        step_s = sum(stages.values())
        return {
            "value": R * S / step_s, "unit": "tokens/s", "kind": "oracle",
            "sample": (f"maxvio-10 routing: plan on all {R * S} tokens; dispatch/combine/"
                       f"combine_bwd on {n} tokens; GEMM on {m} rows + one weight conversion "
                       f"(scaled by {nseg} segments); prefetch/reduce_grad on 1/{self.FRAC} slot "
                       f"(scaled by {used} slots); scaled to one step of {R * S} tokens"),
            # wall time this sample actually took, and what one whole step would take
            "sample_seconds": sum(raw.values()),
            "step_seconds_est": step_s,
            "scale_to_full_step": step_s / sum(raw.values()),
            "stages_s": stages,
        }


def cpu_samples(steps: int, warmup: int, size: str = "baseline"):
    cs = CpuSample(size)
    out = []
    for i in range(warmup + steps):
        r = cs.step()
        if i >= warmup:
            out.append(r)
    return out


def cpu_model() -> str:
    """The host CPU's model name, as the OS reports it."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:   # noqa: BLE001
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_baseline_subprocess(steps: int = 1, warmup: int = 0, size: str = "baseline",
                            threads: int = 1):
    """The oracle timing in a fresh process: single-threaded (the oracle as it stands,
    BLAS threads 1), or on `threads` cores (the same oracle source built with OpenMP,
    numpy's BLAS on as many threads)."""
    env = dict(os.environ, OMP_NUM_THREADS=str(threads), OPENBLAS_NUM_THREADS=str(threads),
               MKL_NUM_THREADS=str(threads))
    if threads > 1:
        env["ORACLE_OPENMP"] = "1"
    else:
        env.pop("ORACLE_OPENMP", None)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", size,
                        "--steps", str(steps), "--warmup", str(warmup)], env=env,
                       capture_output=True, text=True, timeout=1800)
    if r.returncode != 0:
        return [{"error": r.stderr.strip().splitlines()[-1] if r.stderr.strip() else "failed"}]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    for o in out:
        o["cores"] = threads
    return out


def cpu_baseline():
    """cpu_baseline of the bench line: the oracle single-threaded (value, cores = 1) and
    again on every host core (all_cores), one discarded sample before each."""
    nproc = os.cpu_count() or 1
    keep = ("value", "unit", "cores", "kind", "sample", "sample_seconds", "step_seconds_est",
            "scale_to_full_step", "error")
    one = {k: v for k, v in cpu_baseline_subprocess(1, 1)[0].items() if k in keep}
    allc = {k: v for k, v in cpu_baseline_subprocess(1, 1, threads=nproc)[0].items()
            if k in ("value", "cores", "sample_seconds", "step_seconds_est", "error")}
    allc["build"] = ("the same oracle source built with -fopenmp (per-token loops of dispatch, "
                     "combine, combine_bwd, prefetch and reduce_grad on every core); numpy BLAS "
                     "threads = cores for the GEMM rows")
    one["all_cores"] = allc
    one["nproc"] = nproc
    one["cpu_model"] = cpu_model()
    return one


def run_reference(args, rank, world):
    """The reference arm: the oracle on the host cores, each step one bounded sample.
    ms_per_step is the wall time a timed step actually took (one sample); value is the
    sample's throughput scaled to whole steps (each stage by the share of the step it ran)."""
    if rank != 0:
        return None
    res = cpu_baseline_subprocess(args.steps, args.warmup, size="step")
    ok = [r for r in res if "value" in r]
    v = statistics.mean(r["value"] for r in ok) if ok else None
    wall = statistics.mean(r["sample_seconds"] for r in ok) if ok else None
    est = statistics.mean(r["step_seconds_est"] for r in ok) if ok else None
    base = res[-1] if res else {}
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": wall * 1e3 if wall else None, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32/bf16 (oracle)", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD} (R=8, S=8192/rank, E=384, K=8, H=7168, H'=2048, B=48)"},
        "sample": {"per_step": base.get("sample"),
                   "measured_seconds_per_step": wall,
                   "full_step_seconds_est": est,
                   "scale_to_full_step": (est / wall) if wall else None,
                   "scaled_tokens_per_s": v},
        "cpu_baseline": {k: base.get(k) for k in ("kind", "cores", "sample")} | {"value": v},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        **({"error": base["error"]} if "error" in base else {}),
    }


# ----------------------------------------------------------------------------- multi-process
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("BEP_DIST_BACKEND", "gloo")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world, local


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(world, v: float) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", default="bep", choices=("bep", "reference"))
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the separate timing of the backward GEMMs and dispatch backward")
    ap.add_argument("--cpu-sample", choices=tuple(CpuSample.SIZES), default=None,
                    help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_sample:
        print(json.dumps(cpu_samples(args.steps, args.warmup, args.cpu_sample)))
        return
    rank, world, local = dist_init()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if rank == 0:
            print(json.dumps(res))
        return
    res = run_gpu(args, rank, world, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline()
            cb = res["cpu_baseline"]
            res["summary"]["cpu_baseline_tokens_per_s"] = {
                "1_core": cb.get("value"),
                f"{cb['all_cores'].get('cores')}_cores": cb["all_cores"].get("value")}
        # the figures the metric names, last on the line
        res["summary"] = res.pop("summary")
        print(json.dumps(res))


if __name__ == "__main__":
    main()
