"""Benchmark: MoE expert-parallel route -> layout -> dispatch -> combine on GB300.

One step = one pass of the whole hot path over one batch of the prefill
workload: 8 logical data-parallel ranks x 4096 tokens (N = 32768), E = 256
experts, K = 8, H = 7168; route top-K over float32 logits, stable expert-major
layout, FP8 E4M3 1x128 contiguous dispatch, combine of bf16 expert outputs
(the stand-in for the grouped GEMM, N(0,1)) with fp32 accumulation.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  `value` is whole-path tokens/s with inputs
resident in HBM (per-step CUDA events on the launching stream, L2 flushed
between steps with a 512 MiB write); `e2e` times the same path through the
public API with pinned host buffers, host->device copies of the step's inputs
and the device->host read of the combined output inside the timed region.
`--impl reference` times the CPU oracle (single thread) on a bounded sample
of the same workload.  With N > 1 (torchrun) each rank runs an independent
replica of the path on its own GPU and batch (weak scaling; there is no data
exchange between ranks, only a host barrier and a max-reduction of times).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s and achieved HBM GB/s (% of GB300 peak) on 1 GB300"
SPEC_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOAD_DESC = ("prefill: 8 logical ranks x 4096 tokens (N=32768), E=256 experts (32/rank), "
                 "K=8, H=7168; FP8 E4M3 1x128 contiguous dispatch; combine of bf16 expert "
                 "outputs N(0,1), fp32 accumulate")


# ------------------------------------------------------------------ helpers --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    # host-side barrier and max-reduction only: gloo, no GPU collective
    dist.init_process_group("gloo")
    return dist


def max_over_ranks(dist, value: float) -> float:
    """Largest value over all ranks (the slowest rank sets the job time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "combine_ep_route_topk_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, src_files):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
    except Exception:
        return None
    if rec.get("source_hash") != kernel_source_hash(src_files):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms={period_ms}", f"--id={gpu_id}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def describe_workload(w, N):
    return (f"{w.R} logical ranks, {N} tokens, E={w.E}, K={w.K}, H={w.H}, "
            f"{'FP8 E4M3 1x128' if w.dtype else 'bf16'} "
            f"{'masked (capacity %d)' % w.cap if w.layout else 'contiguous'} dispatch, "
            f"bf16 combine" + (", experts renumbered by the balanced partition"
                               if w.relabel else ""))


def gpu_smi_id(local: int) -> str:
    """nvidia-smi --id for this process's CUDA device (its UUID when known)."""
    import torch
    uuid = getattr(torch.cuda.get_device_properties(local), "uuid", None)
    if uuid:
        u = str(uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        parts = [p.strip() for p in vis.split(",") if p.strip()]
        if local < len(parts):
            return parts[local]
    return str(local)


def byte_model(N, E, K, H, fp8=True, delivered=None):
    """Algorithmic bytes per launch (the minimum each kernel must move).
    `delivered` rows are written by dispatch and read by combine (N*K for
    the contiguous layout; the masked layout drops picks past capacity)."""
    D = N * K if delivered is None else delivered
    row_out = (H + H // 128 * 4) if fp8 else H * 2
    return {
        "route": N * E * 4 + N * K * 8,
        "layout": N * K * 4 + N * K * 8,
        "dispatch": N * H * 2 + D * row_out + N * K * 8,
        "combine": D * H * 2 + N * H * 2 + N * K * 12,
        # each pick counted as a full row read and a row written
        "dispatch_rowwise": D * H * 2 + D * row_out,
    }


# ------------------------------------------------------------------ our arm --

def run_ours(args, world, rank, local):
    import torch
    import combine_ep_route_topk_gb300 as ep
    from combine_ep_route_topk_gb300 import workloads as wl
    from combine_ep_route_topk_gb300.pipeline import HostPipeline, host_empty

    dist = init_dist(world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = wl.WORKLOADS[args.workload]
    if args.tokens_per_rank:  # smaller case of the same workload (profiling)
        w = w.scaled(batch=("fixed", args.tokens_per_rank))
    inp = wl.make_inputs(w, seed=args.seed + rank, device=str(dev))
    N, E, K, H, R = inp["N"], w.E, w.K, w.H, w.R
    logits, ro, x, y = inp["logits"], inp["rank_offsets"], inp["x"], inp["y"]
    layout = w.layout
    cap = w.cap if layout == ep.EP_LAYOUT_MASKED else 0
    dtype = w.dtype
    rows = N * K if layout == ep.EP_LAYOUT_CONTIG else E * cap

    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    idx = torch.empty(N, K, dtype=torch.int32, device=dev)
    wt = torch.empty(N, K, dtype=torch.float32, device=dev)
    lay = ep.alloc_layout(N, E, K, R, cap, dev)
    ws = torch.empty(ep.ep_dispatch_layout_workspace_size(N, E, K, R), dtype=torch.uint8,
                     device=dev)
    fp8 = dtype == ep.EP_DTYPE_FP8_E4M3_B128
    q = torch.empty(rows, H, dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    qs = torch.empty(rows, H // 128, dtype=torch.float32, device=dev) if fp8 else None
    comb = torch.empty(N, H, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    fused = args.fused
    ws_fused = torch.empty(ep.ep_route_layout_workspace_size(N, E, K, R), dtype=torch.uint8,
                           device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    emap = None
    if w.relabel:  # balanced renumbering measured on this batch (before timing)
        i0, _ = ep.ep_route_topk(logits, K)
        emap = ep.ep_expert_balance_map(ep.ep_dispatch_layout(i0, ro, E).counts)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        if fused:  # route + layout in one cooperative kernel
            ep.ep_route_layout(logits, ro, K, cap, expert_map=emap, topk_idx=idx, topk_w=wt,
                               out=lay, status=status, workspace=ws_fused)
            if ev:
                ev[1].record(stream)
        else:
            ep.ep_route_topk(logits, K, expert_map=emap, topk_idx=idx, topk_w=wt)
            if ev:
                ev[1].record(stream)
            ep.ep_dispatch_layout(idx, ro, E, cap, out=lay, workspace=ws)
        if ev:
            ev[2].record(stream)
        ep.ep_dispatch(x, idx, lay.pos, lay.expert_offsets, E, layout, cap, dtype, out=q,
                       out_scales=qs)
        if ev:
            ev[3].record(stream)
        ep.ep_combine(y, idx, wt, lay.pos, lay.expert_offsets, E, layout, cap, out=comb)
        if ev:
            ev[4].record(stream)

    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize()
    delivered = N * K if layout == ep.EP_LAYOUT_CONTIG else int(lay.masked_m.sum().item())

    # timed region: one event pair per step, nothing between the kernels (an
    # event between two kernels would keep the second from launching early)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    sampler = ClockSampler(gpu_smi_id(local)) if rank == 0 else None
    barrier(dist)
    torch.cuda.synchronize()
    launches0 = ep.ep_kernel_launch_count()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.fill_((i + 7) & 0xFF)  # L2 flush, outside the step's events
        step_ev[i][0].record(stream)
        step()
        step_ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    barrier(dist)
    launches = ep.ep_kernel_launch_count() - launches0
    clocks = sampler.stop() if sampler else None
    # per-kernel breakdown (roofline): a second pass with events between stages
    n_bd = max(10, min(args.steps, 100))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_bd)]
    for i in range(n_bd):
        flush.fill_((i + 11) & 0xFF)
        step(evs[i])
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("route+layout kernel reported a barrier timeout")


    stage = {n: [e[j].elapsed_time(e[j + 1]) for e in evs]
             for j, n in enumerate(["route", "layout", "dispatch", "combine"])}
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    total_ms = max_over_ranks(dist, sum(step_ms))
    # dispatch + combine time per step, from the breakdown pass
    dc_ms = max_over_ranks(dist, sum(a + b for a, b in zip(stage["dispatch"], stage["combine"])))
    dc_ms *= args.steps / n_bd

    # ---- end to end through the public API, host buffers --------------------
    e2e_line = None
    if not args.no_e2e:
        # Inputs start in pinned host memory and the result goes back to it; the
        # copies are inside the timed region.  Headline: HostPipeline, whose
        # copies in overlap the previous step's kernels and copy out.  Beside it,
        # the latency of one step run alone (copies in, kernels, copy out).
        # Host-link bandwidth is shared with the machine's other users and drifts,
        # so the two schedules alternate in windows and each reports its median
        # window.
        n_win = 5
        e2e_steps = max(2, min(args.steps, 30) // n_win)  # steps per window

        def host_copy(t):  # huge-page page-locked host memory (ep_host_alloc)
            h = host_empty(tuple(t.shape), t.dtype)
            h.copy_(t)
            return h
        x_h, lg_h, ro_h, y_h = (host_copy(t) for t in (x, logits, ro, y))
        outs_h = [host_empty((N, H), torch.bfloat16) for _ in range(2)]
        h2d = x_h.numel() * 2 + lg_h.numel() * 4 + ro_h.numel() * 4 + y_h.numel() * 2
        d2h = outs_h[0].numel() * 2
        hp = HostPipeline(N, E, K, H, R, dtype, dev, cap=cap, expert_map=emap)
        torch.cuda.synchronize()

        def gbs(nbytes, ms):
            return round(nbytes / ms / 1e6, 1) if ms > 0 else None

        def pipelined_window(n):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier(dist)
            a.record(stream)
            for i in range(n):
                hp.step(x_h, lg_h, ro_h, y_h, outs_h[i % 2])
            hp.join(stream)
            b.record(stream)
            torch.cuda.synchronize()
            barrier(dist)
            t_in, t_out = hp.copy_ms()  # the window's last step
            return max_over_ranks(dist, a.elapsed_time(b)), (gbs(h2d, t_in), gbs(d2h, t_out))

        def serial_window(n):
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
            barrier(dist)
            for e in ev:
                e[0].record(stream)
                x.copy_(x_h, non_blocking=True)
                logits.copy_(lg_h, non_blocking=True)
                ro.copy_(ro_h, non_blocking=True)
                y.copy_(y_h, non_blocking=True)
                e[1].record(stream)
                step()
                e[2].record(stream)
                outs_h[0].copy_(comb, non_blocking=True)
                e[3].record(stream)
            torch.cuda.synchronize()
            barrier(dist)
            last = ev[-1]
            rates = (gbs(h2d, last[0].elapsed_time(last[1])),
                     gbs(d2h, last[2].elapsed_time(last[3])))
            return max_over_ranks(dist, sum(e[0].elapsed_time(e[3]) for e in ev)), rates

        pipelined_window(2)  # warm-up of both schedules
        serial_window(1)
        win_pipe, win_serial, rate_pipe, rate_serial = [], [], [], []
        for _ in range(n_win):
            t, r = pipelined_window(e2e_steps)
            win_pipe.append(t)
            rate_pipe.append(r)
            t, r = serial_window(e2e_steps)
            win_serial.append(t)
            rate_serial.append(r)
        e2e_ms = statistics.median(win_pipe)
        serial_ms = statistics.median(win_serial)
        tok_step = N * world * e2e_steps
        e2e_line = {
            "value": round(tok_step / (e2e_ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_ms / e2e_steps, 3), "steps": e2e_steps * n_win,
            "schedule": "ep_host_pipeline_* (C ABI, via pipeline.HostPipeline): step i+1's "
                        "copies in overlap step i's kernels and copy out (double-buffered "
                        "device inputs and result)",
            "host_memory": "ep_host_alloc: page-locked, transparent-huge-page backed",
            "h2d_GB/s": round(h2d * e2e_steps / (e2e_ms / 1e3) / 1e9, 1),
            "windows": f"{n_win} windows of {e2e_steps} steps, alternating with the "
                       "serial schedule; median window",
            "window_ms_per_step": [round(t / e2e_steps, 3) for t in win_pipe],
            "window_last_step_copy_GB/s_in_out": rate_pipe,
            "serial": {"value": round(tok_step / (serial_ms / 1e3), 1),
                       "ms_per_step": round(serial_ms / e2e_steps, 3),
                       "window_ms_per_step": [round(t / e2e_steps, 3) for t in win_serial],
                       "window_last_step_copy_GB/s_in_out": rate_serial,
                       "schedule": "one step alone: copies in, kernels, copy out"}}
        hp.close()
        del hp, x_h, lg_h, ro_h, y_h, outs_h

    # other schedules of the same batch, and the decode step (after the e2e
    # measurement, so their allocations and graphs cannot affect it)
    overlap = chunk = decode = None
    if not args.no_extras and args.workload == "prefill":
        overlap = two_batch_overlap(args, ep, torch, dev, stream, inp, w, flush, dist)
        chunk = chunked_prefill(args, ep, torch, dev, stream, inp, w, flush, dist,
                                T=min(8192, max(8, inp["N"] // 4)))
        decode = decode_latency(args, ep, torch, dev, stream, flush) if rank == 0 else None

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    steps = args.steps
    tok = N * world
    ms_per_step = total_ms / steps
    value = tok * steps / (total_ms / 1e3)
    bm = byte_model(N, E, K, H, fp8=fp8, delivered=delivered)
    peak, peak_kind = measured_peaks()
    mean = {k: statistics.fmean(v) for k, v in stage.items()}
    kernels = {}
    if fused:  # one kernel for route + layout: report it as one stage
        mean["route_layout"] = mean.pop("route") + mean.pop("layout")
        bm["route_layout"] = bm["route"] + bm["layout"]
    for k in (["route_layout"] if fused else ["route", "layout"]) + ["dispatch", "combine"]:
        gbs = bm[k] / (mean[k] / 1e3) / 1e9
        kernels[k] = {"ms": round(mean[k], 4), "bytes": bm[k], "GB/s": round(gbs, 1),
                      "frac_of_measured": round(gbs / peak, 4),
                      "frac_of_8TBs": round(gbs / SPEC_HBM_GBS, 4)}
    # what bounds each kernel (ncu summaries in profiles/): routing is integer
    # compare-and-select work in the ALU pipe, the layout kernels are latency
    bounds = {"route": "alu", "layout": "latency", "route_layout": "alu",
              "dispatch": "hbm", "combine": "hbm"}
    for k in kernels:
        kernels[k]["bound"] = bounds[k]
    kernels["dispatch"]["GB/s_rowwise_accounting"] = round(
        bm["dispatch_rowwise"] / (mean["dispatch"] / 1e3) / 1e9, 1)
    dc_bytes = bm["dispatch"] + bm["combine"]
    dc_per = dc_ms / steps
    comb_gbs = bm["combine"] / (mean["combine"] / 1e3) / 1e9
    # the committed counters describe the full-size launch only
    full = not args.tokens_per_rank and args.workload == "prefill"
    traffic = ncu_traffic("combine", ["combine.cu"]) if full else None
    if full:  # the same kind of stored record for the FP8 dispatch launch
        kernels["dispatch"]["traffic"] = ncu_traffic("dispatch", ["dispatch.cu"])
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC if full else
                   f"{args.workload}: {describe_workload(w, N)}",
                   "R": w.R, "N": N, "E": E, "K": K, "H": H,
                   "layout": "contiguous" if layout == ep.EP_LAYOUT_CONTIG else
                   f"masked, capacity {cap}",
                   "dispatch_dtype": "fp8_e4m3_1x128" if fp8 else "bf16",
                   "rows_delivered": delivered,
                   "expert_renumbering": bool(w.relabel),
                   "step": ("route+layout (one fused kernel)" if fused else
                            "route, layout") + ", dispatch, combine",
                   "l2": "flushed between steps (512 MiB write, outside the step events)" +
                         ("; inputs (x 0.47 GB, y 3.76 GB) also exceed L2" if full else ""),
                   "parallelism": f"{world} independent replica(s), one per GPU"},
        "roofline": {"kernel": "combine", "bound": "hbm", "achieved": round(comb_gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(comb_gbs / peak, 4),
                     "peak_source": peak_kind, "traffic": traffic,
                     "traffic_note": "dram__bytes_read.sum + dram__bytes_write.sum per launch "
                                     "from a stored ncu capture of this kernel source "
                                     "(profiles/ncu_traffic.json: 16384 tokens, scaled by 2 "
                                     "to 32768), not measured in this run; null once the "
                                     "source has changed since the capture",
                     "algorithmic_bytes": bm["combine"]},
        "dispatch_combine": {"tokens_per_s": round(tok * steps / (dc_ms / 1e3), 1),
                             "ms": round(dc_per, 4),
                             "GB/s": round(dc_bytes / (dc_per / 1e3) / 1e9, 1),
                             "frac_of_measured": round(dc_bytes / (dc_per / 1e3) / 1e9 / peak, 4),
                             "frac_of_8TBs": round(dc_bytes / (dc_per / 1e3) / 1e9 / SPEC_HBM_GBS,
                                                   4)},
        "kernels": kernels,
        "kernels_note": f"per-kernel CUDA events over a separate pass of {n_bd} steps",
        "two_batch_overlap": overlap,
        "chunked_rounds": chunk,
        "decode_step": decode,
        "e2e": e2e_line,
        "gpu_launches": int(launches),
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 3),
    }
    if args.cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
    if dist is not None:
        dist.destroy_process_group()
    return line


def two_batch_overlap(args, ep, torch, dev, main_stream, inp, w, flush, dist):
    """The same batch as micro-batches of contiguous rank groups, each on its
    own stream (pipeline.two_batch_overlap): one micro-batch's latency-bound
    routing and layout overlap another's HBM-bound dispatch and combine.
    Even halves, and a one-rank first group (only its routing and layout are
    exposed)."""
    from combine_ep_route_topk_gb300 import pipeline as pl
    K, H, R = w.K, w.H, w.R
    comb = torch.empty(inp["N"], H, dtype=torch.bfloat16, device=dev)
    y = inp["y"]
    out = {}
    for name, groups in (("even_halves", [(0, R // 2), (R // 2, R)]),
                         ("first_rank_alone", [(0, 1), (1, R)])):
        mbs = pl.make_micro_batches(inp["logits"], inp["x"], inp["rank_offsets"], K,
                                    ep.EP_DTYPE_FP8_E4M3_B128, comb, rank_groups=groups)

        def step():
            pl.two_batch_overlap(mbs, K, ep.EP_DTYPE_FP8_E4M3_B128,
                                 lambda mb: y[mb.t0 * K:mb.t1 * K], main_stream)

        out[name] = _time_schedule(
            args, torch, main_stream, flush, dist, step, inp["N"],
            "micro-batches of ranks " + ", ".join(f"{a}..{b - 1}" for a, b in groups) +
            " on their own streams")
        del mbs
    return out


def chunked_prefill(args, ep, torch, dev, main_stream, inp, w, flush, dist, T=8192):
    """The same batch in ant-moving rounds of T tokens (pipeline.chunked): the
    dispatch buffer holds T*K rows instead of N*K.  Rounds in order with one
    buffer set, and alternating over two sets (and streams)."""
    from combine_ep_route_topk_gb300 import pipeline as pl
    K, H, E, R = w.K, w.H, w.E, w.R
    comb = torch.empty(inp["N"], H, dtype=torch.bfloat16, device=dev)
    offs = inp["rank_offsets"].cpu().tolist()
    ro_rounds = pl.chunk_rank_offsets(offs, inp["N"], T, dev)
    y = inp["y"]
    out = {}
    for sets in (1, 2):
        bufs = pl.make_chunk_buffers(T, E, K, H, R, ep.EP_DTYPE_FP8_E4M3_B128, dev, sets=sets)

        def step():
            pl.chunked(inp["logits"], inp["x"], offs, K, ep.EP_DTYPE_FP8_E4M3_B128, bufs,
                       lambda t0, n, o, sc, lay: y[t0 * K:(t0 + n) * K], comb,
                       ro_rounds=ro_rounds)

        res = _time_schedule(args, torch, main_stream, flush, dist, step, inp["N"],
                             f"rounds of {T} tokens, {sets} buffer set(s)" +
                             (" on alternating streams" if sets > 1 else ""))
        res["dispatch_buffer_bytes"] = sum(b.dispatch_bytes for b in
                                           (bufs if sets > 1 else [bufs]))
        res["dispatch_buffer_bytes_unchunked"] = inp["N"] * K * (H + H // 128 * 4)
        out["in_order" if sets == 1 else "alternating_2_sets"] = res
        del bufs
    return out


def _time_schedule(args, torch, main_stream, flush, dist, step, N, note):
    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize()
    steps = max(10, min(args.steps, 100))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    barrier(dist)
    for i in range(steps):
        flush.fill_((i + 3) & 0xFF)
        evs[i][0].record(main_stream)
        step()
        evs[i][1].record(main_stream)
    torch.cuda.synchronize()
    total = max_over_ranks(dist, sum(e[0].elapsed_time(e[1]) for e in evs))
    world = 1 if dist is None else dist.get_world_size()
    return {"tokens_per_s": round(N * world * steps / (total / 1e3), 1),
            "ms_per_step": round(total / steps, 4), "steps": steps, "note": note}


def decode_latency(args, ep, torch, dev, stream, flush):
    """Latency of one decode step (the low-latency, masked layout): 8 ranks x
    128 tokens, E=256, K=8, H=7168, capacity 128; route, layout, masked bf16
    dispatch and masked combine, in four arrangements: ep_route_dispatch
    (route, layout and dispatch in two launches) then ep_combine; four
    separate calls (the layout as one block per expert); the same with the
    one-cluster layout (EP_LAYOUT_SMALL=0 while the step is captured and
    launched); route + layout as the cooperative kernel (ep_route_layout).
    L2 flushed before every step."""
    from combine_ep_route_topk_gb300 import workloads as wl
    w = wl.WORKLOADS["decode"]
    inp = wl.make_inputs(w, seed=args.seed + 1, device=str(dev))
    N, E, K, H, R, cap = inp["N"], w.E, w.K, w.H, w.R, w.cap
    idx = torch.empty(N, K, dtype=torch.int32, device=dev)
    wt = torch.empty(N, K, dtype=torch.float32, device=dev)
    lay = ep.alloc_layout(N, E, K, R, cap, dev)
    ws = torch.empty(max(ep.ep_route_layout_workspace_size(N, E, K, R),
                         ep.ep_dispatch_layout_workspace_size(N, E, K, R)), dtype=torch.uint8,
                     device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty(E * cap, H, dtype=torch.bfloat16, device=dev)
    comb = torch.empty(N, H, dtype=torch.bfloat16, device=dev)

    ws_rd = torch.empty(ep.ep_route_dispatch_workspace_size(N, E, K, R), dtype=torch.uint8,
                        device=dev)

    def step(kind):
        if kind == "route_dispatch":  # ep_route_dispatch: two launches, then combine
            ep.ep_route_dispatch(inp["logits"], inp["rank_offsets"], inp["x"], K,
                                 ep.EP_LAYOUT_MASKED, cap, topk_idx=idx, topk_w=wt, lay=lay,
                                 out=out, workspace=ws_rd)
            ep.ep_combine(inp["y"], idx, wt, lay.pos, lay.expert_offsets, E, ep.EP_LAYOUT_MASKED,
                          cap, out=comb)
            return
        if kind == "fused_route_layout":
            ep.ep_route_layout(inp["logits"], inp["rank_offsets"], K, cap, topk_idx=idx,
                               topk_w=wt, out=lay, status=st, workspace=ws)
        else:
            ep.ep_route_topk(inp["logits"], K, topk_idx=idx, topk_w=wt)
            if kind == "cluster_layout":
                os.environ["EP_LAYOUT_SMALL"] = "0"
            try:
                ep.ep_dispatch_layout(idx, inp["rank_offsets"], E, cap, out=lay, workspace=ws)
            finally:
                os.environ.pop("EP_LAYOUT_SMALL", None)
        ep.ep_dispatch(inp["x"], idx, lay.pos, lay.expert_offsets, E, ep.EP_LAYOUT_MASKED,
                       cap, out=out)
        ep.ep_combine(inp["y"], idx, wt, lay.pos, lay.expert_offsets, E, ep.EP_LAYOUT_MASKED,
                      cap, out=comb)

    # L2 before each step: the 512 MiB write, then a 512 MiB read pass, so
    # the step starts with none of its inputs in L2 and with L2 holding clean
    # lines; with the write alone, the step would also write back up to
    # 129 MB of the flush's dirty lines, about half of its own traffic (the
    # default arrangement is timed that way too, for comparison)
    rd = torch.ones(512 << 20, dtype=torch.uint8, device=dev)

    def flush_l2(i, clean=True):
        flush.fill_(i & 0xFF)
        if clean:
            rd.view(torch.int32).amax()

    def graph_loop(step, flush_l2, m=20, replays=5):
        """Steps as a model's own graph would hold them: m of them captured
        in one graph, each after a clean L2 flush, with event-record nodes
        around each step, so that no step pays for a graph launch.  None
        when events cannot be recorded inside a graph here."""
        try:
            evs = [(torch.cuda.Event(enable_timing=True, external=True),
                    torch.cuda.Event(enable_timing=True, external=True)) for _ in range(m)]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(m):
                    flush_l2(i)
                    evs[i][0].record(stream)
                    step("route_dispatch")
                    evs[i][1].record(stream)
            ts = []
            for r in range(replays + 1):
                g.replay()
                torch.cuda.synchronize()
                if r:  # the first replay warms up
                    ts += [a.elapsed_time(b) * 1e3 for a, b in evs]
            del g
        except (RuntimeError, TypeError):
            return None
        ts.sort()
        mean = statistics.fmean(ts)
        return {"us_median": round(ts[len(ts) // 2], 2), "us_mean": round(mean, 2),
                "us_min": round(ts[0], 2), "tokens_per_s": round(N / (mean / 1e6), 1),
                "steps": len(ts),
                "how": f"{m} steps in one CUDA graph, each after the clean L2 flush, "
                       "timed by event-record nodes around the step (no graph launch "
                       "per step)"}

    res = {}
    for fused in ("route_dispatch", "separate", "cluster_layout", "fused_route_layout"):
        for i in range(3):
            step(fused)
        torch.cuda.synchronize()
        # the step captured once in a CUDA graph (the low-latency mode's
        # static shapes allow it), so the timing is the GPU's, not Python's
        # launch path; eager launches are timed too for comparison
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step(fused)
        modes = (("graph", "eager", "graph_l2_dirty") if fused in ("separate", "route_dispatch")
                 else ("graph", "eager"))
        for mode in modes:
            n = 100
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n)]
            for i in range(n):
                flush_l2(i, clean=mode != "graph_l2_dirty")
                evs[i][0].record(stream)
                if mode != "eager":
                    graph.replay()
                else:
                    step(fused)
                evs[i][1].record(stream)
            torch.cuda.synchronize()
            ts = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
            mean = statistics.fmean(ts)
            key = {"route_dispatch": "route_dispatch_then_combine_",
                   "fused_route_layout": "fused_route_layout_",
                   "cluster_layout": "separate_cluster_layout_",
                   "separate": "separate_route_layout_"}[fused] + mode
            # event times on this GPU come in steps of about 2 us: the mean of many
            # steps resolves finer than the median
            res[key] = {"us_median": round(ts[n // 2], 2), "us_mean": round(mean, 2),
                        "us_min": round(ts[0], 2),
                        "tokens_per_s": round(N / (mean / 1e6), 1)}
        del graph
        if fused == "route_dispatch":
            res["route_dispatch_then_combine_graph_loop"] = graph_loop(step, flush_l2)
    if int(st.item()) != 0:
        raise RuntimeError("route+layout kernel reported a barrier timeout")
    res["workload"] = "decode: 8 ranks x 128 tokens, E=256, K=8, H=7168, masked cap 128, bf16"
    res["l2"] = ("before each step: 512 MiB write then 512 MiB read (clean L2, no input "
                 "resident); *_l2_dirty: the write alone (the step also writes back the "
                 "flush's dirty lines)")
    return res


# ------------------------------------------------------------- CPU oracle --

def oracle_sample(workload: str, tokens_per_rank: int, seed: int):
    """The workload's recipe at a bounded size: its R ranks x tokens_per_rank
    tokens (0: the workload's own batch sizes), same E/K/H, distributions,
    layout and dtypes."""
    import numpy as np
    import torch
    from combine_ep_route_topk_gb300 import workloads as wl
    w = wl.WORKLOADS[workload]
    if tokens_per_rank:
        w = w.scaled(batch=("fixed", tokens_per_rank))
    inp = wl.make_inputs(w, seed=seed)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    return w, dict(logits=inp["logits"].numpy(), ro=inp["rank_offsets"].numpy(),
                   x=bits(inp["x"]), y=bits(inp["y"]), N=inp["N"])


def oracle_step(w, s):
    """The oracle's whole path for one sample: route (with the balanced
    renumbering measured on the sample when the workload uses it), layout,
    dispatch, combine."""
    import oracle
    cap = w.cap if w.layout == oracle.LAYOUT_MASKED else 0
    emap = None
    if w.relabel:
        i0, _ = oracle.route_topk(s["logits"], w.K)
        emap = oracle.balance_map(oracle.layout(i0, s["ro"], w.E)["counts"])
    idx, wt = oracle.route_topk(s["logits"], w.K, expert_map=emap)
    lay = oracle.layout(idx, s["ro"], w.E, cap)
    oracle.dispatch(s["x"], idx, lay["pos"], lay["expert_offsets"], w.E, layout=w.layout,
                    cap=cap, dtype=w.dtype)
    oracle.combine(s["y"], idx, wt, lay["pos"], lay["expert_offsets"], w.E, layout=w.layout,
                   cap=cap)


def host_cpu():
    """The host CPU as /proc/cpuinfo names it (the model name on x86; the
    implementer and part numbers on Arm), the machine type and the core count."""
    import platform
    model = ""
    try:
        info = {}
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = (t.strip() for t in line.split(":", 1))
                    info.setdefault(k, v)
        model = info.get("model name") or (
            f"implementer {info['CPU implementer']} part {info['CPU part']}"
            if "CPU implementer" in info and "CPU part" in info else "")
    except OSError:
        pass
    return {"cpu": model or platform.processor() or "unknown", "machine": platform.machine(),
            "host_cores": os.cpu_count()}


def cpu_baseline(budget_s: float = 12.0):
    """The oracle as it stands, one thread, on sub-batches of the prefill
    workload (8 ranks x 256 tokens each) until about budget_s of CPU work."""
    per_rank = 256
    w, s = oracle_sample("prefill", per_rank, seed=1000)
    total_tok, total_s, reps = 0, 0.0, 0
    while total_s < budget_s and reps < 64:
        t0 = time.perf_counter()
        oracle_step(w, s)
        total_s += time.perf_counter() - t0
        total_tok += s["N"]
        reps += 1
    return {"value": round(total_tok / total_s, 1), "unit": "tokens/s", "cores": 1,
            "kind": "oracle", **host_cpu(),
            "sample": f"one sub-batch of the prefill workload (8 ranks x {per_rank} tokens, "
                      f"E=256, K=8, H=7168; route, layout, FP8 dispatch, combine) run {reps} "
                      f"times: {total_tok} tokens in {total_s:.1f} s, single-threaded"}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    from combine_ep_route_topk_gb300 import workloads as wl
    w0 = wl.WORKLOADS[args.workload]
    # per-token cost from a small calibration sample, then a per-step sample
    # sized so warm-up + steps take about 90 s of CPU
    wc, sc = oracle_sample(args.workload, 8, seed=args.seed)
    t0 = time.perf_counter()
    oracle_step(wc, sc)
    per_token_s = max(1e-7, (time.perf_counter() - t0) / sc["N"])
    per_rank = int(90.0 / (per_token_s * max(1, args.steps + args.warmup)) / w0.R)
    full = wl.make_inputs(w0, seed=args.seed, with_y=False)["N"] // w0.R
    if per_rank >= full:
        per_rank = 0  # the workload's own batch fits the budget
    else:
        per_rank = max(4, per_rank)
    w, s = oracle_sample(args.workload, per_rank, seed=args.seed)
    for _ in range(args.warmup):
        oracle_step(w, s)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(w, s)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = s["N"] * args.steps / tot
    sample = (f"each step: the whole batch ({s['N']} tokens)" if not per_rank else
              f"each step: {w.R} ranks x {per_rank} tokens ({s['N']} tokens) of the workload")
    desc = WORKLOAD_DESC if args.workload == "prefill" else \
        f"{args.workload}: {describe_workload(w0, full * w0.R)}"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": desc, "step": "route+layout+dispatch+combine",
                   "sample_per_step": sample},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": 1,
                         "kind": "oracle", "sample": sample, **host_cpu()},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--fused", action="store_true",
                    help="route + layout as the one cooperative kernel (ep_route_layout)")
    ap.add_argument("--workload", default="prefill",
                    choices=["toy", "lumpy", "decode", "prefill", "skew"],
                    help="the workload a step runs (default: prefill, the headline)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end host-buffer measurement (its pipeline holds "
                         "about 11 GB more on the device); for profiling runs")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the overlap, chunked and decode measurements (profiling)")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the decode step (for profiling its kernels)")
    ap.add_argument("--tokens-per-rank", type=int, default=0,
                    help="run a smaller case of the workload (default: the full 4096)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.decode_only:
        import torch
        import combine_ep_route_topk_gb300 as ep
        torch.cuda.set_device(local)
        dev = torch.device("cuda", local)
        stream = torch.cuda.Stream(device=dev)
        torch.cuda.set_stream(stream)
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        line = {"decode_step": decode_latency(args, ep, torch, dev, stream, flush)}
    elif args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_ours(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
