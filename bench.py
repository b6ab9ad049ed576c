#!/usr/bin/env python
"""Benchmark of the multi-LoRA SGMV hot path on one B300 per process.

One step = lora_segment (per-token adapter ids -> segments) + sgmv_fused (or
sgmv_multi) over one batch, inputs resident in HBM.  Default workload:
Llama2-7B decode projection 4096 -> 4096, r = 16, 32 tokens, each token a
different adapter of a 64-adapter pool (mixed adapters), s = 1.

Prints one JSON line.  `value` is microseconds per step (lower is better),
timed with CUDA events around a CUDA graph of K steps that rotates over
input copies whose touched bytes exceed twice the L2, so every step reads
HBM.  `roofline` grades the fused kernel against measured HBM bandwidth;
`e2e` times the same step through the Python API from pinned host buffers;
`cpu_baseline` times the CPU oracle (test infrastructure) on host cores.

--impl reference times the CPU oracle as the reference arm.
Multi-GPU (torchrun): every rank runs its own replica of the workload
(independent batches, no data-path collective); timing is the max over ranks.
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import WORKLOADS, distinct_ids, make_inputs  # noqa: E402

DEFAULT_WORKLOAD = "7b_proj_distinct"
# streams taking the end-to-end steps in turn (1 / 2 / 3 / 4 / 6 measured 50-73 / 31-39 /
# 24-29 / 22.3-22.9 / 23.3-24.0 us per step on the 7B projection: from 4 the host-to-device
# copies, not the host enqueue, bound it)
E2E_STREAMS = 4
METRIC = "fused SGMV µs & % HBM roofline, Llama2-7B dims r=16 bs32 mixed adapters"
L2_BYTES = 126 * 2 ** 20
FALLBACK_HBM_GBS = 6400.0


# ----------------------------------------------------------------- accounting

def algorithmic_bytes(wl, ids: np.ndarray) -> int:
    """Unique bytes one call must move: A and B slabs of every distinct valid
    adapter of every projection, each distinct x once, y read and written."""
    valid = ids[(ids >= 0) & (ids < wl.P)]
    D = int(np.unique(valid).size)
    n = int(ids.size)
    w = sum((p.h_in * wl.r + wl.r * p.h_out) * 2 for p in wl.projs) * D
    xs = {}
    for p in wl.projs:
        xs[p.x_key] = p.h_in
    x = sum(n * h * 2 for h in xs.values())
    y = sum(n * p.h_out * 2 * 2 for p in wl.projs)
    return w + x + y


def flops(wl, ids: np.ndarray) -> int:
    n = int(((ids >= 0) & (ids < wl.P)).sum())
    return sum(2 * n * wl.r * (p.h_in + p.h_out) for p in wl.projs)


def dominant_kernel(wl) -> str:
    """The kernel that does the call's work: the tensor-tile kernel when
    segments are long on average (prefill), else the split-K decode kernel.
    Mirrors the library's dispatch rule (tokens per possible segment >= 64 or
    at least 512 tokens, r in {16, 32, 64}); the measured time covers the whole
    call either way."""
    n = wl.n
    if wl.r in (16, 32, 64) and n >= 64 and (n // max(1, min(n, wl.P)) >= 64 or n >= 512):
        return "sgmv_tc_kernel"
    return "sgmv_cc_kernel"


def one_launch(wl) -> bool:
    """True when the library segments the batch inside the SGMV launch (a
    small decode-like batch): mirrors its rule (n <= 128, P <= 1024, no
    tensor-tile path)."""
    return wl.n <= 128 and wl.P <= 1024 and dominant_kernel(wl) == "sgmv_cc_kernel"


def launches_per_step(wl) -> int:
    if one_launch(wl):
        return 1
    return 3 if dominant_kernel(wl) == "sgmv_tc_kernel" else 2


def config_of(wl, ids: np.ndarray, world: int) -> dict:
    """The workload description both arms print (identical keys and values)."""
    return {"workload": wl.description, "name": wl.name, "n_tokens": wl.n, "rank": wl.r, "pool": wl.P,
            "distinct_adapters": int(np.unique(ids[(ids >= 0) & (ids < wl.P)]).size),
            "projections": len(wl.projs), "parallelism": "replicas" if world > 1 else "single"}


def n_copies(step_bytes: int, max_copies: int) -> int:
    """Independent input copies the timed graphs rotate over so that the bytes
    touched per cycle exceed 2.2x the L2 (every step reads HBM); one copy when
    a single step already moves more than four L2s."""
    if step_bytes > 4 * L2_BYTES:
        return 1
    return max(2, min(max_copies, int(np.ceil(2.2 * L2_BYTES / step_bytes))))


def bf16_peaks():
    """(sustained, burst) dense bf16 TFLOP/s from MEASURED_PEAKS.json, else the
    fallback figures (1400, 1800)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), float(d["bf16_tflops"])
    except Exception:
        return 1400.0, 1800.0


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {"sgmv_cc_kernel": ("sgmv_cc.cu", "seg_warp.cuh", "ptx.cuh"), "sgmv_tc_kernel": ("sgmv_tc.cu", "ptx.cuh")}


def _code_only(text: str) -> str:
    """Source text without comments and with whitespace collapsed (a comment
    edit leaves the kernel, and so its recorded counters, unchanged)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_hash(kernel: str) -> str:
    """Hash of the device code of `kernel` (its .cu file and the device headers it includes)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "adapter_gemm_02_b300", "csrc", name), encoding="utf-8") as fh:
            h.update(name.encode())
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    want = source_hash(kernel)
    for line in open(path):
        parts = line.split()
        if len(parts) == 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload \
                and parts[2] == want:
            return int(parts[3])
    return None


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        pw = [float(r[4]) for r in rows if r[4].replace(".", "", 1).isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for nm, val in zip(names, r[6:10]):
                if val.lower() == "active":
                    reasons.add(nm)
        loaded = [s for s, p in zip(sm, pw)] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ----------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, world: int) -> float:
    """Max over ranks (gloo or nccl); identity for one process."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ----------------------------------------------------------------- oracle timing

def time_oracle(wl, inp_cpu, seconds: float, threads: int, max_calls: int = 10 ** 9):
    """Seconds per full call of the CPU oracle (segmentation + per-token
    SGMV over every projection) on this host, over max_calls calls or until
    `seconds` have passed (whichever comes first; at least one call);
    returns (s_per_call, calls)."""
    import oracle  # test infrastructure: the CPU baseline leg only

    ids = inp_cpu.ids.numpy()
    x = {k: oracle.bits(v) for k, v in inp_cpu.x.items()}
    A = [oracle.bits(a) for a in inp_cpu.A]
    B = [oracle.bits(b) for b in inp_cpu.B]
    Y = [oracle.bits(y) for y in inp_cpu.y0]
    calls = 0
    t0 = time.perf_counter()
    while True:
        oracle.lora_segment_ref(ids, wl.P)
        for i, p in enumerate(wl.projs):
            oracle.sgmv_ref(x[p.x_key], A[i], B[i], ids, wl.scale, Y[i], threads=threads)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds or calls >= max_calls:
            return el / calls, calls


def run_reference(args) -> None:
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import torch

    wl = WORKLOADS[args.workload]
    threads = os.cpu_count() or 1
    inp = make_inputs(wl, "cpu")
    # warm-up: W calls and at least 2 s of calls (the OpenMP pool and the
    # caches reach steady state), then K timed calls (fewer if they pass the
    # time cap: the oracle of a prefill batch takes seconds per call)
    time_oracle(wl, inp, args.ref_seconds / 4, threads, max_calls=args.warmup)
    time_oracle(wl, inp, min(2.0, args.ref_seconds / 4), threads)
    per, calls = time_oracle(wl, inp, args.ref_seconds, threads, max_calls=max(1, args.steps))
    us = per * 1e6
    out = {
        "impl": "reference", "metric": METRIC, "value": round(us, 3), "unit": "us", "n_gpus": args.gpus,
        "steps": calls, "warmup": args.warmup, "ms_per_step": round(per * 1e3, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_of(wl, wl.ids(), world),
        "cpu_baseline": {"value": round(us, 3), "unit": "us", "cores": threads, "kind": "oracle",
                         "sample": f"{calls} full calls (segmentation + per-token fp32 SGMV, all tokens)"},
        "e2e": {"value": round(us, 3), "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "torch": torch.__version__,
    }
    print(json.dumps(out), flush=True)


# ----------------------------------------------------------------- our arm

def run_ours(args) -> None:
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    import adapter_gemm_02_b300 as lsg

    wl = WORKLOADS[args.workload]
    K, Wm = args.steps, args.warmup

    ids_np = wl.ids()
    abytes = algorithmic_bytes(wl, ids_np)
    nflop = flops(wl, ids_np)
    copy_bytes = abytes  # bytes one step touches
    NB = n_copies(copy_bytes, args.max_copies)

    copies = []
    for c in range(NB):
        inp = make_inputs(wl, dev, copy=c)
        seg = lsg.Segments.empty(wl.n, wl.P, dev)
        projs = [(inp.x[p.x_key], inp.A[i], inp.B[i], inp.y0[i], wl.scale) for i, p in enumerate(wl.projs)]
        copies.append((inp, seg, projs, lsg.make_projs(projs)))
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(k):
        # the whole path in one call: segmentation (inside the SGMV launch for
        # small batches), gather, shrink, expand
        inp, seg, projs, cproj = copies[k % NB]
        lsg.sgmv_multi_segment(projs, inp.ids, wl.P, out=seg, err_flag=err, c_projs=cproj)

    def fused_only(k):
        inp, seg, projs, cproj = copies[k % NB]
        if len(projs) == 1:
            x, A, B, y, s = projs[0]
            lsg.sgmv_fused(x, A, B, seg, y, s, err_flag=err)
        else:
            lsg.sgmv_multi(projs, seg, err_flag=err, c_projs=cproj)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for k in range(max(Wm, NB)):
            step(k)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flag {int(err.item())}"

    # graph of K steps (value) ...
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=side):
        for k in range(K):
            step(k)
    # ... graph of K fused launches alone (kernel time per launch) and of K
    # segmentation launches alone (breakdown)
    g_kern = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_kern, stream=side):
        for k in range(K):
            fused_only(k)
    g_seg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_seg, stream=side):
        for k in range(K):
            inp, seg, _, _ = copies[k % NB]
            lsg.lora_segment(inp.ids, wl.P, out=seg, err_flag=err)
    torch.cuda.synchronize()

    # end to end from pinned host memory through the C-ABI host-step call
    # (measured before the clock sampler starts: once nvidia-smi has run in
    # this process's lifetime, host-side CUDA calls were measured to cost
    # 2-4x more, which this host-bound loop would inherit).
    # E2E_STREAMS pipelines (stream, pinned host buffers, device workspace)
    # take the steps in turn, so one step's uploads overlap the previous
    # steps' kernels and downloads; every step still copies its own inputs in
    # and its y out.
    e2e = None
    if not args.no_e2e:
        inp0 = copies[0][0]
        pipes = []
        for _ in range(E2E_STREAMS):
            h_ids = inp0.ids.cpu().pin_memory()
            h_x = {k: v.cpu().pin_memory() for k, v in inp0.x.items()}
            h_y = [y.cpu().pin_memory() for y in inp0.y0]
            hprojs = [(h_x[p.x_key], inp0.A[i], inp0.B[i], h_y[i], wl.scale) for i, p in enumerate(wl.projs)]
            chp = lsg.make_host_projs(hprojs)
            ws = torch.empty(lsg.sgmv_multi_host_workspace_bytes(chp, wl.n, wl.P), dtype=torch.uint8, device=dev)
            pipes.append((torch.cuda.Stream(dev), h_ids, hprojs, chp, ws))
        bi = h_ids.numel() * 4 + sum(v.numel() * 2 for v in h_x.values()) + sum(y.numel() * 2 for y in h_y)
        bo = sum(y.numel() * 2 for y in h_y)

        def e2e_step(k, n_pipes):
            st, h_ids, hprojs, chp, ws = pipes[k % n_pipes]
            lsg.sgmv_multi_host(hprojs, h_ids, workspace=ws, err_flag=err, stream=st, c_projs=chp)

        def e2e_time(n_pipes, reps=3):
            """Median over `reps` timed runs of K steps (device time, host enqueue time)."""
            main = torch.cuda.current_stream()
            for k in range(max(Wm, 8 * n_pipes)):
                e2e_step(k, n_pipes)
            torch.cuda.synchronize()
            barrier(world)
            dev_us, host_us = [], []
            for _ in range(reps):
                f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                f0.record(main)
                for st, *_ in pipes[:n_pipes]:
                    st.wait_event(f0)
                h0 = time.perf_counter()
                for k in range(K):
                    e2e_step(k, n_pipes)
                host_us.append((time.perf_counter() - h0) / K * 1e6)
                for st, *_ in pipes[:n_pipes]:
                    ev = torch.cuda.Event()
                    ev.record(st)
                    main.wait_event(ev)
                f1.record(main)
                torch.cuda.synchronize()
                dev_us.append(f0.elapsed_time(f1) / K * 1e3)
            barrier(world)
            return reduce_max(statistics.median(dev_us), world), statistics.median(host_us)

        e2e_us, host_us = e2e_time(E2E_STREAMS)
        two_us, _ = e2e_time(2)
        serial_us, _ = e2e_time(1)
        e2e = {"value": round(e2e_us, 3), "unit": "us", "h2d_bytes_per_step": int(bi),
               "d2h_bytes_per_step": int(bo), "host_enqueue_us_per_step": round(host_us, 2),
               "one_stream_us": round(serial_us, 3), "two_streams_us": round(two_us, 3),
               "path": f"sgmv_multi_host (C ABI): H2D of ids, x, y0 from pinned host memory, segmentation, SGMV, "
                       f"D2H of y, one library call per step; {E2E_STREAMS} streams take the steps in turn, each "
                       f"with its own pinned buffers and workspace; median of 3 timed runs of K steps (one_stream_us / "
                       f"two_streams_us: 1 or 2 streams)"}

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    # settle clocks under load (untimed), then the timed region
    t_end = time.perf_counter() + args.settle
    while time.perf_counter() < t_end:
        g_step.replay()
        torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g_step.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    ms_total = e0.elapsed_time(e1)
    ms_step = reduce_max(ms_total / K, world)

    if one_launch(wl):
        # the step is one launch of the SGMV kernel (segmentation inside)
        kern_avg_ms = reduce_max(_time_graph_median(g_step, side)[0] / K, world)
        seg_avg_ms = None
    else:
        kern_avg_ms = reduce_max(_time_graph_median(g_kern, side)[0] / K, world)
        seg_avg_ms = reduce_max(_time_graph_median(g_seg, side)[0] / K, world)
    clocks = sampler.stop()
    assert int(err.item()) == 0, f"device error flag {int(err.item())}"

    # mixed vs single adapter on the same shape (Punica: almost no difference)
    mixed = None
    if args.workload.startswith("7b_proj_") and not args.no_mixed:
        mixed = {"how": "us per step (segment + fused, one call); median of 7 replays of a K-step graph after "
                        "0.2 s of replays; [min, max] of the 7 beside it"}
        for pat in ("same", "zipf", "distinct"):
            med, lo, hi = _time_variant(f"7b_proj_{pat}", K, Wm, dev, lsg, args.max_copies)
            mixed[pat] = round(med, 3)
            mixed[pat + "_range"] = [round(lo, 3), round(hi, 3)]
        mixed["distinct_over_same"] = round(mixed["distinct"] / mixed["same"], 3)
        mixed["zipf_over_same"] = round(mixed["zipf"] / mixed["same"], 3)

    peak, peak_kind = hbm_peak()
    achieved = abytes / (kern_avg_ms * 1e-3) / 1e9
    kname = dominant_kernel(wl)
    traffic = recorded_traffic(kname, wl.name)
    out = {
        "metric": METRIC, "value": round(ms_step * 1e3, 3), "unit": "us", "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": round(ms_step, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(wl, ids_np, world),
        "timing": {"l2": f"rotating {NB} input copies (x, ids, y, pool); {NB * copy_bytes / L2_BYTES:.1f}x L2 "
                         "touched per cycle",
                   "value": "CUDA graph of K steps, CUDA events around one replay after 0.5 s of replays",
                   "kernel": "median of 7 replays of a K-launch graph"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": peak_kind,
                     "kernel": kname, "kernel_us": round(kern_avg_ms * 1e3, 3),
                     "algorithmic_bytes_per_launch": int(abytes), "flops_per_launch": int(nflop),
                     "tflops": round(nflop / (kern_avg_ms * 1e-3) / 1e12, 4)},
        "breakdown_us": ({kname + " (segmentation inside)": round(kern_avg_ms * 1e3, 3),
                          "how": "one launch per step: the step graph, events around the replay, / K"}
                         if seg_avg_ms is None else
                         {"lora_segment": round(seg_avg_ms * 1e3, 3), kname: round(kern_avg_ms * 1e3, 3),
                          "how": "graph of K launches of that kernel alone, events around the replay, / K"}),
        "gpu_launches": launches_per_step(wl) * K,
        "clocks": clocks,
        "e2e": e2e,
    }
    if mixed is not None:
        out["mixed_vs_single_us"] = mixed
    if not args.no_per_config and world == 1:
        out["per_config"] = per_config(K, Wm, dev, lsg, args.max_copies, peak)
    if not args.no_batch_curve and world == 1:
        out["batch_curve_us"] = batch_curve(K, Wm, dev, lsg, args.max_copies)
    if not args.no_backbone and world == 1:
        out["backbone_fused"] = backbone_fused(Wm, dev, lsg, bf16_peaks())
    if not args.no_slots and world == 1:
        out["slot_pool_us"] = slots_measure(K, Wm, dev, lsg, args.max_copies, peak)
        out["pool_loader"] = pool_loader_measure(g_step, K, dev, lsg)
    if rank == 0 and world == 1 and not args.no_cpu:
        threads = os.cpu_count() or 1
        inp_cpu = make_inputs(wl, "cpu")
        per, calls = time_oracle(wl, inp_cpu, args.cpu_seconds, threads)
        out["cpu_baseline"] = {"value": round(per * 1e6, 3), "unit": "us", "cores": threads, "kind": "oracle",
                               "sample": f"{calls} full calls of the workload in {args.cpu_seconds:.0f} s "
                                         "(segmentation + per-token fp32 SGMV, all tokens)"}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def _time_graph_median(g, stream, reps: int = 7, settle_s: float = 0.0):
    """(median, min, max) milliseconds of one replay of graph `g` over `reps`
    replays, each timed with CUDA events on the stream it replays on (after
    one untimed replay, and `settle_s` seconds of untimed replays)."""
    import torch

    times = []
    with torch.cuda.stream(stream):
        g.replay()
        stream.synchronize()
        t_end = time.perf_counter() + settle_s
        while time.perf_counter() < t_end:
            g.replay()
            stream.synchronize()
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            stream.synchronize()
            times.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    return statistics.median(times), min(times), max(times)


def _time_variant(name, K, Wm, dev, lsg, max_copies):
    """Microseconds per step (segment + fused) of another id pattern."""
    import torch

    wl = WORKLOADS[name]
    ids_np = wl.ids()
    NB = n_copies(algorithmic_bytes(wl, ids_np), max_copies)
    copies = []
    for c in range(NB):
        inp = make_inputs(wl, dev, copy=c)
        copies.append((inp, lsg.Segments.empty(wl.n, wl.P, dev)))
    side = torch.cuda.Stream(dev)

    def step(k):
        inp, seg = copies[k % NB]
        lsg.sgmv_fused_segment(inp.x["x"], inp.A[0], inp.B[0], inp.ids, inp.y0[0], wl.scale, out=seg)

    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for k in range(max(Wm, NB)):
            step(k)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for k in range(K):
            step(k)
    med, lo, hi = _time_graph_median(g, side, reps=7, settle_s=0.2)
    del g, copies
    torch.cuda.empty_cache()
    return med / K * 1e3, lo / K * 1e3, hi / K * 1e3


def _time_ids(wl, ids, K, Wm, dev, lsg, max_copies):
    """Microseconds per step (segment + fused) of projection 0 of `wl` on the
    given adapter ids (inputs rotated over copies that exceed twice the L2)."""
    import torch

    ids = np.asarray(ids, np.int32)
    NB = n_copies(algorithmic_bytes(wl, ids), max_copies)
    copies = []
    for c in range(NB):
        inp = make_inputs(wl, dev, copy=c, ids=ids)
        copies.append((inp, lsg.Segments.empty(ids.size, wl.P, dev)))
    p0 = wl.projs[0]
    side = torch.cuda.Stream(dev)

    def step(k):
        inp, seg = copies[k % NB]
        lsg.sgmv_fused_segment(inp.x[p0.x_key], inp.A[0], inp.B[0], inp.ids, inp.y0[0], wl.scale, out=seg)

    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for k in range(max(Wm, NB)):
            step(k)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for k in range(K):
            step(k)
    t = _time_graph_median(g, side, reps=5)[0] / K * 1e3
    del g, copies
    torch.cuda.empty_cache()
    return round(t, 3)


def _time_slots(h_in, h_out, ids, rank_of, n_slots, r_max, ranks, K, Wm, dev, lsg, max_copies, name):
    """Microseconds per step (segment + sgmv_multi_slots, one projection)."""
    import torch
    from workloads import make_slot_inputs

    P = len(rank_of)
    used = np.unique(ids)
    bytes_ = int(sum((h_in + h_out) * 2 * int(rank_of[a]) for a in used) + ids.size * (h_in + 2 * h_out) * 2)
    NB = n_copies(bytes_, max_copies)
    copies = []
    for c in range(NB):
        si = make_slot_inputs(h_in, h_out, ids, rank_of, n_slots, r_max, dev, copy=c, name=name)
        tab = lsg.SlotTable(si.slot_of, si.rank_of, n_slots, r_max, lsg.rank_mask(ranks))
        cp = lsg.make_slot_projs([(si.x, si.A_arena, si.B_arena, si.y0, 1.0)], tab)
        copies.append((si, tab, cp, lsg.Segments.empty(ids.size, P, dev)))
    side = torch.cuda.Stream(dev)

    def step(k):
        si, tab, cp, seg = copies[k % NB]
        lsg.lora_segment(si.ids, P, out=seg)
        lsg.sgmv_multi_slots([(si.x, si.A_arena, si.B_arena, si.y0, 1.0)], tab, seg, c_projs=cp)

    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for k in range(max(Wm, NB)):
            step(k)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for k in range(K):
            step(k)
    t = _time_graph_median(g, side, reps=5)[0] / K * 1e3
    del g, copies
    torch.cuda.empty_cache()
    return round(t, 3), bytes_


def slots_measure(K, Wm, dev, lsg, max_copies, peak):
    """Slot arenas (capacity r=64, 96 slots, pool of 64 adapters) on the
    Llama2-7B decode projection 4096->4096, 32 tokens of 32 distinct adapters:
    ranks 8/16/32/64 mixed in one launch, against the same batch with every
    adapter at r=16 through the slot table (one-rank kernel)."""
    P, n, n_slots, r_max = 64, 32, 96, 64
    ids = np.asarray(distinct_ids(n, P, seed=0), np.int32)
    mixed_r = np.array([(8, 16, 32, 64)[a % 4] for a in range(P)], np.int32)
    out = {"workload": "Llama2-7B decode projection 4096->4096, 32 tokens, 32 distinct adapters of 64, "
                       "96 slots of capacity r=64"}
    us, b = _time_slots(4096, 4096, ids, mixed_r, n_slots, r_max, (8, 16, 32, 64), K, Wm, dev, lsg, max_copies,
                        "slots_mixed")
    out["mixed_ranks_8_16_32_64"] = {"us": us, "algorithmic_bytes": b, "gbs": round(b / us / 1e3, 1),
                                     "frac_of_measured_hbm": round(b / us / 1e3 / peak, 4)}
    us16, b16 = _time_slots(4096, 4096, ids, np.full(P, 16, np.int32), n_slots, r_max, (16,), K, Wm, dev, lsg,
                            max_copies, "slots_r16")
    out["all_rank_16"] = {"us": us16, "algorithmic_bytes": b16, "gbs": round(b16 / us16 / 1e3, 1),
                          "frac_of_measured_hbm": round(b16 / us16 / 1e3 / peak, 4)}
    return out


def pool_loader_measure(g_step, K, dev, lsg, n_layers=32, reps=5):
    """Loading one Llama2-7B adapter (r=16, 32 layers x 7 projections: 224 A
    and 224 B matrices, 80 MB) from pinned host memory into free slots of the
    layers' arenas (lora_slot_copy + lora_slot_assign on a loader stream), as
    the pages' on-demand loads; alone, and while the bench's step graph runs
    on the compute stream."""
    import torch
    from workloads import llama_projs

    r, r_max, n_slots, P = 16, 16, 4, 64
    projs = llama_projs("7b")
    arenas, shapes = [], []
    for _ in range(n_layers):
        for pr in projs:
            arenas.append((torch.empty(n_slots, pr.h_in * r_max, dtype=torch.bfloat16, device=dev),
                           torch.empty(n_slots, r_max * pr.h_out, dtype=torch.bfloat16, device=dev)))
            shapes.append((pr.h_in, pr.h_out))
    total = sum(hi * r + r * ho for hi, ho in shapes)
    host = torch.randn(total, dtype=torch.float32).to(torch.bfloat16).pin_memory()
    srcs, off = [], 0
    for (Aa, Ba), (hi, ho) in zip(arenas, shapes):
        A_src = host[off: off + hi * r].view(hi, r)
        off += hi * r
        B_src = host[off: off + r * ho].view(r, ho)
        off += r * ho
        srcs.append((Aa, Ba, A_src, B_src))
    c_srcs = lsg.make_slot_srcs(srcs, r_max)
    table = lsg.SlotTable(torch.full((P,), -1, dtype=torch.int32, device=dev),
                          torch.zeros(P, dtype=torch.int32, device=dev), n_slots, r_max, lsg.rank_mask([r]))
    loader = torch.cuda.Stream(dev)
    compute = torch.cuda.current_stream()

    def load(i):
        lsg.lora_slot_copy(None, n_slots, r_max, i % n_slots, r, stream=loader, c_srcs=c_srcs)
        lsg.lora_slot_assign(table, i % P, i % n_slots, r, stream=loader)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    load(0)
    torch.cuda.synchronize()
    alone, host_ms = [], []
    for i in range(reps):
        e0, e1 = ev(), ev()
        e0.record(loader)
        t0 = time.perf_counter()
        load(i + 1)
        host_ms.append((time.perf_counter() - t0) * 1e3)
        e1.record(loader)
        torch.cuda.synchronize()
        alone.append(e0.elapsed_time(e1))
    # the step graph alone, then with a load issued right after it
    f0, f1 = ev(), ev()
    f0.record(compute)
    g_step.replay()
    f1.record(compute)
    torch.cuda.synchronize()
    step_alone = f0.elapsed_time(f1) / K * 1e3
    f0, f1, e0, e1 = ev(), ev(), ev(), ev()
    f0.record(compute)
    g_step.replay()
    f1.record(compute)
    e0.record(loader)
    load(reps + 1)
    e1.record(loader)
    torch.cuda.synchronize()
    step_during = f0.elapsed_time(f1) / K * 1e3
    med = float(np.median(alone))
    return {"adapter": "Llama2-7B, r=16, 32 layers x 7 projections", "bytes": int(total * 2),
            "copies": 2 * len(srcs), "load_ms": round(med, 3), "gbs": round(total * 2 / med / 1e6, 1),
            "host_enqueue_ms": round(float(np.median(host_ms)), 3),
            "load_ms_during_steps": round(e0.elapsed_time(e1), 3),
            "step_us_alone": round(step_alone, 3), "step_us_during_load": round(step_during, 3),
            "how": "pinned host -> slot arenas, one cudaMemcpyAsync per matrix on a loader stream, then the "
                   "table entry; CUDA events on the loader and compute streams"}


PER_CONFIG = ("7b_layer", "13b_prefill", "13b_prefill_interleaved", "70b_decode_r8", "70b_decode_r16",
              "70b_decode_r32", "70b_decode_r64")


def per_config(K, Wm, dev, lsg, max_copies, peak):
    """Times and roofline fractions of the multi-projection workloads (the
    Llama2-7B decode layer, the Llama2-13B prefill batch, the Llama2-70B
    decode batches at ranks 8-64), each with its own L2 rotation.
    step_us: one sgmv_multi_segment call (segmentation + SGMV); sgmv_us: the
    SGMV launches alone (segmentation given); segment_us: lora_segment alone
    (n ids, P adapters); kernel_us: the step when it is
    one launch, else the SGMV launches.  Each is the median of 7 replays of a
    K-call graph, timed with CUDA events on the replay stream."""
    import torch

    out = {"how": "median of 7 replays of a K-call graph (CUDA events on the replay stream); frac = "
                  "algorithmic bytes / kernel_us / measured HBM peak"}
    for name in PER_CONFIG:
        wl = WORKLOADS[name]
        ids = wl.ids()
        ab, nf = algorithmic_bytes(wl, ids), flops(wl, ids)
        NB = n_copies(ab, max_copies)
        copies = []
        for c in range(NB):
            inp = make_inputs(wl, dev, copy=c)
            projs = [(inp.x[p.x_key], inp.A[i], inp.B[i], inp.y0[i], wl.scale) for i, p in enumerate(wl.projs)]
            copies.append((inp, lsg.Segments.empty(wl.n, wl.P, dev), projs, lsg.make_projs(projs)))
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        ws_bytes = lsg.lora_segment_workspace_bytes(wl.n, wl.P)
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) if ws_bytes else None
        side = torch.cuda.Stream(dev)

        def step(k):
            inp, seg, projs, cp = copies[k % NB]
            lsg.sgmv_multi_segment(projs, inp.ids, wl.P, out=seg, workspace=ws, err_flag=err, c_projs=cp)

        def sgmv(k):
            inp, seg, projs, cp = copies[k % NB]
            lsg.sgmv_multi(projs, seg, err_flag=err, c_projs=cp)

        def segment(k):
            inp, seg, projs, cp = copies[k % NB]
            lsg.lora_segment(inp.ids, wl.P, out=seg, workspace=ws, err_flag=err)

        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for k in range(max(Wm, NB)):
                step(k)
        torch.cuda.synchronize()
        graphs = []
        for fn in (step, sgmv, segment):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for k in range(K):
                    fn(k)
            graphs.append(g)
        step_ms = _time_graph_median(graphs[0], side, settle_s=0.2)[0] / K
        sgmv_ms = _time_graph_median(graphs[1], side)[0] / K
        seg_ms = _time_graph_median(graphs[2], side)[0] / K
        assert int(err.item()) == 0, f"{name}: device error flag {int(err.item())}"
        kern_ms = step_ms if one_launch(wl) else sgmv_ms
        kname = dominant_kernel(wl)
        gbs = ab / (kern_ms * 1e-3) / 1e9
        out[name] = {"step_us": round(step_ms * 1e3, 3), "sgmv_us": round(sgmv_ms * 1e3, 3),
                     "segment_us": round(seg_ms * 1e3, 3),
                     "kernel_us": round(kern_ms * 1e3, 3), "kernel": kname,
                     "launches_per_step": launches_per_step(wl), "algorithmic_bytes": int(ab), "flops": int(nf),
                     "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                     "tflops": round(nf / (kern_ms * 1e-3) / 1e12, 3),
                     "distinct_adapters": int(np.unique(ids).size), "input_copies": NB,
                     "traffic": recorded_traffic(kname, name)}
        del graphs, copies, ws
        torch.cuda.empty_cache()
    return out


def backbone_fused(Wm, dev, lsg, bf16_peaks):
    """The Llama2-13B prefill layer (7 projections, 6224 tokens, r=64) with
    synthetic backbone weights W: the backbone projection with its LoRA delta
    as gemm_lora (the expand fused into the GEMM's accumulator, y written
    once; one call per projection), against cuBLAS x @ W per projection
    followed by one sgmv_multi for the layer.  Segmentation given (computed
    once).  TFLOP/s count 2*n*h_in*h_out per projection plus the LoRA flops."""
    import torch
    from workloads import make_backbone_weights

    wl = WORKLOADS["13b_prefill"]
    ids = wl.ids()
    inp = make_inputs(wl, dev)
    Ws = make_backbone_weights(wl, dev)
    seg = lsg.lora_segment(inp.ids, wl.P)
    n = wl.n
    ys = [torch.empty(n, p.h_out, dtype=torch.bfloat16, device=dev) for p in wl.projs]
    ws = torch.empty(lsg.gemm_lora_workspace_bytes(n, wl.r), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    projs = [(inp.x[p.x_key], inp.A[i], inp.B[i], ys[i], wl.scale) for i, p in enumerate(wl.projs)]
    cproj = lsg.make_projs(projs)

    def fused():
        for i, p in enumerate(wl.projs):
            lsg.gemm_lora(inp.x[p.x_key], Ws[i], inp.A[i], inp.B[i], seg, ys[i], wl.scale, workspace=ws,
                          err_flag=err)

    def unfused():
        for i, p in enumerate(wl.projs):
            torch.matmul(inp.x[p.x_key], Ws[i], out=ys[i])
        lsg.sgmv_multi(projs, seg, err_flag=err, c_projs=cproj)

    def gemm_only():
        for i, p in enumerate(wl.projs):
            torch.matmul(inp.x[p.x_key], Ws[i], out=ys[i])

    side = torch.cuda.Stream(dev)
    out = {"workload": wl.description + "; synthetic W ~ N(0, 1/h_in) per projection",
           "how": "CUDA graph of 3 layer passes, median of 5 replays (events on the replay stream)"}
    gemm_flops = sum(2 * n * p.h_in * p.h_out for p in wl.projs)
    lora_flops = flops(wl, ids)
    reps = 3
    for name, fn in (("fused_gemm_lora", fused), ("cublas_gemm_then_sgmv_multi", unfused),
                     ("cublas_gemm_alone", gemm_only)):
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(max(1, Wm // 2)):
                fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for _ in range(reps):
                fn()
        ms = _time_graph_median(g, side, reps=5, settle_s=0.3)[0] / reps
        del g
        f = gemm_flops + (0 if name == "cublas_gemm_alone" else lora_flops)
        tf = f / (ms * 1e-3) / 1e12
        out[name] = {"us": round(ms * 1e3, 1), "tflops": round(tf, 1),
                     "frac_of_bf16_sustained": round(tf / bf16_peaks[0], 4) if bf16_peaks[0] else None,
                     "frac_of_bf16_burst": round(tf / bf16_peaks[1], 4) if bf16_peaks[1] else None}
    assert int(err.item()) == 0, f"device error flag {int(err.item())}"
    out["fused_over_unfused"] = round(out["fused_gemm_lora"]["us"] / out["cublas_gemm_then_sgmv_multi"]["us"], 4)
    del inp, Ws, ys, ws
    torch.cuda.empty_cache()
    return out


def batch_curve(K, Wm, dev, lsg, max_copies):
    """Step latency against batch size, identical vs mixed adapters, for a
    decode projection (Llama2-7B 4096->4096, r=16) and a prefill projection
    (Llama2-13B 5120->5120, r=64): the kernel-level analogue of measuring
    latency against batch size per stage (Punica: Multi-Tenant LoRA Serving,
    "Interesting ideas" I5; "Key points": identical vs mixed adapters)."""
    from workloads import Proj, Workload

    out = {}
    dec_n = [1, 4, 16, 32, 64, 128, 256]
    rows = {"n": dec_n, "identical_us": [], "mixed_us": []}
    for n in dec_n:
        P = max(64, n)
        wl = Workload("curve_dec", (Proj("proj", 4096, 4096, "x"),), 16, P, n, 1.0, lambda: None, "", "curve_dec")
        rng = np.random.default_rng(n)
        rows["identical_us"].append(_time_ids(wl, np.full(n, 3, np.int32), K, Wm, dev, lsg, max_copies))
        rows["mixed_us"].append(_time_ids(wl, rng.choice(P, n, replace=False), K, Wm, dev, lsg, max_copies))
    out["decode_llama2_7b_proj_r16"] = rows
    pre_n = [128, 512, 1024, 2048, 4096]
    rows = {"n": pre_n, "identical_us": [], "mixed_us": [], "mixed_requests": []}
    for n in pre_n:
        P = 32
        wl = Workload("curve_pre", (Proj("proj", 5120, 5120, "x"),), 64, P, n, 1.0, lambda: None, "", "curve_pre")
        nreq = max(1, n // 256)
        mixed = np.repeat(np.arange(nreq, dtype=np.int32), n // nreq)
        mixed = np.concatenate([mixed, np.full(n - mixed.size, nreq - 1, np.int32)])
        rows["identical_us"].append(_time_ids(wl, np.zeros(n, np.int32), max(3, K // 4), Wm, dev, lsg, max_copies))
        rows["mixed_us"].append(_time_ids(wl, mixed, max(3, K // 4), Wm, dev, lsg, max_copies))
        rows["mixed_requests"].append(nreq)
    out["prefill_llama2_13b_proj_r64"] = rows
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--settle", type=float, default=0.5, help="seconds of untimed replays before timing")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--max-copies", type=int, default=256)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-mixed", action="store_true")
    ap.add_argument("--no-slots", action="store_true", help="skip the slot-arena / mixed-rank measurement")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="time cap of the reference arm's timed calls")
    ap.add_argument("--no-batch-curve", action="store_true",
                    help="skip step latency against batch size (decode and prefill, identical vs mixed adapters)")
    ap.add_argument("--backbone-only", action="store_true",
                    help="only the backbone GEMM + LoRA comparison (a diagnostic line, not the benchmark contract)")
    ap.add_argument("--no-backbone", action="store_true",
                    help="skip the backbone GEMM with the fused LoRA expand against cuBLAS + SGMV")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload kernel times of the 7B layer, 13B prefill and 70B decode batches")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.backbone_only:
        import torch

        import adapter_gemm_02_b300 as lsg

        print(json.dumps({"backbone_fused": backbone_fused(args.warmup, torch.device("cuda", 0), lsg, bf16_peaks())}),
              flush=True)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
