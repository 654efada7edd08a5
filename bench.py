#!/usr/bin/env python3
"""Benchmark of the NSA selection-attention forward on GB300.

One step = one forward over the whole workload (every (b, m, g) row): one
launch of the library's kernel. Default workload: B=1, M=N=65536, H=64, G=8,
D=128, block_size=64, T=16 (block 0, the two most recent causal blocks and
13 random earlier ones per row), fp16 inputs, seeded synthetic data.

Prints ONE JSON line (rank 0):
  value         TFLOP/s over the timed steps (4*D FLOPs per query, head and
                visible gathered key), inputs resident in HBM, L2 flushed
                between steps (a 512 MiB write outside the timed events);
  gathered_gbs  gathered K/V bytes per second (whole selected blocks);
  speedup_vs_dense_fa  time of dense causal attention at the same sequence
                length on the same Q/K/V (the library's tcgen05 flash kernel,
                nsa_swa_fwd with window (-1, 0)) over the sparse time;
  speedup_vs_dense_causal  time of the same build with every causal block
                listed (T=1024, same Q/K/V) over the sparse time;
  roofline      gathered bytes per second against the gather ceiling
                measured in the same run (the probe kernel issuing the
                forward's TMA copies from L2-resident K/V and nothing else);
                the fraction of HBM bandwidth is kept under "hbm";
  e2e           the same metric through the C ABI's host-buffer entry point
                (pinned host inputs uploaded and O / LSE downloaded every step,
                chunked so copies overlap the kernels);
  cpu_baseline  the CPU oracle timed on a bounded row sample, host cores;
  clocks        nvidia-smi SM clocks and throttle reasons during the steps.

``--impl reference`` times the CPU oracle instead (the only reference that
exists for this method), on the same workload, metric and unit.

Under torchrun (N > 1) every rank runs its own workload (seed + rank) on its
own GPU -- independent problems, weak scaling, no collective on the data
path; the time is the max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sel-attn fwd TFLOP/s & gathered-KV GB/s (M=64k,T=16,bs=64); x vs dense causal"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="m64k_bs64")
    ap.add_argument("--dense-steps", type=int, default=3)
    ap.add_argument("--skip-dense", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-bwd", action="store_true")
    ap.add_argument("--skip-swa", action="store_true",
                    help="skip timing the sliding-window attention kernel")
    ap.add_argument("--swa-seq", type=int, default=65536)
    ap.add_argument("--skip-topk", action="store_true",
                    help="skip timing the top-k block selection kernel")
    ap.add_argument("--skip-variants", action="store_true",
                    help="skip timing the bf16-input and 16-bit-O forward variants")
    ap.add_argument("--skip-two-pass", action="store_true",
                    help="skip the two-pass forward (nsa_sel_attn_fwd_shared) leg")
    ap.add_argument("--skip-l2-ceiling", action="store_true",
                    help="skip measuring the gather ceiling (the roofline then falls back to "
                         "HBM bandwidth)")
    ap.add_argument("--skip-dense-fa", action="store_true",
                    help="skip timing dense causal attention (nsa_swa_fwd) on the same inputs")
    ap.add_argument("--cpu-rows", type=int, default=393216,
                    help="rows of the CPU-oracle sample (about 10-15 s of work on 16 cores)")
    ap.add_argument("--seed", type=int, default=None)
    ap.add_argument("--chunk-m", type=int, default=0,
                    help="queries per chunk of the host-buffer pipeline (0: default)")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


FWD_KERNEL_SOURCES = ("common.cuh", "ptx.cuh", "sel_attn_fwd.cu", "sel_attn_fwd.cuh", "status.cuh")


def kernel_source_hash():
    """Hash of the files the forward kernel is compiled from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nsa_block_selection_gb300", "csrc")
    for f in FWD_KERNEL_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def profiled(workload):
    """The committed ncu figures of the workload's forward kernel, or {} when
    the kernel sources changed since they were taken."""
    path = os.path.join(ROOT, "profiles", f"{workload}_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return {}
    if d.get("kernel_source_sha") != kernel_source_hash():
        return {}
    return d


def profiled_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, or None."""
    return profiled(workload).get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons (200 ms)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if self.gpu_id is not None:
                cmd += ["-i", str(self.gpu_id)]
            self.proc = subprocess.Popen(cmd, stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [r.split(",") for r in self.tmp.read().strip().splitlines() if r.strip()]
        os.unlink(self.tmp.name)
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                power.append(float(r[3]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "power_w_max": max(power) if power else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def gpu_smi_id(dev):
    import torch

    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[dev.index or 0] if vis else (dev.index or 0)


def reduce_over_ranks(t_ms, flops, nbytes, dist=None):
    """Whole-job figures: the slowest rank's time, the work summed over ranks
    (independent problems per rank; one scalar all-reduce, no data path)."""
    if dist is None:
        return float(t_ms), float(flops), float(nbytes)
    import torch

    tt = torch.tensor([float(t_ms)], dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    tot = torch.tensor([float(flops), float(nbytes)], dtype=torch.float64)
    dist.all_reduce(tot)
    return float(tt.item()), float(tot[0]), float(tot[1])


def time_steps(fn, steps, warmup, flush, barrier):
    """Per-step CUDA-event times (ms) of fn() on the current stream; flush()
    runs before every step outside the events."""
    import torch

    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    barrier()
    st = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    wall0 = time.perf_counter()
    for s, e in evs:
        flush()
        s.record(st)
        fn()
        e.record(st)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier()
    return [s.elapsed_time(e) for s, e in evs], wall


def sample_rows(w, n_rows, seed):
    import numpy as np

    rng = np.random.default_rng(seed)
    b = rng.integers(w.B, size=n_rows)
    m = rng.integers(w.M, size=n_rows)
    g = rng.integers(w.G, size=n_rows)
    return b, m, g


def cpu_oracle_sample(timer, idx, w, n_rows, seed):
    """(TFLOP/s, info) of the oracle on a seeded sample of rows."""
    from nsa_block_selection_gb300.metrics import count_rows

    b, m, g = sample_rows(w, n_rows, seed)
    rows = [(int(x), int(y), int(z)) for x, y, z in zip(b, m, g)]
    flops = count_rows(idx[b, m, g], m, w.N, w.block_size, w.heads_per_group, w.D)
    secs = timer.time_rows(rows)
    tflops = flops / secs / 1e12
    return tflops, {
        "value": tflops, "unit": "TFLOP/s", "cores": timer.workers, "kind": "oracle",
        "sample": f"{n_rows} seeded random (b,m,g) rows of {w.name} "
                  f"({flops / 1e9:.2f} GFLOP), fp64 numpy, {timer.workers} spawn workers x "
                  f"1 BLAS thread, {secs:.2f} s",
        "host_cpu_count": os.cpu_count(),
    }


# --------------------------------------------------------------------------
# arms
# --------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from nsa_block_selection_gb300 import inputs as gen

    w = gen.workload(args.workload)
    seed = args.seed if args.seed is not None else gen.default_seed(w.name)
    q, k, v, idx = gen.make_inputs(w, seed)
    from oracle.cpu_baseline import OracleTimer, host_cores

    rows_per_step = 256 * host_cores()
    vals = []
    info = None
    with OracleTimer(q, k, v, idx, w.block_size, w.scale) as timer:
        for i in range(args.warmup + args.steps):
            tf, info = cpu_oracle_sample(timer, idx, w, rows_per_step, seed + 7 + i)
            if i >= args.warmup:
                vals.append(tf)
    value = statistics.mean(vals)
    info["value"] = value
    rows_total = w.B * w.M * w.G
    from nsa_block_selection_gb300.metrics import count_work
    import torch

    work = count_work(torch.from_numpy(idx), w.N, w.block_size, w.heads_per_group, w.D)
    ms = work["flops"] / (value * 1e12) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "M": w.M, "N": w.N, "H": w.H, "G": w.G,
                   "D": w.D, "block_size": w.block_size, "T": w.T,
                   "rows_per_step": rows_per_step, "rows_total": rows_total,
                   "note": "ms_per_step extrapolates the sample throughput to the whole "
                           "workload"},
        "cpu_baseline": info,
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


class nvtx_range:
    """An NVTX range around a bench leg (visible in a profiler's timeline;
    a no-op without one)."""

    def __init__(self, name):
        self.name = name

    def __enter__(self):
        try:
            import torch

            torch.cuda.nvtx.range_push(self.name)
            self.pushed = True
        except Exception:  # noqa: BLE001 -- no NVTX: nothing to mark
            self.pushed = False
        return self

    def __exit__(self, *exc):
        if self.pushed:
            import torch

            torch.cuda.nvtx.range_pop()
        return False


def run_leg(enabled, fn, *a):
    """fn(*a) when enabled, else None; an exception becomes {"error": repr}
    (also printed to stderr), so one failing auxiliary measurement does not
    take the measured headline with it. Each leg runs in an NVTX range of its
    name."""
    if not enabled:
        return None
    try:
        with nvtx_range(fn.__name__):
            return fn(*a)
    except Exception as e:  # noqa: BLE001 -- reported in the JSON line, not hidden
        print(f"bench: {fn.__name__} failed: {e!r}", file=sys.stderr, flush=True)
        return {"error": repr(e)}


def run_ours(args):
    import numpy as np
    import torch

    from nsa_block_selection_gb300 import _lib, inputs as gen, sel_attn_fwd
    from nsa_block_selection_gb300.metrics import count_work

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")
        barrier = dist.barrier
    else:
        dist = None

        def barrier():
            return None

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _lib.load()
    w = gen.workload(args.workload)
    seed = (args.seed if args.seed is not None else gen.default_seed(w.name)) + rank
    q_np, k_np, v_np, idx_np = gen.make_inputs(w, seed)

    # CPU baseline first (spawned pool, before any timing), rank 0 at N=1 only
    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        from oracle.cpu_baseline import OracleTimer

        with OracleTimer(q_np, k_np, v_np, idx_np, w.block_size, w.scale) as timer:
            _, cpu = cpu_oracle_sample(timer, idx_np, w, args.cpu_rows, seed + 99)

    q = torch.from_numpy(q_np).to(dev)
    k = torch.from_numpy(k_np).to(dev)
    v = torch.from_numpy(v_np).to(dev)
    idx = torch.from_numpy(idx_np).to(dev)
    out = torch.empty((w.B, w.M, w.H, w.D), dtype=torch.float32, device=dev)
    lse = torch.empty((w.B, w.H, w.M), dtype=torch.float32, device=dev)
    work = count_work(idx, w.N, w.block_size, w.heads_per_group, w.D)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.fill_(1.0)

    def step():
        sel_attn_fwd(q, k, v, idx, w.block_size, w.scale, out=out, lse=lse)

    clocks = ClockSampler(gpu_smi_id(dev))
    clocks.start()
    with nvtx_range("headline forward"):
        times, wall = time_steps(step, args.steps, args.warmup, flush, barrier)
    clk = clocks.stop()
    t_ms, flops_all, bytes_all = reduce_over_ranks(statistics.mean(times), work["flops"],
                                                   work["gathered_bytes"], dist)
    tflops = flops_all / (t_ms * 1e-3) / 1e12
    gbs = bytes_all / (t_ms * 1e-3) / 1e9

    # e2e: host buffers through the C ABI each step
    e2e = None
    if not args.skip_e2e:
        with nvtx_range("e2e host buffers"):
            e2e = run_e2e(w, q_np, k_np, v_np, idx_np, work, args, barrier, dev, dist)

    # The legs below run on rank 0 of a 1-GPU run only. A leg that raises is
    # reported in its own key ({"error": ...}) so the measured headline above
    # is still printed.
    solo = rank == 0 and world == 1

    def leg(skip, fn, *a):
        return run_leg(solo and not skip, fn, *a)

    # backward (dQ, dK, dV) on the same inputs, after the timed forward
    backward = leg(args.skip_bwd, run_backward, w, q, k, v, idx, out, lse, work, flush, args)
    # top-k block selection producing an index tensor of this workload's shape
    topk = leg(args.skip_topk, run_topk, w, flush, args, dev)
    # GQA sliding-window attention (the pages' second kernel), tcgen05
    swa = leg(args.skip_swa, run_swa, flush, args, dev)
    # the same forward in two passes (blocks common to a 16-query tile once)
    two_pass = leg(args.skip_two_pass, run_two_pass, w, q, k, v, idx, work, flush, args, t_ms)
    # element-type variants of the forward on the same workload
    variants = leg(args.skip_variants, run_variants, w, q, k, v, idx, work, flush, args)
    # dense-causal-equivalent run: same Q/K/V, every causal block listed
    dense = leg(args.skip_dense, run_dense, w, q, k, v, out, lse, flush, args, t_ms)
    # dense causal attention (tcgen05 flash kernel) on the same Q/K/V
    dense_fa = leg(args.skip_dense_fa, run_dense_fa, w, q, k, v, work, flush, args, t_ms)

    # the gather ceiling: the forward's own TMA copies from the L2-resident
    # K/V of one group, nothing else (measured on this GPU, in this run)
    ceiling = run_leg(not args.skip_l2_ceiling, run_l2_ceiling, w, k, v, idx, work, flush, dev)
    peaks = load_peaks()
    roofline = make_roofline(w, work, statistics.mean(times), peaks, ceiling)
    if dense_fa and "ms_per_step" in dense_fa and ceiling and "peak_gbs" in ceiling:
        t_floor = work["gathered_bytes"] / (ceiling["peak_gbs"] * 1e9) * 1e3
        dense_fa["gather_floor_ms"] = t_floor
        dense_fa["speedup_bound_at_floor"] = dense_fa["ms_per_step"] / t_floor
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "M": w.M, "N": w.N, "H": w.H, "G": w.G,
                   "D": w.D, "block_size": w.block_size, "T": w.T, "seed": seed,
                   "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write, "
                         "outside the timed events)",
                   "parallelism": f"independent replicas x{world}" if world > 1 else "1 GPU",
                   "accumulate": "fp32"},
        "gathered_gbs": gbs,
        "flops_per_step": work["flops"], "gathered_bytes_per_step": work["gathered_bytes"],
        "speedup_vs_dense_fa": dense_fa.get("speedup") if dense_fa else None,
        "dense_fa": dense_fa,
        "speedup_vs_dense_causal": dense.get("speedup") if dense else None,
        "dense_causal": dense,
        "l2_ceiling": ceiling,
        "backward": backward,
        "variants": variants,
        "two_pass": two_pass,
        "topk": topk,
        "swa": swa,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clk,
        "gpu_launches": args.steps,
        "wall_s_timed": wall,
        "kernel_source_sha": kernel_source_hash(),
        "device": torch.cuda.get_device_name(dev),
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def make_roofline(w, work, t_kernel_ms, peaks, ceiling):
    """Roofline of the headline kernel. Its K/V blocks are served from L2
    (one group's K/V stays resident while its queries run), so the bound is
    the gather ceiling measured by the probe in this run; the ratio to HBM
    bandwidth is kept beside it."""
    achieved = work["gathered_bytes"] / (t_kernel_ms * 1e-3) / 1e9
    t_roof_hbm = max(work["flops"] / (peaks["bf16_tflops"] * 1e12),
                     work["gathered_bytes"] / (peaks["hbm_gbs"] * 1e9))
    hbm = {"achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
           "frac": achieved / peaks["hbm_gbs"], "t_roofline_ms": t_roof_hbm * 1e3,
           "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, burst copy)"}
    common = {
        "traffic": profiled_traffic(w.name),
        "traffic_note": "ncu DRAM bytes per launch (read + write); gathered bytes come from L2",
        "flop_frac_of_tensor_peak": (work["flops"] / (t_kernel_ms * 1e-3))
                                     / (peaks["bf16_tflops"] * 1e12),
        "units_per_launch": work["gathered_bytes"],
        "unit_note": "achieved = gathered K/V bytes (whole selected blocks, exact from the "
                     "index tensor) / mean CUDA-event time of the launch",
    }
    if ceiling and "peak_gbs" in ceiling:
        peak = ceiling["peak_gbs"]
        return dict({"bound": "l2", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "peak_source": "measured in this run: the best of the gather probes "
                                    "(the forward's TMA copies alone on every SM, random "
                                    "blocks and the workload's own rows; l2_ceiling key), "
                                    f"from {ceiling['peak_from']}",
                     "t_floor_ms": work["gathered_bytes"] / (peak * 1e9) * 1e3,
                     "hbm": hbm}, **common)
    return dict({"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                 "unit": "GB/s", "frac": hbm["frac"], "peak_source": hbm["peak_source"],
                 "t_roofline_ms": hbm["t_roofline_ms"],
                 "note": "gather ceiling not measured; blocks are re-read from L2, so the "
                         "fraction of HBM bandwidth can exceed 1"}, **common)


def run_l2_ceiling(w, k, v, idx, work, flush, dev):
    """The gather ceiling for this workload: random blocks of its K/V (group
    0), and its own index rows' copies alone (no computation)."""
    from nsa_block_selection_gb300 import l2_ceiling

    return l2_ceiling.measure(k, v, w.block_size, g=0, idx=idx,
                              gathered_bytes=work["gathered_bytes"], flush=flush,
                              clocks=ClockSampler(gpu_smi_id(dev)))


def run_dense_fa(w, q, k, v, work, flush, args, t_sparse_ms):
    """Dense causal attention at the same sequence length on the same Q/K/V:
    nsa_swa_fwd with window (-1, 0) (tcgen05 flash kernel, every key <= the
    query), the "dense FA at same seqlen" of the page's performance target.
    FLOPs: 4*D per (query, head, key <= query)."""
    import torch

    from nsa_block_selection_gb300 import swa_fwd

    if w.M != w.N:
        return {"error": "dense causal attention is timed for M == N only"}
    o16 = torch.empty((w.B, w.M, w.H, w.D), dtype=q.dtype, device=q.device)
    lse = torch.empty((w.B, w.H, w.M), dtype=torch.float32, device=q.device)

    def step():
        swa_fwd(q, k, v, window=(-1, 0), scale=w.scale, out=o16, lse=lse)

    steps = max(3, args.steps // 6)
    times, _ = time_steps(step, steps, 3, flush, lambda: None)
    t = statistics.mean(times)
    flops = 4 * w.D * w.H * w.B * swa_pairs(w.M, w.N, -1, 0)
    del o16, lse
    torch.cuda.empty_cache()
    return {"kernel": "nsa_swa_fwd, window (-1, 0), fp16 in / fp16 O, same Q/K/V",
            "ms_per_step": t, "tflops": flops / (t * 1e-3) / 1e12, "flops": flops,
            "speedup": t / t_sparse_ms, "steps": steps,
            "work_ratio": flops / work["flops"]}


def swa_pairs(M, N, left, right):
    """(query, key) pairs inside the windows: sum over i of |[i-left, i+right] & [0, N)|."""
    import numpy as np

    i = np.arange(M, dtype=np.int64)
    lo = np.zeros(M, np.int64) if left < 0 else np.maximum(0, i - left)
    hi = np.full(M, N - 1, np.int64) if right < 0 else np.minimum(N - 1, i + right)
    return int(np.maximum(hi - lo + 1, 0).sum())


def run_swa(flush, args, dev):
    """nsa_swa_fwd, bf16, B=1, H=64, H_kv=8, D=128 (the page's API example
    shape) at seq = --swa-seq for the page's windows. FLOPs: 4*D per (query,
    head, key in the window). Inputs drawn on the device; L2 flushed."""
    import torch

    from nsa_block_selection_gb300 import swa_fwd

    B, S, H, Hkv, D = 1, args.swa_seq, 64, 8, 128
    g = torch.Generator(device=dev).manual_seed(5)
    q = torch.randn((B, S, H, D), generator=g, device=dev).bfloat16()
    k = torch.randn((B, S, Hkv, D), generator=g, device=dev).bfloat16()
    v = torch.randn((B, S, Hkv, D), generator=g, device=dev).bfloat16()
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    peaks = load_peaks()
    res = {"shape": {"B": B, "seq": S, "H": H, "H_kv": Hkv, "D": D, "dtype": "bf16"},
           "windows": []}
    for left, right in ((512, 0), (1024, 0), (4096, 0), (8192, 0), (-1, 0)):
        def step():
            swa_fwd(q, k, v, window=(left, right), out=out, lse=lse)

        steps = max(3, args.steps // 6)
        times, _ = time_steps(step, steps, 3, flush, lambda: None)
        t = statistics.mean(times)
        flops = 4 * D * H * B * swa_pairs(S, S, left, right)
        tf = flops / (t * 1e-3) / 1e12
        res["windows"].append({"window": [left, right], "ms_per_step": t, "tflops": tf,
                               "tensor_frac": tf / peaks["bf16_tflops"], "flops": flops,
                               "steps": steps})
    if not args.skip_cpu:
        res["cpu_oracle"] = swa_cpu_oracle(q, k, v, (4096, 0))
    del q, k, v, out, lse
    torch.cuda.empty_cache()
    return res


def swa_cpu_oracle(q, k, v, window, n_rows=96, seed=4):
    """oracle/swa.py on a seeded sample of (i, KV head) rows of the same
    inputs, one process; TFLOP/s counted like the kernel's (4*D per query,
    head and key in the window)."""
    import numpy as np

    import oracle.swa as W

    B, S, H, D = q.shape
    Hkv = k.shape[2]
    hpg = H // Hkv
    rng = np.random.default_rng(seed)
    ms = rng.integers(0, S, n_rows)
    gs = rng.integers(0, Hkv, n_rows)
    kh = k.float().cpu().numpy()
    vh = v.float().cpu().numpy()
    qrows = {int(m): q[0, int(m)].float().cpu().numpy() for m in ms}

    class _Q:  # the sampled query rows, indexed like Q [B, S, H, D]
        shape = (B, S, H, D)

        def __getitem__(self, key):
            b, i, hs = key
            return qrows[int(i)][hs]

    flops = 0
    t0 = time.perf_counter()
    for m, g in zip(ms, gs):
        W.swa_row(_Q(), kh, vh, 0, int(m), int(g), window[0], window[1])
        flops += 4 * D * hpg * len(W.window_keys(int(m), S, window[0], window[1]))
    secs = time.perf_counter() - t0
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "window": list(window),
            "sample": f"{n_rows} seeded random (query, KV head) rows, fp64 numpy, one process, "
                      f"{secs:.2f} s"}


def topk_bytes(B, M, N, G, T, bs, n_init, n_local):
    """Algorithmic bytes of nsa_topk_blocks: the scores of the free
    candidates of rows with more than T candidates (read once) and the
    index rows (written)."""
    import numpy as np

    m = np.arange(M, dtype=np.int64)
    c = np.minimum(m, N - 1) // bs if N > 0 else np.full(M, -1)
    free = np.where(c + 1 > T, c + 1 - n_init - n_local, 0)
    return int(B * G * (4 * free.sum() + 4 * T * M))


def topk_cpu_oracle(sc, w, nblk, n_rows=2048, seed=3):
    """oracle/topk.py on a seeded sample of rows of the same score tensor, one
    process; GB/s counted like the kernel's algorithmic bytes."""
    import numpy as np

    import oracle.topk as K

    rng = np.random.default_rng(seed)
    ms = rng.integers(0, w.M, n_rows)
    gs = rng.integers(0, w.G, n_rows)
    rows = sc[0, ms, gs].cpu().numpy()
    t0 = time.perf_counter()
    for r in range(n_rows):
        K.topk_row(rows[r], int(ms[r]), w.N, w.block_size, w.T, 1, 2)
    secs = time.perf_counter() - t0
    c = np.minimum(ms, w.N - 1) // w.block_size
    nbytes = int((4 * np.where(c + 1 > w.T, c + 1 - 3, 0) + 4 * w.T).sum())
    return {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n_rows} seeded random (m, g) rows, one process, {secs:.2f} s"}


def run_topk(w, flush, args, dev):
    """nsa_topk_blocks on i.i.d. scores [B, M, G, ceil(N/bs)] (drawn on the
    device), T, block 0 and the two most recent blocks forced: the index
    rule of the workload as a top-k."""
    import torch

    from nsa_block_selection_gb300 import inputs as gen
    from nsa_block_selection_gb300 import topk_blocks

    nblk = -(-w.N // w.block_size)
    sc = gen.make_block_scores_torch(w.B, w.M, w.G, nblk, 99, dev)
    out = torch.empty((w.B, w.M, w.G, w.T), dtype=torch.int32, device=dev)

    def step():
        topk_blocks(sc, w.N, w.block_size, w.T, 1, 2, out=out)

    steps = max(5, args.steps // 4)
    times, _ = time_steps(step, steps, 3, flush, lambda: None)
    t = statistics.mean(times)
    nbytes = topk_bytes(w.B, w.M, w.N, w.G, w.T, w.block_size, 1, 2)
    peaks = load_peaks()
    gbs = nbytes / (t * 1e-3) / 1e9
    res = {"ms_per_step": t, "gbs": gbs, "bytes_per_step": nbytes,
           "hbm_frac": gbs / peaks["hbm_gbs"], "rows": w.B * w.M * w.G, "steps": steps,
           "scores_bytes": sc.numel() * 4, "n_init": 1, "n_local": 2,
           "note": "bytes = scores of the free candidates of rows with more than T "
                   "candidates + the index rows written; L2 flushed between steps"}
    if not args.skip_cpu:
        res["cpu_oracle"] = topk_cpu_oracle(sc, w, nblk)
    del sc, out
    torch.cuda.empty_cache()
    return res


def run_variants(w, q, k, v, idx, work, flush, args):
    """The forward with bf16 Q/K/V and/or a 16-bit O (nsa_sel_attn_fwd_ex),
    timed like the headline run on the same index tensor (Q/K/V converted on
    the device; the timing does not depend on the values)."""
    import torch

    from nsa_block_selection_gb300 import sel_attn_fwd

    res = {}
    steps = max(3, args.steps // 6)
    lse = torch.empty((w.B, w.H, w.M), dtype=torch.float32, device=q.device)
    for qkv, odt in (("bf16", "f32"), ("f16", "f16"), ("bf16", "bf16")):
        dt = torch.bfloat16 if qkv == "bf16" else torch.float16
        ot = torch.float32 if odt == "f32" else dt
        tq, tk, tv = (x.to(dt) for x in (q, k, v))
        out = torch.empty((w.B, w.M, w.H, w.D), dtype=ot, device=q.device)

        def step():
            sel_attn_fwd(tq, tk, tv, idx, w.block_size, w.scale, out=out, lse=lse)

        times, _ = time_steps(step, steps, 3, flush, lambda: None)
        t = statistics.mean(times)
        res[f"{qkv}_in_{odt}_out"] = {"ms_per_step": t,
                                      "tflops": work["flops"] / (t * 1e-3) / 1e12,
                                      "steps": steps}
        del tq, tk, tv, out
    torch.cuda.empty_cache()
    return res


def run_two_pass(w, q, k, v, idx, work, flush, args, t_one_ms):
    """nsa_sel_attn_fwd_shared on the headline inputs, timed like the headline
    run (three kernels per step: per-tile lists of the blocks every query of
    a 16-query tile lists, the tile's own block included; their softmax on
    tcgen05, masked per row; the gather
    kernel over the remaining blocks). FLOPs and gathered bytes are those of
    the operation, as for the headline, so the numbers compare directly."""
    import torch

    from nsa_block_selection_gb300 import _lib

    ws = torch.empty(max(_lib.shared_workspace_bytes(w.B, w.M, w.G), 256), dtype=torch.uint8,
                     device=q.device)
    out = torch.empty((w.B, w.M, w.H, w.D), dtype=torch.float32, device=q.device)
    lse = torch.empty((w.B, w.H, w.M), dtype=torch.float32, device=q.device)

    def step():
        _lib.sel_attn_fwd_shared(q, k, v, idx, w.block_size, w.scale, out=out, lse=lse,
                                 workspace=ws)

    steps = max(5, args.steps // 4)
    times, _ = time_steps(step, steps, 3, flush, lambda: None)
    t = statistics.mean(times)
    ntiles = -(-w.M // 16)
    rec = ws[:w.B * w.G * ntiles * 32].view(torch.int32).reshape(-1, 8)
    cnt = rec[:, 0].float()
    res = {"ms_per_step": t, "tflops": work["flops"] / (t * 1e-3) / 1e12,
           "gathered_gbs": work["gathered_bytes"] / (t * 1e-3) / 1e9,
           "speedup_vs_one_pass": t_one_ms / t, "steps": steps,
           "kernels_per_step": 3,
           "shared_blocks_per_tile_mean": float(cnt.mean()),
           "tiles_with_shared_blocks": float((cnt > 0).float().mean())}
    del ws, out, lse
    torch.cuda.empty_cache()
    return res


def local_entries(idx, w):
    """(visible entries, entries of the query's own block c or of block
    c - 1) of the index tensor [B, M, G, T]: the backward's dQ reductions
    are the visible entries minus the local ones (rows list a block once)."""
    import torch

    m = torch.arange(w.M, device=idx.device).view(1, w.M, 1, 1)
    c = m // w.block_size
    nblk = (w.N + w.block_size - 1) // w.block_size
    last = torch.clamp(m, max=w.N - 1)
    t = idx.long()
    vis = (t >= 0) & (t < nblk) & (t * w.block_size <= last)
    loc = vis & ((t == c) | (t == c - 1))
    return int(vis.sum()), int(loc.sum())


def run_backward(w, q, k, v, idx, out, lse, work, flush, args):
    """nsa_sel_attn_bwd on the forward's outputs and a seeded fp32 dO.
    FLOPs: 10*D per (query, head, visible key) -- QK^T, dP, dQ, dK, dV."""
    import torch

    from nsa_block_selection_gb300 import _lib

    gen = torch.Generator(device=q.device).manual_seed(1234)
    do = torch.randn(out.shape, generator=gen, device=q.device, dtype=torch.float32)
    need = _lib.bwd_workspace_bytes(w.B, w.M, w.N, w.H, w.G, w.D, w.T, w.block_size)
    ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(out)
    dk = torch.empty((w.B, w.N, w.G, w.D), dtype=torch.float32, device=q.device)
    dv = torch.empty_like(dk)

    def step():
        _lib.sel_attn_bwd(q, k, v, idx, out, lse, do, w.block_size, w.scale, dq=dq, dk=dk,
                          dv=dv, workspace=ws)

    steps = max(3, args.steps // 6)
    times, _ = time_steps(step, steps, 3, flush, lambda: None)
    t = statistics.mean(times)
    flops = work["flops"] // 4 * 10
    res = {"ms_per_step": t, "tflops": flops / (t * 1e-3) / 1e12, "flops_per_step": flops,
           "workspace_bytes": need, "steps": steps}
    res["bf16"] = run_leg(True, backward_bf16, w, q, k, v, idx, out, lse, do, dq, dk, dv, ws,
                          flush, steps, flops)
    if w.D == 128:
        # dQ = dS K per (query, selected block): every head of the group,
        # D fp32 values each. The entries of a query's own block c and of
        # block c - 1 are summed inside the local-block kernel and stored
        # once per row; the others are added with reductions.
        per_entry = (w.H // w.G) * w.D * 4
        n_entries, n_local = local_entries(idx, w)
        red = (n_entries - n_local) * per_entry
        ceiling = run_leg(True, reduction_ceiling, dq, w)
        res.update({"dq_reduction_bytes": red, "dq_reduction_gbs": red / (t * 1e-3) / 1e9,
                    "dq_local_entries": n_local, "dq_entries": n_entries,
                    "dq_reduction_ceiling": ceiling,
                    "dq_reduction_frac": (red / (t * 1e-3) / 1e9 / ceiling["gbs"]
                                          if ceiling and "gbs" in ceiling else None),
                    "kernels": "prep (fp16 dO, LSE, delta), index transpose (count, scan, "
                               "fill, chunk order; second stream), local-block tcgen05 kernel "
                               "(blocks c and c - 1 of every block row: dQ stored once, dK / dV "
                               "per block row), key-major tcgen05 kernel for the other entries: "
                               "dK, dV (bulk fp32 reductions per chunk) and dQ = dS K (fp32 "
                               "reductions per batch)"})
    else:
        res["kernels"] = ("dQ (query-major, mma.sync), index transpose (count, scan, fill), "
                          "dK/dV (key-major, mma.sync, fp32 atomics)")
    del ws, do, dq, dk, dv
    torch.cuda.empty_cache()
    return res


def backward_bf16(w, q, k, v, idx, out, lse, do, dq, dk, dv, ws, flush, steps, flops):
    """The same backward with bf16 Q/K/V (nsa_sel_attn_bwd_ex): the inputs
    converted once, O and LSE from the bf16 forward (untimed)."""
    import torch

    from nsa_block_selection_gb300 import _lib, sel_attn_fwd

    qb, kb, vb = (x.to(torch.bfloat16) for x in (q, k, v))
    ob, lb = torch.empty_like(out), torch.empty_like(lse)
    sel_attn_fwd(qb, kb, vb, idx, w.block_size, w.scale, out=ob, lse=lb)

    def step():
        _lib.sel_attn_bwd(qb, kb, vb, idx, ob, lb, do, w.block_size, w.scale, dq=dq, dk=dk,
                          dv=dv, workspace=ws)

    times, _ = time_steps(step, steps, 3, flush, lambda: None)
    t = statistics.mean(times)
    del qb, kb, vb, ob, lb
    torch.cuda.empty_cache()
    return {"ms_per_step": t, "tflops": flops / (t * 1e-3) / 1e12, "steps": steps,
            "inputs": "Q, K, V bf16; O, LSE, dO and the gradients fp32"}


def reduction_ceiling(dq, w, seconds=0.3):
    """The rate of the backward's dQ reductions alone on this GPU: 4 KB rows
    (one query's 8 heads of one KV group) added with 16-byte fp32 reductions
    into random rows of the dQ tensor's first group (nsa_probe_reduce_rows;
    adds zeros). Timed with CUDA events on the current stream."""
    import torch

    from nsa_block_selection_gb300 import _lib

    sms = torch.cuda.get_device_properties(dq.device).multi_processor_count
    rows, stride = w.B * w.M, w.H * w.D
    flat = dq.view(-1)
    st = torch.cuda.current_stream(dq.device)
    ctas, warps = sms * 4, 8

    def once(iters):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        n = _lib.probe_reduce_rows(flat, rows, stride, ctas, warps, iters, stream=st)
        e1.record(st)
        e1.synchronize()
        return n, e0.elapsed_time(e1)

    n, ms = once(64)
    iters = max(64, int(n / (ms * 1e-3) * seconds / (ctas * warps * 4096)))
    n, ms = once(iters)
    return {"gbs": n / (ms * 1e-3) / 1e9, "ms": ms, "bytes": n,
            "pattern": f"4 KB fp32 rows (red.global.add.v4.f32, 16 B per lane) into random rows "
                       f"of group 0 of dQ [{w.B}, {w.M}, {w.H}, {w.D}] ({rows} rows, "
                       f"{rows * 4096 / 1e6:.0f} MB spread over {dq.numel() * 4 / 1e9:.2f} GB)"}


def run_dense(w, q, k, v, out, lse, flush, args, t_sparse_ms):
    import torch

    from nsa_block_selection_gb300 import inputs as gen, sel_attn_fwd
    from nsa_block_selection_gb300.metrics import count_work

    T = -(-w.M // w.block_size)
    idx_d = gen.dense_causal_indices_torch(w.B, w.M, w.G, T, w.block_size, q.device)
    work = count_work(idx_d, w.N, w.block_size, w.heads_per_group, w.D)

    def step():
        sel_attn_fwd(q, k, v, idx_d, w.block_size, w.scale, out=out, lse=lse)

    times, _ = time_steps(step, max(1, args.dense_steps), 1, flush, lambda: None)
    t = statistics.mean(times)
    del idx_d
    torch.cuda.empty_cache()
    return {"workload": f"{w.name} with T={T}: every causal block listed",
            "ms_per_step": t, "tflops": work["flops"] / (t * 1e-3) / 1e12,
            "gathered_gbs": work["gathered_bytes"] / (t * 1e-3) / 1e9,
            "speedup": t / t_sparse_ms, "work_ratio": None, "steps": max(1, args.dense_steps)}


def run_e2e(w, q_np, k_np, v_np, idx_np, work, args, barrier, dev, dist):
    """Host (pinned) buffers in and out every step through the C ABI's host
    entry point: chunked uploads of Q / indices / visible K-V rows, the
    forward, downloads of O and LSE, overlapped on three streams, all inside
    the timed events."""
    import torch

    from nsa_block_selection_gb300 import _lib

    hq = torch.from_numpy(q_np).pin_memory()
    hk = torch.from_numpy(k_np).pin_memory()
    hv = torch.from_numpy(v_np).pin_memory()
    hi = torch.from_numpy(idx_np).pin_memory()
    ho = torch.empty((w.B, w.M, w.H, w.D), dtype=torch.float32).pin_memory()
    hl = torch.empty((w.B, w.H, w.M), dtype=torch.float32).pin_memory()
    need = _lib.host_workspace_bytes(w.B, w.M, w.N, w.H, w.G, w.D, w.T, w.block_size,
                                     args.chunk_m)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)

    def step():
        _lib.sel_attn_fwd_host(hq, hk, hv, hi, w.block_size, w.scale, out=ho, lse=hl,
                               chunk_m=args.chunk_m, workspace=ws, device=dev, sync=False)

    steps = max(5, args.steps // 4)
    times, _ = time_steps(step, steps, 2, lambda: None, barrier)
    # host-memory bandwidth is shared with other tenants of the machine: the
    # median step is the figure, the mean is reported beside it
    t, flops, _ = reduce_over_ranks(statistics.median(times), work["flops"], 0, dist)
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hi))
    d2h = sum(x.numel() * x.element_size() for x in (ho, hl))
    return {"value": flops / (t * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": t,
            "ms_per_step_mean": statistics.mean(times), "ms_min": min(times),
            "statistic": "median over steps",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "workspace_bytes": need,
            "path": "pinned host -> nsa_sel_attn_fwd_host (chunked H2D / forward / D2H "
                    "pipeline) -> pinned host"}


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
