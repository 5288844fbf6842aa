#!/usr/bin/env python3
"""Benchmark of hc_mix_fused (hyper-connection mix statistics + Sinkhorn) at M=4096.

One step = one hc_mix_fused call over one batch: x[4096, 20480] bf16 (168 MB,
larger than the 129 MB L2, so no flush is needed between steps), W[24, 20480]
fp32, hc_scale[3], hc_base[24], sinkhorn_iters 20 -> pre, post, comb.  Inputs
are the seeded synthetic tensors of hcmix_inputs.

Our arm prints one JSON line with:
  value      device-timed us per call (CUDA events around exactly K calls,
             replayed from CUDA graphs of 10 calls and one remainder graph;
             with N ranks, max elapsed / (K * N));
  roofline   the dominant kernel with CUDA events on its stream: on the
             tensor-core path the whole call is one launch of hcmix_tc_kernel
             (contraction, in-kernel W conversion, grid barrier, slice-ordered
             reduce and epilogue), so its duration is the call's; on the
             two-launch paths the contraction kernel is timed alone.
             Algorithmic bytes (x once + W once) / average duration, against
             the measured HBM copy bandwidth; the contraction phase alone is
             reported beside it;
  e2e        the same metric through the C ABI with host buffers: every step
             copies x, W, hc_scale, hc_base from pinned host memory and reads
             pre, post, comb back; x goes in four row blocks, each block's call
             starting once its rows have landed;
  cpu_baseline  the CPU oracle on the same workload (rank 0, N = 1 only);
  clocks     nvidia-smi samples taken during the timed region.
`--impl reference` times the CPU oracle instead (bounded row samples per step).
`--sweep` times the other workloads instead, one JSON line each: the decode
sweep M in {1, 4, 16, 64, 128, 256} on both paths, M = 512 with outlier
channels, the stock split-K / fused full-K A/B at M in {512, 1024, 2048, 4096},
the 4096-row call on a W packed once, and one 86-call forward (M = 16384, distinct W / scale / base per
call) replayed from a single CUDA graph.
`--protocols` times the 4096-row call with four x buffers in rotation and with
a 512 MB L2 scrub before each call, and the oracle on one thread and on every
host core for the 16-, 512-, 4096-row, decode and 86-call configurations.
Multi-GPU (torchrun): each rank runs its own 4096 rows (weak scaling, rows are
independent, no collective on the data path).
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

M_ROWS = 4096
K_COLS = 20480
ITERS = 20
RMS_EPS = 1e-6
HC_EPS = 0.0
METRIC = "µs/call and HBM GB/s (% of 8 TB/s roofline) for hc_mix_fused at M=4096"
UNIT = "µs/call"
WORKLOAD = f"hc_mix_fused M={M_ROWS} K={K_COLS} mix=24 hc=4 sinkhorn_iters={ITERS}"
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--path", choices=("auto", "simt", "tc"), default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="time the other workloads (one JSON line each) instead of the headline")
    ap.add_argument("--profile-rows", type=int, default=0,
                    help="no timing: four hc_mix_fused calls of this many rows (the command the "
                         "committed ncu summaries capture)")
    ap.add_argument("--protocols", action="store_true",
                    help="the 4096-row call with rotated x buffers and with a scrubbed L2, and "
                         "the oracle on one thread and on every host core (one JSON line each)")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def rank_rows(rank: int, rows_per_rank: int = M_ROWS) -> int:
    """First row of rank `rank`'s batch in the seed-0 activation stream."""
    return rank * rows_per_rank


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "hyper_connection_mix_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def profiled_traffic(kernel: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    from the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_sha") != source_sha():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    def __init__(self, gpu_index: int, interval_ms: int = 100):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", str(self.interval)],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) != 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]),
                                 [p == "Active" for p in parts[5:9]]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [r for r in rows if r[2] > 200.0] or rows
        reasons = sorted({REASONS[i] for r in loaded for i, a in enumerate(r[3]) if a})
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r[2] for r in rows)}


def reduce_max(value: float, world: int, device) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_oracle_time(x, W, sc, bs, rows: int, threads: int):
    """Seconds for one oracle call on the first `rows` rows (all host threads)."""
    import numpy as np
    import oracle
    xs = np.ascontiguousarray(x[:rows])
    t0 = time.perf_counter()
    oracle.fused(xs, W, sc, bs, ITERS, RMS_EPS, HC_EPS, threads=threads)
    return time.perf_counter() - t0


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step one oracle call on a bounded
    row sample, scaled to the 4096-row call; rank 0 only."""
    if rank != 0:
        return
    import hcmix_inputs as hi
    import oracle
    oracle.build()
    cores = host_cores()
    x = hi.make_x(M_ROWS)
    W, sc, bs = hi.make_w(), hi.make_scale(), hi.make_base()
    cal = max(cores, 64)
    t_cal = cpu_oracle_time(x, W, sc, bs, cal, cores)
    per_row = t_cal / cal
    budget_s = 150.0
    rows = int(max(1, min(M_ROWS, budget_s / max(1, args.steps + args.warmup) / per_row)))
    for _ in range(args.warmup):
        cpu_oracle_time(x, W, sc, bs, rows, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_oracle_time(x, W, sc, bs, rows, cores)
    el = time.perf_counter() - t0
    us_call = el / args.steps * (M_ROWS / rows) * 1e6
    from hyper_connection_mix_gb300 import traffic
    line = {
        "impl": "reference", "metric": METRIC, "value": us_call, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M_ROWS, "K": K_COLS,
                   "sample_rows_per_step": rows},
        "hbm_gbs": traffic.algorithmic_bytes(M_ROWS, K_COLS) / (us_call * 1e-6) / 1e9,
        "cpu_baseline": {"value": us_call, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{rows} of {M_ROWS} rows per step, scaled to {M_ROWS}"},
        "e2e": {"value": us_call, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import hcmix_inputs as hi
    from hyper_connection_mix_gb300 import binding, traffic

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    M, K = M_ROWS, K_COLS
    x_h = hi.make_x(M, row0=rank_rows(rank))
    W_h, sc_h, bs_h = hi.make_w(), hi.make_scale(), hi.make_base()
    x = torch.from_numpy(x_h.view(np.int16)).view(torch.bfloat16).to(device)
    W, sc, bs = (torch.from_numpy(a).to(device) for a in (W_h, sc_h, bs_h))
    ws = binding.alloc_workspace(M, K, device)
    out = (torch.empty(M, 4, device=device), torch.empty(M, 4, device=device),
           torch.empty(M, 4, 4, device=device))
    path = args.path if args.path != "auto" else binding.hc_mix_auto_path(M)
    stream = torch.cuda.Stream(device)

    def call(s=stream, xx=x, WW=W, ss=sc, bb=bs, oo=out):
        binding.hc_mix_fused(xx, WW, ss, bb, ITERS, RMS_EPS, HC_EPS, out=oo, workspace=ws,
                             stream=s, path=path)

    with torch.cuda.stream(stream):
        call()
        torch.cuda.synchronize()
        graphs = calls_graphs(call, stream)
    # tc / tc_tf32x3: one cooperative launch per call; simt / tc_staged: the
    # contraction, then the reduce + epilogue kernel
    single_launch = path in ("tc", "tc_tf32x3")
    launches_per_call = 1 if single_launch else 2

    # ---- device-timed value: exactly K calls, as CUDA-graph replays of
    # GRAPH_CALLS calls each (and one remainder graph)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            replay_calls(graphs, args.warmup)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            replay_calls(graphs, args.steps)
        e1.record(stream)
        e1.synchronize()
        barrier(world)
        torch.cuda.synchronize()
    ms = reduce_max(e0.elapsed_time(e1), world, device)
    ms_per_step = ms / args.steps
    us_call = ms * 1e3 / (args.steps * world)
    alg_bytes = traffic.algorithmic_bytes(M, K)

    # ---- the contraction phase alone (tail = 0: no grid barrier, reduce or
    # epilogue), replayed from CUDA graphs so that host launch cost is not timed
    n_k = max(3, min(args.steps, 2000))
    with torch.cuda.stream(stream):
        contract = lambda: binding.hc_mix_contract(x, W, ws, stream=stream, path=path)
        contract()
        torch.cuda.synchronize()
        kgraphs = calls_graphs(contract, stream)
        replay_calls(kgraphs, 3 * GRAPH_CALLS)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        replay_calls(kgraphs, n_k)
        c1.record(stream)
        c1.synchronize()
    contract_us = c0.elapsed_time(c1) * 1e3 / n_k
    peak, peak_kind = measured_peaks()
    if single_launch:  # the call is one launch of the kernel: its duration is the call's
        k_us = us_call * world
        kernel_name = "hcmix_tc_kernel"
    else:
        k_us = contract_us
        kernel_name = "hcmix_simt_slice_kernel" if path == "simt" else "hcmix_tc_kernel"
    achieved = alg_bytes / (k_us * 1e-6) / 1e9

    # ---- end to end through the C ABI with host buffers
    x_pin = torch.from_numpy(x_h.view(np.int16)).view(torch.bfloat16).pin_memory()
    W_pin, sc_pin, bs_pin = (torch.from_numpy(a).pin_memory() for a in (W_h, sc_h, bs_h))
    out_pin = tuple(torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in out)
    xd, Wd, scd, bsd = (torch.empty_like(t, device=device) for t in (x_pin, W_pin, sc_pin, bs_pin))
    h2d = sum(t.numel() * t.element_size() for t in (x_pin, W_pin, sc_pin, bs_pin))
    d2h = sum(t.numel() * t.element_size() for t in out_pin)

    # Rows are independent, so the copy of x is cut into row blocks on a copy
    # stream and each block's call starts as soon as its rows have landed: the
    # calls hide behind the host-to-device copy, which the host link bounds
    # (~210 GB/s on this part, whatever the number of streams).
    copy_stream = torch.cuda.Stream(device)
    n_blocks = 4 if M % 4 == 0 else 1
    rows_b = M // n_blocks
    step_done = torch.cuda.Event()
    step_done.record(stream)

    def e2e_step():
        copy_stream.wait_event(step_done)  # the previous step no longer reads xd
        landed = []
        with torch.cuda.stream(copy_stream):
            for d, h in ((Wd, W_pin), (scd, sc_pin), (bsd, bs_pin)):
                d.copy_(h, non_blocking=True)
            for b in range(n_blocks):
                rs = slice(b * rows_b, (b + 1) * rows_b)
                xd[rs].copy_(x_pin[rs], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
                landed.append(ev)
        with torch.cuda.stream(stream):
            for b in range(n_blocks):
                rs = slice(b * rows_b, (b + 1) * rows_b)
                stream.wait_event(landed[b])
                call(stream, xd[rs], Wd, scd, bsd, tuple(o[rs] for o in out))
            for h, d in zip(out_pin, out):
                h.copy_(d, non_blocking=True)
            step_done.record(stream)
    n_e2e = max(3, min(args.steps, 100))
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True); t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    step_done.record(stream)  # the first copies start after t0
    for _ in range(n_e2e):
        e2e_step()
    t1.record(stream)
    t1.synchronize()
    e2e_ms = reduce_max(t0.elapsed_time(t1), world, device)
    e2e_us = e2e_ms * 1e3 / (n_e2e * world)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cores = host_cores()
        t = cpu_oracle_time(x_h, W_h, sc_h, bs_h, M, cores)
        reps = 1
        if t * cores < 10.0:
            reps = 2
            t = (t + cpu_oracle_time(x_h, W_h, sc_h, bs_h, M, cores)) / 2
        cpu = {"value": t * 1e6, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"full {M}-row call, mean of {reps}"}

    line = {
        "metric": METRIC, "value": us_call, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "K": K, "path": path,
                   "cuda_graph": f"{GRAPH_CALLS} calls per graph replay",
                   "l2": "inputs larger than L2: x is 168 MB per call (L2 129 MB), no flush",
                   "inputs": "x bf16 N(0,1) seed 0 (rank r: rows 4096r..), W fp32 std K^-1/2"},
        "hbm_gbs": alg_bytes / (us_call * 1e-6) / 1e9,
        "roofline_pct_of_8tbs": alg_bytes / (us_call * 1e-6) / 8e12 * 100,
        "rows_per_s": M / (us_call * 1e-6),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": kernel_name, "kernel_us": k_us,
                     "launches_per_call": launches_per_call,
                     "traffic": profiled_traffic(kernel_name),
                     "algorithmic_bytes": alg_bytes,
                     "contraction_phase_us": contract_us,
                     "contraction_phase_frac": alg_bytes / (contract_us * 1e-6) / 1e9 / peak},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "calls_per_step": n_blocks, "rows_per_call": rows_b,
                "note": (f"one step = {n_blocks} hc_mix_fused calls of {rows_b} rows each "
                         f"(each converts W again), every call starting once its rows "
                         f"have landed from pinned host memory")},
        "gpu_launches": args.steps * launches_per_call,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


GRAPH_CALLS = 10  # calls per CUDA graph in the timed loops


def calls_graphs(fn, stream):
    """CUDA graphs holding GRAPH_CALLS calls of fn() and one call of it."""
    import torch
    graphs = []
    for n in (GRAPH_CALLS, 1):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(n):
                fn()
        graphs.append(g)
    return graphs


def replay_calls(graphs, calls: int) -> None:
    """Exactly `calls` calls: replays of the GRAPH_CALLS-call graph, then of
    the one-call graph for the remainder."""
    many, one = graphs
    for _ in range(calls // GRAPH_CALLS):
        many.replay()
    for _ in range(calls % GRAPH_CALLS):
        one.replay()


def graph_us(fn, stream, replays: int, warmup: int = 5) -> float:
    """Device time per replay of a CUDA graph holding fn(), in µs."""
    import torch
    with torch.cuda.stream(stream):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(replays):
            g.replay()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) * 1e3 / replays


def run_sweep(args):
    """The decode sweep, the outlier config, the split-K / full-K A/B and the
    86-call forward."""
    import numpy as np
    import torch

    import hcmix_inputs as hi
    from hyper_connection_mix_gb300 import binding, traffic

    device = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device)
    dev = lambda a: torch.from_numpy(a).to(device)
    W, sc, bs = dev(hi.make_w()), dev(hi.make_scale()), dev(hi.make_base())

    def fused_case(x, path, calls=100):
        M, K = x.shape
        ws = binding.alloc_workspace(M, K, device)
        out = (torch.empty(M, 4, device=device), torch.empty(M, 4, device=device),
               torch.empty(M, 4, 4, device=device))

        def fn():  # `calls` back-to-back calls per graph, as a decode loop issues them
            for _ in range(calls):
                binding.hc_mix_fused(x, W, sc, bs, ITERS, RMS_EPS, HC_EPS, out=out, workspace=ws,
                                     stream=stream, path=path)
        return graph_us(fn, stream, replays=10) / calls

    x256 = hi.make_x(256)
    for M in (1, 4, 16, 64, 128, 256):
        x = torch.from_numpy(np.ascontiguousarray(x256[:M]).view(np.int16)).view(
            torch.bfloat16).to(device)
        for path in ("simt", "tc"):
            us = fused_case(x, path)
            gbs = traffic.algorithmic_bytes(M, K_COLS) / (us * 1e-6) / 1e9
            print(json.dumps({"config": f"decode M={M} K={K_COLS}", "path": path,
                              "us_per_call": us, "hbm_gbs": gbs,
                              "auto_path": binding.hc_mix_auto_path(M)}), flush=True)
    x = torch.from_numpy(hi.make_x(512, outliers=True).view(np.int16)).view(
        torch.bfloat16).to(device)
    us = fused_case(x, "auto", calls=20)
    print(json.dumps({"config": f"M=512 outliers K={K_COLS}", "path": binding.hc_mix_auto_path(512),
                      "us_per_call": us,
                      "hbm_gbs": traffic.algorithmic_bytes(512, K_COLS) / (us * 1e-6) / 1e9}),
          flush=True)

    # The page's A/B of its two designs at prefill sizes (its table: rows,
    # stock split-K -> fused full-K, us per call), here on the same CUDA-core
    # arithmetic, with the tensor-core split-K path beside them.
    designs = {"simt": "stock split-K (CUDA cores)", "simt_fullk": "fused full-K (CUDA cores)",
               "tc": "split-K (tensor cores)",
               "tc_tf32x3": "split-K (tensor cores, the page's tf32x3 chunk dots)"}
    x4096 = hi.make_x(4096)
    for M in (512, 1024, 2048, 4096):
        x = torch.from_numpy(np.ascontiguousarray(x4096[:M]).view(np.int16)).view(
            torch.bfloat16).to(device)
        for path, design in designs.items():
            us = fused_case(x, path, calls=10)
            print(json.dumps({"config": f"A/B M={M} K={K_COLS}", "path": path, "design": design,
                              "us_per_call": us,
                              "hbm_gbs": traffic.algorithmic_bytes(M, K_COLS) / (us * 1e-6) / 1e9}),
                  flush=True)

    # W packed once (a layer's weight during inference): the same 4096-row
    # call without the per-call conversion of W
    x = torch.from_numpy(x4096.view(np.int16)).view(torch.bfloat16).to(device)
    packed = binding.pack_w(W, stream=stream)
    ws4 = binding.alloc_workspace(4096, K_COLS, device)
    out4 = (torch.empty(4096, 4, device=device), torch.empty(4096, 4, device=device),
            torch.empty(4096, 4, 4, device=device))

    def packed_calls():
        for _ in range(10):
            binding.hc_mix_fused_packed(x, packed, sc, bs, ITERS, RMS_EPS, HC_EPS, out=out4,
                                        workspace=ws4, stream=stream)
    us = graph_us(packed_calls, stream, replays=10) / 10
    print(json.dumps({"config": f"M=4096 K={K_COLS}, W packed once", "path": "tc (packed W)",
                      "us_per_call": us,
                      "hbm_gbs": traffic.algorithmic_bytes(4096, K_COLS) / (us * 1e-6) / 1e9}),
          flush=True)

    # 86 calls per forward (43 layers x 2), M = 16384, one shared x, distinct
    # W / scale / base per call (the stack test's seeds), one CUDA graph
    M, K, calls = 16384, K_COLS, 86
    x = torch.from_numpy(hi.make_x(M).view(np.int16)).view(torch.bfloat16).to(device)
    Ws, scs, bss = [], [], []
    for i in range(calls):
        s_w, s_s, s_b = hi.layer_seeds(i)
        Ws.append(dev(hi.make_w(seed=s_w)))
        scs.append(dev(hi.make_scale(seed=s_s)))
        bss.append(dev(hi.make_base(seed=s_b)))
    ws = binding.alloc_workspace(M, K, device)
    outs = [(torch.empty(M, 4, device=device), torch.empty(M, 4, device=device),
             torch.empty(M, 4, 4, device=device)) for _ in range(calls)]

    def forward():
        for i in range(calls):
            binding.hc_mix_fused(x, Ws[i], scs[i], bss[i], ITERS, RMS_EPS, HC_EPS, out=outs[i],
                                 workspace=ws, stream=stream, path="auto")
    us = graph_us(forward, stream, replays=5, warmup=2)
    per_call = traffic.algorithmic_bytes(M, K)
    print(json.dumps({"config": f"86-call forward M={M} K={K} (CUDA graph)",
                      "path": binding.hc_mix_auto_path(M), "us_per_forward": us,
                      "us_per_call": us / calls,
                      "hbm_gbs": calls * per_call / (us * 1e-6) / 1e9,
                      "roofline_us_at_8tbs": calls * per_call / 8e12 * 1e6}), flush=True)


def run_protocols(args):
    """The 4096-row call timed two more ways, and the oracle's timings.

    GPU: (i) four distinct x buffers in rotation, one CUDA graph of four calls
    (x never comes from L2; W stays warm); (ii) each call alone after a 512 MB
    memset that is not timed (x and W cold), median of the calls.  Host: the
    oracle on one thread and on every host core for the 16-row, 512-row
    (outlier), 4096-row and decode configurations in full, and for the 86-call
    forward at 16384 rows on every core (the one-thread figure is one call,
    scaled by 86, and says so)."""
    import numpy as np
    import torch

    import hcmix_inputs as hi
    import oracle
    from hyper_connection_mix_gb300 import binding, traffic

    device = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device)
    M, K = M_ROWS, K_COLS
    dev = lambda a: torch.from_numpy(a).to(device)
    x_h = hi.make_x(M)
    W_h, sc_h, bs_h = hi.make_w(), hi.make_scale(), hi.make_base()
    W, sc, bs = dev(W_h), dev(sc_h), dev(bs_h)
    xs = [torch.from_numpy(x_h.view(np.int16)).view(torch.bfloat16).to(device) for _ in range(4)]
    ws = binding.alloc_workspace(M, K, device)
    out = (torch.empty(M, 4, device=device), torch.empty(M, 4, device=device),
           torch.empty(M, 4, 4, device=device))
    alg = traffic.algorithmic_bytes(M, K)

    def call(x):
        binding.hc_mix_fused(x, W, sc, bs, ITERS, RMS_EPS, HC_EPS, out=out, workspace=ws,
                             stream=stream, path="auto")

    def rotation():
        for x in xs:
            call(x)
    us = graph_us(rotation, stream, replays=max(3, min(args.steps, 200)), warmup=args.warmup) / 4
    print(json.dumps({"config": f"M={M} K={K}, 4 x buffers in rotation (warm W)",
                      "us_per_call": us, "hbm_gbs": alg / (us * 1e-6) / 1e9}), flush=True)

    scrub = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    times = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(args.warmup + max(3, min(args.steps, 100))):
            scrub.fill_(i & 0xff)
            e0.record(stream)
            call(xs[0])
            e1.record(stream)
            e1.synchronize()
            if i >= args.warmup:
                times.append(e0.elapsed_time(e1) * 1e3)
    us = float(np.median(times))
    print(json.dumps({"config": f"M={M} K={K}, each call after a 512 MB scrub (cold x and W)",
                      "us_per_call": us, "hbm_gbs": alg / (us * 1e-6) / 1e9,
                      "calls": len(times)}), flush=True)
    del xs, scrub
    torch.cuda.empty_cache()

    # the oracle: one thread and every core, in full
    oracle.build()
    cores = host_cores()

    def oracle_s(x, W_, sc_, bs_, threads):
        t0 = time.perf_counter()
        oracle.fused(np.ascontiguousarray(x), W_, sc_, bs_, ITERS, RMS_EPS, HC_EPS, threads=threads)
        return time.perf_counter() - t0
    cases = [("M=16", x_h[:16]), ("M=512 outliers", hi.make_x(512, outliers=True)),
             (f"M={M}", x_h)] + [(f"decode M={m}", x_h[:m]) for m in (1, 4, 16, 64, 128, 256)]
    for name, x in cases:
        for threads in (1, cores):
            s_ = oracle_s(x, W_h, sc_h, bs_h, threads)
            print(json.dumps({"config": f"oracle {name} K={K}", "threads": threads,
                              "us_per_call": s_ * 1e6}), flush=True)
    M5, calls = 16384, 86
    x5 = hi.make_x(M5)
    t_all = 0.0
    for i in range(calls):
        s_w, s_s, s_b = hi.layer_seeds(i)
        t_all += oracle_s(x5, hi.make_w(seed=s_w), hi.make_scale(seed=s_s),
                          hi.make_base(seed=s_b), cores)
    s_w, s_s, s_b = hi.layer_seeds(0)
    t_one = oracle_s(x5, hi.make_w(seed=s_w), hi.make_scale(seed=s_s), hi.make_base(seed=s_b), 1)
    print(json.dumps({"config": f"oracle 86-call forward M={M5} K={K}", "threads": cores,
                      "us_per_forward": t_all * 1e6}), flush=True)
    print(json.dumps({"config": f"oracle 86-call forward M={M5} K={K}", "threads": 1,
                      "us_per_forward": t_one * calls * 1e6,
                      "extrapolated": "one call on one thread, times 86"}), flush=True)


def run_profile(args):
    """Four hc_mix_fused calls of --profile-rows rows (seeded inputs), then a
    check of the device status word; for ncu captures of one launch."""
    import numpy as np
    import torch

    import hcmix_inputs as hi
    from hyper_connection_mix_gb300 import binding

    M = args.profile_rows
    path = args.path if args.path != "auto" else binding.hc_mix_auto_path(M)
    x = torch.from_numpy(hi.make_x(M).view(np.int16)).view(torch.bfloat16).cuda()
    W, sc, bs = (torch.from_numpy(a).cuda() for a in (hi.make_w(), hi.make_scale(), hi.make_base()))
    ws = binding.alloc_workspace(M, K_COLS)
    out = (torch.empty(M, 4, device="cuda"), torch.empty(M, 4, device="cuda"),
           torch.empty(M, 4, 4, device="cuda"))
    for _ in range(4):
        binding.hc_mix_fused(x, W, sc, bs, ITERS, RMS_EPS, HC_EPS, out=out, workspace=ws, path=path)
    torch.cuda.synchronize()
    status = binding.hc_mix_device_status(ws)
    print(json.dumps({"profile_rows": M, "path": path, "device_status": status}), flush=True)
    if status != 0:
        raise SystemExit(1)


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    rank, world, local = dist_env()
    if args.profile_rows:
        if rank == 0:
            run_profile(args)
        return
    if args.sweep:
        if rank == 0:
            run_sweep(args)
        return
    if args.protocols:
        if rank == 0:
            run_protocols(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
