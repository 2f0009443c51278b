"""Benchmark of the low-latency AllReduce on one B300 (virtual ranks).

Metric: microseconds per AllReduce of 8 virtual ranks x 16 KiB bf16 (8192
elements per rank), and GB/s of the 64 MiB-per-rank AllReduce, each against
its roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Latency leg (the headline `value`): one step = one persistent launch that
runs ITERS back-to-back AllReduces on the same buffers with no barrier
between them (the 16 KiB, 8-rank decode-step shape). L2 is flushed between
steps by writing a 256 MiB buffer outside the timed events.
Bandwidth leg: one step = BW_REPS AllReduces of 64 MiB per rank over 8
ranks with the fixed-order two-shot path; its 1 GiB of inputs and outputs
per AllReduce is larger than L2. Each step (the latency leg's launch, the
bandwidth leg's BW_REPS back-to-back launches) is timed with CUDA events on
the launching stream.

With --gpus N > 1 (torchrun, one process per GPU) every rank runs an
independent replica: the path has no exchange between GPUs. Rank 0 prints
one JSON line with the max over ranks.

--impl reference times the CPU oracle (oracle/, numpy) on the same
workload, on the host cores, a bounded sample per step.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per AllReduce (8 virtual ranks, 16 KB bf16) and GB/s at 64 MB vs roofline"
NRANKS = 8
DTYPE = "bf16"
COUNT = 8192               # 16 KiB bf16 per rank
ITERS = 10000              # AllReduces per persistent launch in the latency leg
BW_COUNT = 32 << 20        # 64 MiB bf16 per rank
BW_REPS = 10               # AllReduces per step in the bandwidth leg
E2E_CALLS = 200            # host-buffer calls per step in the end-to-end leg
E2E_WARMUP_S = 0.5         # seconds of host-buffer calls before the end-to-end leg is timed
FLUSH_BYTES = 256 << 20    # > 126 MB L2
FALLBACK_HBM_GBS = 6400.0


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--protocol", default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration table")
    ap.add_argument("--leg", default="all",
                    choices=["all", "latency", "bandwidth", "llbuffer", "config", "polls", "segments"],
                    help="run one leg only (small profiling cases); llbuffer: the LL buffer rows alone; "
                         "config: one row of the per-configuration table (--case); segments: the "
                         "ReduceScatter / AllGather bandwidth row at --bw-mib MiB per rank")
    ap.add_argument("--case", default="C4_sentinel", choices=sorted(CONFIG_CASES) + sorted(FUSED_CASES),
                    help="row for --leg config")
    ap.add_argument("--iters", type=int, default=ITERS, help="AllReduces per latency launch")
    ap.add_argument("--bw-mib", type=int, default=BW_COUNT * 2 >> 20, help="MiB per rank, bandwidth leg")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ helpers
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg, device=None):
    if pg is not None:
        if device is not None:
            pg.barrier(device_ids=[device])
        else:
            pg.barrier()


def max_over_ranks(pg, value, device="cpu"):
    if pg is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, value, device="cpu"):
    if pg is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    pg.all_reduce(t)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


# the translation unit of the kernels whose DRAM traffic profiles/ records
KERNEL_SOURCES = ("tp_allreduce_persistent_b300/csrc/llar_kernels.cu",
                  "tp_allreduce_persistent_b300/csrc/llar_device.cuh",
                  "tp_allreduce_persistent_b300/csrc/llar_internal.h",
                  "include/llar_llbuffer.cuh", "include/llar_llbuffer.h")


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(os.path.basename(rel).encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    sources are unchanged since it was captured; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    item = rec.get(kernel, {})
    if item.get("workload") != workload or item.get("source_hash") != kernel_source_hash():
        return None
    return item.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        return self.parse(self.lines)

    @staticmethod
    def parse(lines):
        """Median SM clock, max clock and the throttle reasons seen active."""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ our CUDA path
def _events(n):
    import torch
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]


def latency_leg(args, llar, inputs, torch, dev, stream, flush, pg, local):
    """ITERS back-to-back 16 KiB AllReduces per launch; returns a dict."""
    iters = args.iters
    x = inputs.normal(NRANKS, COUNT, DTYPE, seed=1, scale=0.02)
    ins = [x[r].to(dev) for r in range(NRANKS)]
    outs = [torch.empty_like(t) for t in ins]
    proto = args.protocol
    for _ in range(args.warmup):
        llar.llar_allreduce_iters(ins, outs, COUNT, proto, iters, 0, 0, 0.0)
    torch.cuda.synchronize()
    used_proto, g, t, _ = llar.llar_last_launch()
    ev = _events(args.steps)
    barrier(pg, local)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(k & 0xFF)  # evict L2 between timed launches (outside the events)
        ev[k][0].record(stream)
        llar.llar_allreduce_iters(ins, outs, COUNT, proto, iters, 0, 0, 0.0)
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    barrier(pg, local)
    wall = time.perf_counter() - wall0
    code = llar.llar_get_status()[0]
    if code != llar.OK:
        raise RuntimeError(f"device status {code} during the latency leg")
    step_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    placed = llar.llar_sol_probe_placed()  # over the CTAs a launch of this shape places
    dep = dependent_chain_us(args, llar, torch, ins, outs, stream, flush)
    return {"us_per_ar": step_ms * 1e3 / iters, "step_ms": step_ms, "proto": used_proto,
            "G": g, "T": t, "wall_s": wall, "x": x, "dependent": dep, "placed": placed}


def dependent_chain_us(args, llar, torch, ins, outs, stream, flush):
    """The same shape as a chain of DEPENDENT AllReduces in one persistent
    launch: each one's input is 1/N times the previous output (rounded), so
    no AllReduce can start before the previous one has finished everywhere
    and the values stay put. Microseconds per AllReduce, mean over steps."""
    iters, proto = args.iters, args.protocol
    for _ in range(max(1, args.warmup)):
        llar.llar_allreduce_iters(ins, outs, COUNT, proto, iters, 0, 0, 1.0 / NRANKS)
    torch.cuda.synchronize()
    used = llar.llar_last_launch()
    ev = _events(args.steps)
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        ev[k][0].record(stream)
        llar.llar_allreduce_iters(ins, outs, COUNT, proto, iters, 0, 0, 1.0 / NRANKS)
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    if llar.llar_get_status()[0] != llar.OK:
        raise RuntimeError("device status not ok in the dependent chain")
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    return {"us_per_ar": ms * 1e3 / iters, "proto": used[0], "G": used[1], "T": used[2]}


def bandwidth_leg(args, llar, torch, dev, stream, pg, local):
    """BW_REPS AllReduces of bw_mib MiB per rank per step, fixed two-shot."""
    count = (args.bw_mib << 20) // 2
    gen = torch.Generator(device=dev)
    bw_ins = []
    for r in range(NRANKS):
        gen.manual_seed(5 + r)
        bw_ins.append(torch.randn(count, device=dev, generator=gen).to(torch.bfloat16))
    bw_outs = [torch.empty_like(a) for a in bw_ins]
    for _ in range(args.warmup):
        llar.llar_allreduce(bw_ins, bw_outs, count, "fixed_twoshot")
    torch.cuda.synchronize()
    shape = llar.llar_last_launch()
    # one event pair per step around its BW_REPS launches, back to back as a
    # stream of AllReduces runs (an event pair around every launch would add
    # its own gap to each); 1 GiB of inputs and outputs per launch is more
    # than L2 holds, so no launch finds the previous one's data there
    bev = _events(args.steps)
    barrier(pg, local)
    torch.cuda.synchronize()
    for i in range(args.steps):
        bev[i][0].record(stream)
        for _ in range(BW_REPS):
            llar.llar_allreduce(bw_ins, bw_outs, count, "fixed_twoshot")
        bev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(pg, local)
    launch_s = statistics.mean(a.elapsed_time(b) for a, b in bev) * 1e-3 / BW_REPS
    alg_bytes = 2 * NRANKS * count * 2
    return {"gbs": alg_bytes / launch_s / 1e9, "launch_s": launch_s, "alg_bytes": alg_bytes,
            "count": count, "G": shape[1], "T": shape[2]}


def e2e_leg(args, llar, torch, stream, x, pg, local):
    """One AllReduce per llar_allreduce_host call on pinned host buffers."""
    proto = args.protocol
    hx = x.contiguous().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    llar.llar_host_register(hx)  # pinned buffers declared once, as a serving loop would
    llar.llar_host_register(hy)
    try:
        # warm-up: W steps of E2E_CALLS calls each, as timed, and at least
        # E2E_WARMUP_S of calls: on a fresh box the host link takes a few
        # tenths of a second of traffic to settle (one box: 15 -> 7.3 us per
        # call over the first 0.26 s)
        done, t0 = 0, time.perf_counter()
        while done < args.warmup * E2E_CALLS or time.perf_counter() - t0 < E2E_WARMUP_S:
            llar.llar_allreduce_host(hx, hy, COUNT, proto)
            done += 1
        torch.cuda.synchronize()
        calls = max(3, args.steps // 5) * E2E_CALLS
        e0, e1 = _events(1)[0]
        barrier(pg, local)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(calls):
            llar.llar_allreduce_host(hx, hy, COUNT, proto)
        e1.record(stream)
        torch.cuda.synchronize()
    finally:
        llar.llar_host_unregister(hx)
        llar.llar_host_unregister(hy)
    return e0.elapsed_time(e1) * 1e3 / calls


def timed_config(llar, torch, dev, stream, n, dtype, count, proto, iters, chain=0.0, chunk=None, max_bytes=None):
    """One workload configuration: a warm-up launch of min(iters, 20)
    AllReduces, then one timed launch of `iters`; microseconds per AllReduce."""
    from tp_allreduce_persistent_b300 import inputs
    llar.llar_init(n, dtype, max_bytes or max(count * inputs.ELEM_BYTES[dtype], 4096))
    try:
        if chunk:
            llar.llar_set_sentinel_chunk(chunk)
        gen = torch.Generator(device=dev)
        gen.manual_seed(7)
        td = inputs.TORCH_DTYPE[dtype]
        ins = [(torch.randn(count, device=dev, generator=gen) * 0.02).to(td) for _ in range(n)]
        outs = [torch.empty_like(t) for t in ins]
        llar.llar_allreduce_iters(ins, outs, count, proto, min(iters, 20), 0, 0, chain)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        llar.llar_allreduce_iters(ins, outs, count, proto, iters, 0, 0, chain)
        b.record(stream)
        torch.cuda.synchronize()
        if llar.llar_get_status()[0] != llar.OK:
            raise RuntimeError("device status not ok")
        return round(a.elapsed_time(b) * 1e3 / iters, 3)
    finally:
        llar.llar_destroy()


# single rows of the per-configuration table, for profiling one kernel
# (`--leg config --case NAME`): (ranks, dtype, elements per rank, protocol,
# AllReduces per launch, chain scale, sentinel chunk bytes)
CONFIG_CASES = {
    "C3_ll128_1MiB": (8, "bf16", 1024 * 512, "ll128", 200, 0.0, None),
    "C3_ll128_16KiB": (8, "bf16", 16 * 512, "ll128", 1000, 0.0, None),
    "C4_sentinel": (8, "fp16", 32768, "sentinel", 1000, 0.0, 8192),
    "C5_ll128_chain_N8": (8, "bf16", 65536, "ll128", 160, 0.5, None),
    "C3_ll128_direct_1MiB": (8, "bf16", 1024 * 512, "ll128_direct", 200, 0.0, None),
    "headline_dependent_ll": (8, "bf16", 8192, "ll", 10000, 1.0 / 8, None),
    "C3_ll128_direct_16KiB": (8, "bf16", 16 * 512, "ll128_direct", 1000, 0.0, None),
    "C2_ll": (4, "bf16", 8192, "ll", 10000, 0.0, None),
    "C2_sentinel": (4, "bf16", 8192, "sentinel", 10000, 0.0, 16384),
    "C5_sentinel_chain_N8": (8, "bf16", 65536, "sentinel", 160, 0.5, None),
    "C5_ll_chain_N4": (4, "bf16", 65536, "ll", 160, 0.5, None),
    "C5_ll_chain_N8": (8, "bf16", 65536, "ll", 160, 0.5, None),
}
# fused decode layers for `--leg config --case NAME`: (ranks, tokens m, K, H), bf16
FUSED_CASES = {
    "fused_m1_k1024": (8, 1, 1024, 8192),
    "fused_m16_k1024": (8, 16, 1024, 8192),
}


def fused_case_us(llar, torch, dev, stream, n, m, k, h, calls=4):
    """A warm-up call, then `calls` timed calls of the fused layer on one
    weight set; microseconds per call."""
    from tp_allreduce_persistent_b300 import inputs
    x, w = inputs.linear_layer(n, m, k, h, "bf16", seed=100)
    xs = [x[r].to(dev) for r in range(n)]
    ws = [w[r].to(dev) for r in range(n)]
    outs = [torch.empty(m * h, dtype=torch.bfloat16, device=dev) for _ in range(n)]
    with llar.LLBuffer(n, m * h * 2) as buf:
        buf.fused_linear_allreduce(xs, ws, outs, m, k, h, "bf16")
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(calls):
            buf.fused_linear_allreduce(xs, ws, outs, m, k, h, "bf16")
        b.record(stream)
        torch.cuda.synchronize()
        if buf.status()[0] != llar.OK:
            raise RuntimeError("LL buffer status not ok")
    return round(a.elapsed_time(b) * 1e3 / calls, 3)


def configs_leg(llar, torch, dev, stream):
    """Per-AllReduce time of each workload configuration (persistent launches)."""
    def timed(n, dtype, count, proto, iters, chain=0.0, chunk=None, max_bytes=None):
        return timed_config(llar, torch, dev, stream, n, dtype, count, proto, iters, chain, chunk, max_bytes)

    out = {
        "C1_2ranks_128B_fp32_us": {p: timed(2, "fp32", 32, p, 1000) for p in ("ll", "fixed_oneshot")},
        "C2_4ranks_16KiB_bf16_us": {p: timed(4, "bf16", 8192, p, 10000, chunk=16384) for p in ("ll", "sentinel")},
        "C3_ll128_8ranks_bf16_us": {f"{kb}KiB": timed(8, "bf16", kb * 512, "ll128", 200 if kb > 64 else 1000)
                                    for kb in (4, 16, 64, 256, 1024)},
        # the variant whose AllGather reads the owners' lines directly
        "C3_ll128_direct_8ranks_bf16_us": {f"{kb}KiB": timed(8, "bf16", kb * 512, "ll128_direct",
                                                             200 if kb > 64 else 1000)
                                           for kb in (4, 16, 64, 256, 1024)},
        "fixed_twoshot_8ranks_bf16_us": {f"{kb}KiB": timed(8, "bf16", kb * 512, "fixed_twoshot",
                                                           200 if kb > 64 else 1000)
                                         for kb in (4, 16, 64, 256, 1024)},
        C4_KEY: timed(8, "fp16", 32768, "sentinel", 1000, chunk=8192),
        "C5_chain_160_layers_128KiB_bf16_us": {
            f"N{n}": {p: timed(n, "bf16", 65536, p, 160, chain=0.5)  # the library's sentinel chunk
                      for p in ("ll", "sentinel", "ll128", "ll128_direct", "fixed_oneshot", "fixed_twoshot")}
            for n in (4, 8)},
    }
    # the headline shape as a chain of dependent AllReduces (input of each =
    # RNE(previous output / 8)), every protocol
    out["dependent_chain_8ranks_16KiB_bf16_us"] = {
        p: timed(8, "bf16", 8192, p, 2000, chain=1.0 / 8) for p in ("ll", "sentinel", "ll128", "ll128_direct",
                                                                   "fixed_oneshot", "fixed_twoshot")}
    out["C2_mode_b_graph_10000_launches_4ranks_16KiB_bf16_us"] = {
        p: mode_b_us(llar, torch, dev, stream, p) for p in ("ll", "sentinel")}
    out["noalloc_8ranks_16KiB_bf16"] = noalloc_rows(llar, torch, dev, stream)
    # single calls, one launch each, replayed from a CUDA graph of 200 calls
    # (GPU time per call including launch gaps, without host overhead)
    def graph_call_us(kind, proto, n=8, count=8192, dtype="bf16"):
        from tp_allreduce_persistent_b300 import inputs
        llar.llar_init(n, dtype, count * inputs.ELEM_BYTES[dtype])
        try:
            td = inputs.TORCH_DTYPE[dtype]
            seg = -(-count // n)
            full_in = [torch.randn(count, device=dev).to(td) for _ in range(n)]
            seg_in = [torch.randn(seg, device=dev).to(td) for _ in range(n)]
            full_out = [torch.empty(count, dtype=td, device=dev) for _ in range(n)]
            seg_out = [torch.empty(seg, dtype=td, device=dev) for _ in range(n)]
            call = {"allreduce": lambda: llar.llar_allreduce(full_in, full_out, count, proto),
                    "reduce_scatter": lambda: llar.llar_reduce_scatter(full_in, seg_out, count, proto),
                    "all_gather": lambda: llar.llar_all_gather(seg_in, full_out, count, proto)}[kind]
            call()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(200):
                    call()
            g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(5):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            if llar.llar_get_status()[0] != llar.OK:
                raise RuntimeError("device status not ok")
            return round(a.elapsed_time(b) * 1e3 / 1000, 3)
        finally:
            llar.llar_destroy()

    out["single_call_graph_8ranks_16KiB_bf16_us"] = {
        "allreduce": {p: graph_call_us("allreduce", p) for p in ("ll", "sentinel", "ll128", "ll128_direct",
                                                                 "fixed_oneshot", "fixed_twoshot")},
        "reduce_scatter": {p: graph_call_us("reduce_scatter", p) for p in ("ll", "sentinel", "ll128", "fixed_oneshot")},
        "all_gather": {p: graph_call_us("all_gather", p) for p in ("ll", "sentinel", "fixed_oneshot")},
    }
    # point-to-point hand-off along a ring of 8 ranks (every rank sends 16 KiB
    # bf16 to the next), back-to-back transfers in one launch
    def p2p_us(proto, iters):
        n, count = 8, 8192
        llar.llar_init(n, "bf16", count * 2)
        try:
            sends = [torch.randn(count, device=dev).to(torch.bfloat16) for _ in range(n)]
            recvs = [torch.empty_like(t) for t in sends]
            ring = [(r + 1) % n for r in range(n)]
            llar.llar_sendrecv(sends, recvs, ring, count, proto, 20)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            llar.llar_sendrecv(sends, recvs, ring, count, proto, iters)
            b.record(stream)
            torch.cuda.synchronize()
            if llar.llar_get_status()[0] != llar.OK:
                raise RuntimeError("device status not ok")
            return round(a.elapsed_time(b) * 1e3 / iters, 3)
        finally:
            llar.llar_destroy()

    out["p2p_ring_8ranks_16KiB_bf16_us"] = {p: p2p_us(p, 10000) for p in ("ll", "sentinel", "fixed_oneshot")}
    out.update(llbuffer_rows(llar, torch, dev, stream))
    sweep = {}
    for mib in (1, 4, 16, 64, 256):
        count = (mib << 20) // 2
        iters = 3 if mib >= 64 else 10
        us = timed(8, "bf16", count, "fixed_twoshot", iters, max_bytes=mib << 20)
        sweep[f"{mib}MiB"] = {"us": us, "GB/s": round(2 * 8 * count * 2 / (us * 1e-6) / 1e9, 1)}
    out["C5_sweep_8ranks_bf16_fixed_twoshot"] = sweep
    out[SEG_KEY] = segments_rows(llar, torch, dev, stream)
    return out


SEG_KEY = "segments_8ranks_64MiB_bf16_fixed"


def segments_rows(llar, torch, dev, stream, mib=64, n=8, reps=10, warmup=3):
    """The standalone halves at bandwidth size: ReduceScatter and AllGather
    of n ranks x `mib` MiB bf16 by direct copies (AUTO's choice there), `reps`
    launches back to back between one event pair. Algorithmic bytes per
    launch: ReduceScatter reads n x S and writes S, AllGather reads S and
    writes n x S (S = mib MiB); both more than L2 holds."""
    count = (mib << 20) // 2
    seg = count // n
    torch.cuda.synchronize()
    torch.cuda.empty_cache()  # fresh allocations, not blocks cached by earlier rows
    llar.llar_init(n, "bf16", mib << 20)
    try:
        gen = torch.Generator(device=dev)
        gen.manual_seed(11)
        full_in = [torch.randn(count, device=dev, generator=gen).to(torch.bfloat16) for _ in range(n)]
        seg_buf = [torch.empty(seg, dtype=torch.bfloat16, device=dev) for _ in range(n)]
        full_out = [torch.empty(count, dtype=torch.bfloat16, device=dev) for _ in range(n)]
        alg = (n + 1) * count * 2
        rows = {}
        for kind, call in (("reduce_scatter", lambda: llar.llar_reduce_scatter(full_in, seg_buf, count, "auto")),
                           ("all_gather", lambda: llar.llar_all_gather(seg_buf, full_out, count, "auto"))):
            for _ in range(warmup):
                call()
            torch.cuda.synchronize()
            shape = llar.llar_last_launch()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                call()
            b.record(stream)
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / reps
            rows[kind] = {"us": round(us, 2), "GB/s": round(alg / (us * 1e-6) / 1e9, 1),
                          "algorithmic_bytes": alg, "protocol": shape[0], "ctas_per_rank": shape[1],
                          "threads_per_cta": shape[2]}
        if llar.llar_get_status()[0] != llar.OK:
            raise RuntimeError("device status not ok")
        return rows
    finally:
        llar.llar_destroy()


def mode_b_us(llar, torch, dev, stream, proto, n=4, count=8192, launches=10000):
    """C2 Mode B: a CUDA graph of `launches` single-AllReduce launches of
    N=4 x 16 KiB bf16 on the same buffers, replayed; microseconds per launch
    including the gaps between launches (no host overhead)."""
    llar.llar_init(n, "bf16", count * 2)
    try:
        llar.llar_set_sentinel_chunk(16384)
        gen = torch.Generator(device=dev)
        gen.manual_seed(1)
        ins = [(torch.randn(count, device=dev, generator=gen) * 0.02).to(torch.bfloat16) for _ in range(n)]
        outs = [torch.empty_like(t) for t in ins]
        llar.llar_allreduce(ins, outs, count, proto)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(launches):
                llar.llar_allreduce(ins, outs, count, proto)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        if llar.llar_get_status()[0] != llar.OK:
            raise RuntimeError("device status not ok")
        del g
        return round(a.elapsed_time(b) * 1e3 / launches, 3)
    finally:
        llar.llar_destroy()


def noalloc_rows(llar, torch, dev, stream, n=8, count=8192, calls=2000):
    """The allocation-free entry point against llar_allreduce (LL, 8 ranks
    x 16 KiB bf16): GPU time per call when calls are queued back to back
    (the stream stays busy, so the allocation-free call skips its status
    check), and host wall time per call when every call is followed by a
    stream synchronisation (each allocation-free call then finds the stream
    idle and pays its status check: a 4-byte copy and a synchronisation)."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    ins = [(torch.randn(count, device=dev, generator=gen) * 0.02).to(torch.bfloat16) for _ in range(n)]
    outs = [torch.empty_like(t) for t in ins]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def queued(fn):
        for _ in range(20):
            fn()
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(calls):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / calls

    def synced(fn, reps=500):
        for _ in range(20):
            fn()
            torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
            torch.cuda.synchronize()
        return (time.perf_counter() - t0) * 1e6 / reps

    def noalloc():
        llar.llar_allreduce_noalloc(ins, outs, count, n, "bf16")

    def regular():
        llar.llar_allreduce(ins, outs, count, "ll")

    rows = {"noalloc_queued_us": round(queued(noalloc), 3),
            "noalloc_sync_each_host_us": round(synced(noalloc), 3)}
    llar.llar_init(n, "bf16", count * 2)
    try:
        rows["allreduce_queued_us"] = round(queued(regular), 3)
        rows["allreduce_sync_each_host_us"] = round(synced(regular), 3)
        if llar.llar_get_status()[0] != llar.OK:
            raise RuntimeError("device status not ok")
    finally:
        llar.llar_destroy()
    return rows


def llbuffer_rows(llar, torch, dev, stream):
    """The LL buffer API: AllReduces built from the public device primitives
    (among them the two-rank 128-byte one-shot), and the row-parallel decode
    linear layer with its AllReduce fused into the GEMV epilogue against
    the unfused pipeline (GEMV launch, then the library's LL AllReduce)."""
    from tp_allreduce_persistent_b300 import inputs
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def per_call_us(fn, iters):
        fn(min(iters, 20))
        torch.cuda.synchronize()
        a.record(stream)
        fn(iters)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / iters

    rows = {}
    for name, n, dtype, count, iters in (("2ranks_128B_fp32", 2, "fp32", 32, 10000),
                                         ("8ranks_16KiB_bf16", 8, "bf16", 8192, 10000)):
        with llar.LLBuffer(n, count * inputs.ELEM_BYTES[dtype]) as buf:
            x = inputs.normal(n, count, dtype, seed=7, scale=0.02, exclude_sentinel=True)
            ins = [x[r].to(dev) for r in range(n)]
            outs = [torch.empty_like(t) for t in ins]
            rows[name] = {}
            for proto in ("ll", "sentinel", "ll128"):
                us = per_call_us(lambda it: buf.allreduce(ins, outs, count, dtype, proto, it),
                                 iters if proto == "ll" else iters // 10)
                if buf.status()[0] != llar.OK:
                    raise RuntimeError("LL buffer status not ok")
                rows[name][proto] = round(us, 3)
    res = {"llbuffer_allreduce_us": rows}

    # decode layers of a hidden-8192 model over 8 ranks (m tokens): attention
    # output projection (K = 8192 / 8) and MLP down projection (K = 28672 / 8);
    # weight sets rotate so that each call streams weights not in L2
    peak = measured_peaks()[0]["hbm_gbs"]
    layers = {}
    for name, m, k, sets in (("attn_out_k1024_m1", 1, 1024, 4), ("attn_out_k1024_m8", 8, 1024, 4),
                             ("attn_out_k1024_m16", 16, 1024, 4), ("mlp_down_k3584_m1", 1, 3584, 2)):
        n, h, dtype = 8, 8192, "bf16"
        xs, ws = [], []
        for sidx in range(sets):
            x, w = inputs.linear_layer(n, m, k, h, dtype, seed=100 + sidx)
            xs.append([x[r].to(dev) for r in range(n)])
            ws.append([w[r].to(dev) for r in range(n)])
        outs = [torch.empty(m * h, dtype=torch.bfloat16, device=dev) for _ in range(n)]
        parts = [torch.empty(m * h, dtype=torch.bfloat16, device=dev) for _ in range(n)]
        llar.llar_init(n, dtype, m * h * 2)
        try:
            with llar.LLBuffer(n, m * h * 2) as buf:
                def fused(s_):
                    buf.fused_linear_allreduce(xs[s_], ws[s_], outs, m, k, h, dtype)

                def unfused(s_):
                    llar.llar_linear_partials(xs[s_], ws[s_], parts, m, k, h, dtype)
                    llar.llar_allreduce(parts, outs, m * h, "ll")

                def gemv(s_):
                    llar.llar_linear_partials(xs[s_], ws[s_], parts, m, k, h, dtype)

                timing = {}
                for label, fn in (("fused", fused), ("unfused", unfused), ("gemv_only", gemv)):
                    for s_ in range(sets):
                        fn(s_)
                    torch.cuda.synchronize()
                    g = torch.cuda.CUDAGraph()
                    reps = 5
                    with torch.cuda.graph(g):
                        for _ in range(reps):
                            for s_ in range(sets):
                                fn(s_)
                    g.replay()
                    torch.cuda.synchronize()
                    a.record(stream)
                    g.replay()
                    b.record(stream)
                    torch.cuda.synchronize()
                    timing[label] = a.elapsed_time(b) * 1e3 / (reps * sets)
                if buf.status()[0] != llar.OK or llar.llar_get_status()[0] != llar.OK:
                    raise RuntimeError("device status not ok")
        finally:
            llar.llar_destroy()
        wbytes = n * k * h * 2
        gbs = wbytes / (timing["fused"] * 1e-6) / 1e9
        layers[name] = {"fused_us": round(timing["fused"], 2), "unfused_us": round(timing["unfused"], 2),
                        "gemv_only_us": round(timing["gemv_only"], 2), "weight_bytes": wbytes,
                        "fused_weight_GB/s": round(gbs, 1), "fused_frac_of_measured_hbm": round(gbs / peak, 4)}
        del xs, ws
    res["fused_linear_allreduce_8ranks_h8192_bf16"] = layers
    return res


# poll-count cases: (ranks, dtype, elements per rank, protocol, AllReduces
# per launch, chain scale, sentinel chunk bytes)
POLL_CASES = {
    "ll_8ranks_16KiB_bf16": (8, "bf16", 8192, "ll", 1000, 0.0, None),
    "ll_8ranks_16KiB_bf16_dependent": (8, "bf16", 8192, "ll", 1000, 1.0 / 8, None),
    "sentinel_8ranks_16KiB_bf16": (8, "bf16", 8192, "sentinel", 1000, 0.0, None),
    "sentinel_C4_8ranks_64KiB_fp16_8KiB_chunks": (8, "fp16", 32768, "sentinel", 200, 0.0, 8192),
    "ll128_8ranks_16KiB_bf16": (8, "bf16", 8192, "ll128", 1000, 0.0, None),
    "ll128_8ranks_1MiB_bf16": (8, "bf16", 1 << 19, "ll128", 100, 0.0, None),
    "ll128_direct_8ranks_16KiB_bf16": (8, "bf16", 8192, "ll128_direct", 1000, 0.0, None),
    "ll128_direct_8ranks_1MiB_bf16": (8, "bf16", 1 << 19, "ll128_direct", 100, 0.0, None),
}


def polls_leg(llar, torch, dev):
    """Polling per AllReduce, counted by the poll-counting build (run with
    LLAR_LIBRARY pointing at it): line loads per AllReduce (all ranks),
    loads per awaited line (1 = the line was there at its first load) and
    polling rounds per wait. Its timings are not the library's."""
    from tp_allreduce_persistent_b300 import inputs
    rows = {}
    for name, (n, dtype, count, proto, iters, chain, chunk) in POLL_CASES.items():
        llar.llar_init(n, dtype, count * inputs.ELEM_BYTES[dtype])
        try:
            if chunk:
                llar.llar_set_sentinel_chunk(chunk)
            gen = torch.Generator(device=dev)
            gen.manual_seed(7)
            td = inputs.TORCH_DTYPE[dtype]
            ins = [(torch.randn(count, device=dev, generator=gen) * 0.02).to(td) for _ in range(n)]
            outs = [torch.empty_like(t) for t in ins]
            llar.llar_allreduce_iters(ins, outs, count, proto, min(iters, 20), 0, 0, chain)
            llar.llar_debug_poll_stats(reset=True)
            llar.llar_allreduce_iters(ins, outs, count, proto, iters, 0, 0, chain)
            rounds, loads, waits, awaited = llar.llar_debug_poll_stats(reset=True)
            if llar.llar_get_status()[0] != llar.OK:
                raise RuntimeError("device status not ok")
            rows[name] = {"line_loads_per_allreduce": round(loads / iters, 1),
                          "lines_awaited_per_allreduce": round(awaited / iters, 1),
                          "loads_per_awaited_line": round(loads / max(awaited, 1), 3),
                          "rounds_per_wait": round(rounds / max(waits, 1), 3)}
        finally:
            llar.llar_destroy()
    return rows


def poll_counts_subprocess():
    """Run the polls leg in a child process on the poll-counting build, if it
    has been built; None otherwise."""
    from tp_allreduce_persistent_b300 import build as b
    if not os.path.exists(b.POLLS_LIB):
        return None
    env = dict(os.environ, LLAR_LIBRARY=b.POLLS_LIB)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--leg", "polls"], env=env,
                       capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout).strip().splitlines()[-1:]}
    return json.loads(r.stdout.strip().splitlines()[-1])["poll_counts"]


C4_KEY = "C4_sentinel_8ranks_64KiB_fp16_8KiB_chunks_us"
C4_CHUNKS = 8  # 64 KiB in 8 KiB chunks


def chunked_floor_us(chunks, l2_us, write_us):
    """Latency floor of an AllReduce carried in `chunks` dependent steps:
    by the credit rule chunk t + 1 leaves only after chunk t has arrived
    from every peer, and each step needs a publication to become visible
    (one write) and a poll that sees it (one L2 round trip); the first
    input read adds one more round trip. With one chunk this is the speed
    of light, 2 x L2 round trip + one write."""
    return l2_us + chunks * (write_us + l2_us)


def per_config_roofline(per_config, sol_us, hbm_gbs, l2_us=None, write_us=None):
    """Each row against its roofline: latency rows (microseconds per
    operation) as speed of light / time, with the speed of light measured in
    this run (2 x L2 round trip + one write: a per-operation floor whatever
    the size); bandwidth rows as GB/s / the measured HBM copy bandwidth.
    The chunked sentinel row is also given against the floor of its
    dependent chunk steps (chunked_floor_us)."""
    def lat(v):
        if isinstance(v, dict):
            return {k: lat(x) for k, x in v.items()}
        return round(sol_us / v, 4) if isinstance(v, (int, float)) and v > 0 else None

    out = {"definition": "latency rows: sol_us / us (above 1 where back-to-back operations of one "
                         "persistent launch overlap: the next one's lines leave before this one's "
                         "reduction); bandwidth rows: GB/s / measured hbm_gbs",
           "sol_us": round(sol_us, 4), "hbm_gbs": hbm_gbs}
    for key, val in per_config.items():
        if key.endswith("_us"):
            out[key] = lat(val)
        elif key in ("C5_sweep_8ranks_bf16_fixed_twoshot", SEG_KEY):
            out[key] = {k: round(v["GB/s"] / hbm_gbs, 4) for k, v in val.items()}
        elif key.startswith("fused_linear"):
            out[key] = {k: v["fused_frac_of_measured_hbm"] for k, v in val.items()}
    c4 = per_config.get(C4_KEY)
    if l2_us is not None and write_us is not None and isinstance(c4, (int, float)) and c4 > 0:
        floor = chunked_floor_us(C4_CHUNKS, l2_us, write_us)
        out["C4_chunked_floor"] = {
            "floor_us": round(floor, 4), "frac": round(floor / c4, 4), "chunks": C4_CHUNKS,
            "definition": "L2 round trip + chunks x (one write + one L2 round trip): the chunks are "
                          "dependent steps (chunk t + 1 leaves after chunk t arrived from every peer)"}
    return out


def run_ours(args, world, rank, local, pg):
    import torch
    from tp_allreduce_persistent_b300 import inputs, llar

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    if args.leg == "config":
        if args.case in FUSED_CASES:
            us = fused_case_us(llar, torch, dev, stream, *FUSED_CASES[args.case])
        else:
            n, dtype, count, proto, iters, chain, chunk = CONFIG_CASES[args.case]
            us = timed_config(llar, torch, dev, stream, n, dtype, count, proto, iters, chain, chunk)
        if rank == 0:
            key = "us_per_call" if args.case in FUSED_CASES else "us_per_allreduce"
            print(json.dumps({"leg": "config", "case": args.case, key: us}))
        return
    if args.leg == "llbuffer":
        if rank == 0:
            print(json.dumps({"leg": "llbuffer", **llbuffer_rows(llar, torch, dev, stream)}))
        return
    if args.leg == "segments":
        if rank == 0:
            print(json.dumps({"leg": "segments", f"segments_8ranks_{args.bw_mib}MiB_bf16_fixed":
                              segments_rows(llar, torch, dev, stream, mib=args.bw_mib)}))
        return
    if args.leg == "polls":
        if rank == 0:
            print(json.dumps({"leg": "polls", "library": os.path.basename(llar.LIB_PATH),
                              "poll_counts": polls_leg(llar, torch, dev)}))
        return
    llar.llar_init(NRANKS, DTYPE, max(args.bw_mib << 20, COUNT * 2))
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peaks, peak_src = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))

    ll_clustered = llar.llar_ll_placement()  # chosen by timing both placements at llar_init
    l2_us, write_us, sol_us = llar.llar_sol_probe()
    detail = llar.llar_sol_probe_detail()
    props = torch.cuda.get_device_properties(local)

    def spread(v):
        v = sorted(v)
        return [round(v[0], 1), round(v[len(v) // 2], 1), round(v[-1], 1)] if v else None
    clocks = ClockSampler(local)
    clocks.start()
    lat = bw = None
    if args.leg in ("all", "latency"):
        lat = latency_leg(args, llar, inputs, torch, dev, stream, flush, pg, local)
    if args.leg in ("all", "bandwidth"):
        bw = bandwidth_leg(args, llar, torch, dev, stream, pg, local)
    clk = clocks.stop()
    e2e_us = None
    if lat is not None and args.leg == "all":
        e2e_us = e2e_leg(args, llar, torch, stream, lat["x"], pg, local)
    llar.llar_destroy()
    per_config = None
    if args.leg == "all" and not args.no_configs:
        per_config = configs_leg(llar, torch, dev, stream)
        if rank == 0:
            per_config["poll_counts"] = poll_counts_subprocess()

    res = {"metric": METRIC, "unit": "us", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "higher_is_better": False, "scaling": "weak",
           "vs_baseline": None, "dtype": "f32-accumulate over bf16",
           "data": "synthetic: N(0,1)*0.02 activations (latency leg), N(0,1) (bandwidth leg), seeded",
           "clocks": clk}
    config = {"replicas": "independent per GPU" if world > 1 else "single GPU",
              "l2": "latency leg: flushed between timed launches (256 MiB write outside the events); "
                    "bandwidth leg: inputs+outputs larger than L2"}
    if lat is not None:
        us = max_over_ranks(pg, lat["us_per_ar"], dev)
        total = sum_over_ranks(pg, args.iters * args.steps, dev)
        res.update({"value": round(us, 4), "ms_per_step": round(lat["step_ms"], 4),
                    "gpu_launches": args.steps, "total_allreduces": int(total),
                    "aggregate_allreduces_per_s": round(total / (lat["step_ms"] * 1e-3 * args.steps), 1),
                    "wall_s_latency_leg": round(lat["wall_s"], 3)})
        config.update({"workload": f"8 virtual ranks x 16 KiB bf16 (8192 elements) AllReduce, "
                                   f"{args.iters} back-to-back per persistent launch",
                       "nranks": NRANKS, "count": COUNT, "iters_per_launch": args.iters,
                       "protocol": lat["proto"], "ctas_per_rank": lat["G"], "threads_per_cta": lat["T"],
                       "ll_clusters_of_n_blocks": bool(ll_clustered)})
        dep_us = max_over_ranks(pg, lat["dependent"]["us_per_ar"], dev)
        res["latency_roofline"] = {
            "kernel": f"k_{lat['proto']}<bf16>", "bound": "latency (L2 round trips)",
            "achieved_us": round(us, 4), "sol_us": round(sol_us, 4),
            "achieved_kind": "per-AllReduce throughput: independent AllReduces back to back in one "
                             "launch, the next one's lines leave before this one's reduction",
            "l2_round_trip_us": round(l2_us, 4), "write_us": round(write_us, 4),
            "frac": round(sol_us / us, 4), "within_2x_sol": bool(us <= 2 * sol_us),
            "dependent": {"us_per_ar": round(dep_us, 4), "frac": round(sol_us / dep_us, 4),
                          "within_2x_sol": bool(dep_us <= 2 * sol_us),
                          "kernel": f"k_{lat['dependent']['proto']}<bf16> (chain)",
                          "kind": f"latency: {args.iters} dependent AllReduces per launch, each input "
                                  "= RNE(output of the previous one / 8)"},
            "placed_worst_pair": {
                "l2_round_trip_us": round(lat["placed"][0], 4), "write_us": round(lat["placed"][1], 4),
                "sol_us": round(lat["placed"][2], 4), "pairs": lat["placed"][3],
                "frac": round(lat["placed"][2] / us, 4), "dependent_frac": round(lat["placed"][2] / dep_us, 4),
                "definition": "the slowest chase among the SMs holding the launch's rank CTAs, and half the "
                              "slowest round trip among the CTA pairs that exchange data"},
            "definition": "SoL = 2 x L2 round trip + one remote write, both measured in this run (medians over "
                          "all SMs and SM pairs; placed_worst_pair: the worst placed pair)",
            "probe_ns_min_median_max": {"l2_chase_per_sm": spread(detail["chase_ns"]),
                                        "pingpong_round_trip_per_pair": spread(detail["rt_ns"])}}
        res["device"] = {"name": props.name, "sms": props.multi_processor_count,
                         "l2_bytes": getattr(props, "L2_cache_size", None),
                         "memory_bytes": props.total_memory}
    if bw is not None:
        gbs = -max_over_ranks(pg, -bw["gbs"], dev)
        mib = args.bw_mib
        wl = f"8 ranks x {mib} MiB bf16, fixed-order two-shot"
        res["bandwidth"] = {
            "value": round(gbs, 1), "unit": "GB/s", "workload": wl,
            "us_per_allreduce": round(bw["launch_s"] * 1e6, 2), "algorithmic_bytes": bw["alg_bytes"],
            "algbw_gbs": round(bw["count"] * 2 / bw["launch_s"] / 1e9, 1),
            "busbw_gbs": round(bw["count"] * 2 / bw["launch_s"] / 1e9 * 2 * (NRANKS - 1) / NRANKS, 1),
            "ctas_per_rank": bw["G"], "threads_per_cta": bw["T"], "launches": args.steps * BW_REPS}
        res["roofline"] = {
            "kernel": "k_fixed_twoshot<bf16>", "bound": "hbm", "achieved": round(gbs, 1),
            "peak": hbm_peak, "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
            "traffic": recorded_traffic("k_fixed_twoshot<bf16>", wl),
            "algorithmic_bytes_per_launch": bw["alg_bytes"],
            "peak_source": f"{peak_src} hbm_gbs (copy bandwidth, burst)",
            "frac_of_nominal_8TBps": round(gbs / 8000.0, 4)}
        config["bandwidth_workload"] = wl
        if lat is None:
            res.update({"value": round(gbs, 1), "unit": "GB/s", "higher_is_better": True,
                        "ms_per_step": round(bw["launch_s"] * 1e3 * BW_REPS, 4),
                        "gpu_launches": args.steps * BW_REPS})
    if e2e_us is not None:
        res["e2e"] = {"value": round(max_over_ranks(pg, e2e_us, dev), 3), "unit": "us",
                      "h2d_bytes_per_step": NRANKS * COUNT * 2, "d2h_bytes_per_step": NRANKS * COUNT * 2,
                      "api": "llar_allreduce_host: pinned, registered host [8][8192] bf16 in, out; one AllReduce per call"}
    res["config"] = config
    if per_config is not None:
        res["per_config"] = per_config
        res["per_config_roofline"] = per_config_roofline(per_config, sol_us, hbm_peak, l2_us, write_us)
    return res


# ------------------------------------------------------- CPU oracle timing
def time_oracle(seconds, count=COUNT, nranks=NRANKS, dtype=DTYPE):
    """Oracle AllReduces of one workload for ~`seconds` (at least one) on one core."""
    from oracle import allreduce as orc
    from tp_allreduce_persistent_b300 import inputs
    xb = inputs.bits_of(inputs.normal(nranks, count, dtype, seed=1, scale=0.02))
    n = 0
    t0 = time.perf_counter()
    while True:
        orc.allreduce(xb, dtype)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return el * 1e6 / n, n


# the configurations' shapes for the CPU baseline: (ranks, dtype, elements per rank)
ORACLE_CONFIGS = {
    "C1_2ranks_128B_fp32": (2, "fp32", 32),
    "C2_4ranks_16KiB_bf16": (4, "bf16", 8192),
    "C3_8ranks_16KiB_bf16": (8, "bf16", 8192),
    "C3_8ranks_1MiB_bf16": (8, "bf16", 1 << 19),
    "C4_8ranks_64KiB_fp16": (8, "fp16", 32768),
    "C5_8ranks_128KiB_bf16": (8, "bf16", 65536),
    "bandwidth_8ranks_64MiB_bf16": (8, "bf16", 32 << 20),
}


def time_oracle_configs(seconds=0.5):
    """The single-core oracle on every configuration's shape (one AllReduce;
    a chain's steps are such AllReduces): us per AllReduce, and GB/s of
    algorithmic bytes (2 N S) for the bandwidth shape."""
    out = {}
    for name, (n, dtype, count) in ORACLE_CONFIGS.items():
        us, reps = time_oracle(seconds, count, n, dtype)
        row = {"us": round(us, 2), "allreduces": reps}
        if name.startswith("bandwidth"):
            row["GB/s"] = round(2 * n * count * 2 / (us * 1e-6) / 1e9, 3)
        out[name] = row
    return out


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


_START = None  # a worker process's start barrier


def _oracle_worker_init(barrier):
    global _START
    _START = barrier


def _oracle_slice_worker(job):
    """One worker process of the all-core CPU baseline: the oracle's
    AllReduce on one element slice, repeated for `seconds` once every
    worker is ready; returns (AllReduces done, seconds taken, the slice's
    result)."""
    xs, seconds = job
    from oracle import allreduce as orc
    y = orc.allreduce(xs, DTYPE)
    _START.wait(timeout=300)  # a worker that never arrives breaks the barrier: an error, not a hang
    n, t0 = 0, time.perf_counter()
    while True:
        y = orc.allreduce(xs, DTYPE)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return n, el, y


def time_oracle_all_cores(seconds, count=COUNT, nranks=NRANKS, parts=None):
    """The same AllReduces, element-partitioned over every host core the
    process may use: one spawned worker process per slice, all starting
    together at a barrier (threads would take turns on the interpreter
    lock, which numpy holds between its small calls). The arithmetic per
    element is the oracle's, so the joined slices are its bits. An
    AllReduce is done when every slice is, so its time is the slowest
    worker's. Returns (us per AllReduce, AllReduces of the slowest worker,
    processes, inputs, joined outputs)."""
    import multiprocessing
    from concurrent.futures import ProcessPoolExecutor

    import numpy as np

    from tp_allreduce_persistent_b300 import inputs
    parts = parts or host_cores()
    xb = inputs.bits_of(inputs.normal(nranks, count, DTYPE, seed=1, scale=0.02))
    bounds = [count * i // parts for i in range(parts + 1)]
    ctx = multiprocessing.get_context("spawn")
    # each worker blocks at the barrier with its task, so every task lands on
    # its own worker; a worker that fails to start raises (BrokenProcessPool)
    with ProcessPoolExecutor(parts, mp_context=ctx, initializer=_oracle_worker_init,
                             initargs=(ctx.Barrier(parts),)) as pool:
        jobs = [(xb[:, bounds[i]:bounds[i + 1]].copy(), seconds) for i in range(parts)]
        res = list(pool.map(_oracle_slice_worker, jobs))
    us = max(el / n for n, el, _ in res) * 1e6
    out = np.concatenate([y for _, _, y in res], axis=1)
    return us, min(n for n, _, _ in res), parts, xb, out


def run_reference(args, world, rank):
    if rank != 0:
        return None
    ref_seconds = 0.5
    for _ in range(args.warmup):
        time_oracle(0.05)
    per = []
    for _ in range(args.steps):
        us, _ = time_oracle(ref_seconds)
        per.append(us)
    v = statistics.mean(per)
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(v, 3), "unit": "us",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ref_seconds * 1e3, 1), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32-accumulate over bf16",
        "data": "synthetic: N(0,1)*0.02, seeded",
        "config": {"workload": "8 virtual ranks x 16 KiB bf16 (8192 elements) AllReduce",
                   "nranks": NRANKS, "count": COUNT},
        "cpu_baseline": {"value": round(v, 3), "unit": "us", "cores": 1, "kind": "oracle",
                         "sample": f"{ref_seconds} s of back-to-back oracle AllReduces per step"},
        "e2e": {"value": round(v, 3), "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world, rank, local, pg = dist_setup(args)
    if args.impl == "reference":
        res = run_reference(args, world, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    res = run_ours(args, world, rank, local, pg)
    if rank == 0 and res is not None:  # the llbuffer and config legs print their own line
        if not args.no_cpu_baseline and world == 1:  # the CPU baseline is a single-GPU figure
            us, n = time_oracle(10.0)
            us_all, n_all, cores, _, _ = time_oracle_all_cores(5.0)
            res["cpu_baseline"] = {"value": round(us, 3), "unit": "us", "cores": 1, "kind": "oracle",
                                   "sample": f"{n} oracle AllReduces of the latency workload in ~10 s "
                                             "on one host core (numpy, single-threaded)",
                                   "nproc": os.cpu_count(),
                                   "all_cores": {"value": round(us_all, 3), "unit": "us", "cores": cores,
                                                 "sample": f"{n_all} oracle AllReduces of the latency "
                                                           f"workload in ~5 s, elements split over "
                                                           f"{cores} worker processes running at "
                                                           "once (same bits)"},
                                   "per_config": time_oracle_configs()}
        print(json.dumps(res), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
