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
per AllReduce is larger than L2. Each launch is timed with CUDA events on
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
FLUSH_BYTES = 256 << 20    # > 126 MB L2
FALLBACK_HBM_GBS = 6400.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--protocol", default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


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


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tp_allreduce_persistent_b300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
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
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
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
def run_ours(args, world, rank, local, pg):
    import torch
    from tp_allreduce_persistent_b300 import inputs, llar

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    llar.llar_init(NRANKS, DTYPE, BW_COUNT * 2)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    # ---- speed of light on this GPU (2 x L2 round trip + one write)
    l2_us, write_us, sol_us = llar.llar_sol_probe()

    # ---- latency leg: 16 KiB bf16 x 8 ranks, ITERS back to back per launch
    x = inputs.normal(NRANKS, COUNT, DTYPE, seed=1, scale=0.02)
    ins = [x[r].to(dev) for r in range(NRANKS)]
    outs = [torch.empty_like(t) for t in ins]
    proto = args.protocol
    for _ in range(args.warmup):
        llar.llar_allreduce_iters(ins, outs, COUNT, proto, ITERS, 0, 0, 0.0)
    torch.cuda.synchronize()
    used_proto, g, t, _ = llar.llar_last_launch()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier(pg, local)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(k & 0xFF)  # evict L2 between timed launches (outside the events)
        ev[k][0].record(stream)
        llar.llar_allreduce_iters(ins, outs, COUNT, proto, ITERS, 0, 0, 0.0)
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    barrier(pg, local)
    wall_lat = time.perf_counter() - wall0
    lat_ms = [a.elapsed_time(b) for a, b in ev]
    code = llar.llar_get_status()[0]
    if code != llar.OK:
        raise RuntimeError(f"device status {code} during the latency leg")
    step_ms = sum(lat_ms) / len(lat_ms)
    us_per_ar = step_ms * 1e3 / ITERS

    # ---- bandwidth leg: 64 MiB bf16 x 8 ranks, fixed-order two-shot
    bw_ins = [torch.randn(BW_COUNT, device=dev, generator=torch.Generator(device=dev).manual_seed(5 + r))
              .to(torch.bfloat16) for r in range(NRANKS)]
    bw_outs = [torch.empty_like(a) for a in bw_ins]
    for _ in range(args.warmup):
        llar.llar_allreduce(bw_ins, bw_outs, BW_COUNT, "fixed_twoshot")
    torch.cuda.synchronize()
    bw_shape = llar.llar_last_launch()
    bev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps * BW_REPS)]
    barrier(pg, local)
    torch.cuda.synchronize()
    i = 0
    for k in range(args.steps):
        for _ in range(BW_REPS):
            bev[i][0].record(stream)
            llar.llar_allreduce(bw_ins, bw_outs, BW_COUNT, "fixed_twoshot")
            bev[i][1].record(stream)
            i += 1
    torch.cuda.synchronize()
    barrier(pg, local)
    clk = clocks.stop()
    bw_ms = [a.elapsed_time(b) for a, b in bev]
    bw_launch_s = statistics.mean(bw_ms) * 1e-3
    alg_bytes = 2 * NRANKS * BW_COUNT * 2
    gbs = alg_bytes / bw_launch_s / 1e9

    # ---- end to end: host buffers through llar_allreduce_host
    hx = x.contiguous().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    for _ in range(args.warmup):
        llar.llar_allreduce_host(hx, hy, COUNT, proto)
    torch.cuda.synchronize()
    e2e_steps = max(3, args.steps // 5)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg, local)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(e2e_steps * E2E_CALLS):
        llar.llar_allreduce_host(hx, hy, COUNT, proto)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_us = e0.elapsed_time(e1) * 1e3 / (e2e_steps * E2E_CALLS)
    llar.llar_destroy()

    # ---- aggregate over ranks (independent replicas)
    us_per_ar = max_over_ranks(pg, us_per_ar, dev)
    gbs_min = -max_over_ranks(pg, -gbs, dev)
    e2e_us = max_over_ranks(pg, e2e_us, dev)
    total_ars = sum_over_ranks(pg, ITERS * args.steps, dev)
    peaks, peak_src = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    bw_workload = "8 ranks x 64 MiB bf16, fixed-order two-shot"
    traffic = recorded_traffic("k_fixed_twoshot<bf16>", bw_workload)
    result = {
        "metric": METRIC,
        "value": round(us_per_ar, 4),
        "unit": "us",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32-accumulate over bf16",
        "data": "synthetic: N(0,1)*0.02 activations (latency leg), N(0,1) (bandwidth leg), seeded",
        "config": {
            "workload": "8 virtual ranks x 16 KiB bf16 (8192 elements) AllReduce, "
                        f"{ITERS} back-to-back per persistent launch",
            "nranks": NRANKS, "count": COUNT, "iters_per_launch": ITERS,
            "protocol": used_proto, "ctas_per_rank": g, "threads_per_cta": t,
            "l2": "flushed between timed launches (256 MiB write outside the events)",
            "bandwidth_workload": bw_workload + "; inputs+outputs 1 GiB > L2",
            "replicas": "independent per GPU" if world > 1 else "single GPU",
        },
        "bandwidth": {
            "value": round(gbs_min, 1), "unit": "GB/s",
            "us_per_allreduce": round(bw_launch_s * 1e6, 2),
            "algorithmic_bytes": alg_bytes,
            "algbw_gbs": round(BW_COUNT * 2 / bw_launch_s / 1e9, 1),
            "busbw_gbs": round(BW_COUNT * 2 / bw_launch_s / 1e9 * 2 * (NRANKS - 1) / NRANKS, 1),
            "ctas_per_rank": bw_shape[1], "threads_per_cta": bw_shape[2],
        },
        "roofline": {
            "kernel": "k_fixed_twoshot<bf16>", "bound": "hbm",
            "achieved": round(gbs_min, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(gbs_min / hbm_peak, 4), "traffic": traffic,
            "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)",
            "frac_of_nominal_8TBps": round(gbs_min / 8000.0, 4),
        },
        "latency_roofline": {
            "kernel": f"k_{used_proto}<bf16>", "bound": "latency (L2 round trips)",
            "achieved_us": round(us_per_ar, 4), "sol_us": round(sol_us, 4),
            "l2_round_trip_us": round(l2_us, 4), "write_us": round(write_us, 4),
            "frac": round(sol_us / us_per_ar, 4),
            "within_2x_sol": bool(us_per_ar <= 2 * sol_us),
            "definition": "SoL = 2 x L2 round trip + one remote write, measured in this run",
        },
        "e2e": {"value": round(e2e_us, 3), "unit": "us",
                "h2d_bytes_per_step": NRANKS * COUNT * 2, "d2h_bytes_per_step": NRANKS * COUNT * 2,
                "api": "llar_allreduce_host (pinned host [8][8192] bf16 in and out, one AllReduce per call)"},
        "gpu_launches": args.steps,
        "gpu_launches_bandwidth_leg": args.steps * BW_REPS,
        "total_allreduces": int(total_ars),
        "wall_s_latency_leg": round(wall_lat, 3),
        "clocks": clk,
    }
    return result


# ------------------------------------------------------- CPU oracle timing
def time_oracle(seconds, count=COUNT, nranks=NRANKS):
    """Oracle AllReduces of the latency workload for ~`seconds` on one core."""
    from oracle import allreduce as orc
    from tp_allreduce_persistent_b300 import inputs
    xb = inputs.bits_of(inputs.normal(nranks, count, DTYPE, seed=1, scale=0.02))
    n = 0
    t0 = time.perf_counter()
    while True:
        orc.allreduce(xb, DTYPE)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return el * 1e6 / n, n


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
    if rank == 0:
        if not args.no_cpu_baseline:
            us, n = time_oracle(10.0)
            res["cpu_baseline"] = {"value": round(us, 3), "unit": "us", "cores": 1, "kind": "oracle",
                                   "sample": f"{n} oracle AllReduces of the latency workload in ~10 s "
                                             "on one host core (numpy, single-threaded)"}
        print(json.dumps(res), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
