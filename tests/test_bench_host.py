"""Host-side logic of bench.py on CPU: cross-rank aggregation over a
world-size-2 gloo group, the clock-record parser, and the reference arm's
JSON line. Nothing here touches a GPU."""

import os
import socket
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench as b
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q.put((rank, b.max_over_ranks(dist, 10.0 + rank), b.sum_over_ranks(dist, 1000.0),
           -b.max_over_ranks(dist, -(5.0 + rank))))
    b.barrier(dist)
    dist.destroy_process_group()


def test_aggregation_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # slowest rank's latency, units summed over ranks, smallest bandwidth
    assert res == [(0, 11.0, 2000.0, 5.0), (1, 11.0, 2000.0, 5.0)]


def test_clock_record_parser():
    lines = ["0, 1900, 2032, 700.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
             "0, 1920, 2032, 800.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "0, 1880, 2032, 650.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "garbage"]
    rec = bench.ClockSampler.parse(lines)
    assert rec["sm_mhz"] == 1900 and rec["sm_max_mhz"] == 2032
    assert rec["reasons"] == ["sw_power_cap"] and rec["samples"] == 3


def test_reference_arm_line(monkeypatch):
    monkeypatch.setattr(bench, "time_oracle", lambda seconds, **k: (123.0, 10))
    args = types.SimpleNamespace(steps=2, warmup=1)
    line = bench.run_reference(args, world=1, rank=0)
    assert line["impl"] == "reference" and line["value"] == 123.0 and line["unit"] == "us"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert bench.run_reference(args, world=2, rank=1) is None


def test_oracle_timing_runs():
    us, n = bench.time_oracle(0.05, count=256, nranks=4)
    assert us > 0 and n >= 1


def test_config_cases_parse_and_match_the_table_rows():
    # `--leg config --case NAME` reruns one row of the per-configuration table
    for name in list(bench.CONFIG_CASES) + list(bench.FUSED_CASES):
        assert bench.parse(["--leg", "config", "--case", name]).case == name
    assert bench.CONFIG_CASES["C4_sentinel"] == (8, "fp16", 32768, "sentinel", 1000, 0.0, 8192)
    assert bench.CONFIG_CASES["C3_ll128_1MiB"][:4] == (8, "bf16", 1 << 19, "ll128")
    with pytest.raises(SystemExit):
        bench.parse(["--leg", "config", "--case", "no_such_row"])


def test_all_core_oracle_gives_the_same_bits():
    # the element-partitioned timing of the CPU baseline (worker processes)
    # computes exactly the single-threaded oracle's result, ragged splits too
    import numpy as np

    from oracle import allreduce as orc
    for parts in (1, 3, 7):
        us, n, used, xb, out = bench.time_oracle_all_cores(0.05, count=1003, nranks=8, parts=parts)
        assert us > 0 and n >= 1 and used == parts
        assert np.array_equal(out, orc.allreduce(xb, "bf16")), parts
    assert bench.time_oracle_all_cores(0.02, count=64, nranks=2)[2] == bench.host_cores()


def test_chunked_floor_reduces_to_the_speed_of_light():
    # one chunk: 2 x L2 round trip + one write, the pages' speed of light
    assert abs(bench.chunked_floor_us(1, 0.306, 0.792) - 1.404) < 1e-12
    # the chunked sentinel row gets its own floor beside the per-operation one
    per = {bench.C4_KEY: 8.0, "C1_2ranks_128B_fp32_us": {"ll": 0.5}}
    out = bench.per_config_roofline(per, 0.6, 6000.0, 0.15, 0.3)
    floor = 0.15 + 8 * (0.3 + 0.15)
    assert abs(out["C4_chunked_floor"]["floor_us"] - floor) < 1e-4
    assert abs(out["C4_chunked_floor"]["frac"] - floor / 8.0) < 1e-4
    assert out[bench.C4_KEY] == round(0.6 / 8.0, 4)
    assert "C4_chunked_floor" not in bench.per_config_roofline(per, 0.6, 6000.0)


def test_segment_bandwidth_rows_go_against_hbm():
    # the ReduceScatter / AllGather bandwidth row is a bandwidth row: GB/s
    # over the measured copy bandwidth, not the latency floor
    per = {bench.SEG_KEY: {"reduce_scatter": {"us": 94.0, "GB/s": 6000.0},
                           "all_gather": {"us": 103.0, "GB/s": 5400.0}}}
    out = bench.per_config_roofline(per, 0.6, 6000.0)
    assert out[bench.SEG_KEY] == {"reduce_scatter": 1.0, "all_gather": 0.9}


def test_oracle_config_timings_cover_every_shape():
    # every configuration shape gets a single-core oracle timing (tiny sample here)
    saved = dict(bench.ORACLE_CONFIGS)
    try:
        bench.ORACLE_CONFIGS.clear()
        bench.ORACLE_CONFIGS.update({"C1_2ranks_128B_fp32": (2, "fp32", 32),
                                     "bandwidth_8ranks_small_bf16": (8, "bf16", 4096)})
        out = bench.time_oracle_configs(0.01)
        assert set(out) == set(bench.ORACLE_CONFIGS)
        assert all(v["us"] > 0 and v["allreduces"] >= 1 for v in out.values())
        assert out["bandwidth_8ranks_small_bf16"]["GB/s"] > 0
    finally:
        bench.ORACLE_CONFIGS.clear()
        bench.ORACLE_CONFIGS.update(saved)
