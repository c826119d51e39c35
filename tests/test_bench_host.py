"""Host-side logic of bench.py that needs no GPU.

* The replica aggregation (barrier, max over ranks, whole-job throughput) on
  two gloo ranks on the CPU, as torchrun would launch them.
* The clock-sample summary (throttle reasons, window selection), the
  parser of nvidia-smi's sample lines, and the sampler's pipe reader against
  a stand-in nvidia-smi that prints samples until it is interrupted.
"""
import os
import socket
import stat
import time

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    secs = 1.0 + rank  # rank 1 is the slow one
    slowest = bench.reduce_max(secs, w)
    out[rank] = (slowest, bench.throughput(32, 100, slowest, w))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        slowest, value = out[r]
        assert slowest == 2.0                      # max over ranks
        assert value == pytest.approx(32 * 100 * 2 / 2.0)  # rows of all ranks / slowest time


def test_single_process_is_identity():
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.throughput(32, 10, 2.0, 1) == 160.0


def test_clock_summary_window_and_reasons():
    c = bench.ClockSampler(0)
    c.samples = [
        dict(t=1.0, sm=2070.0, sm_max=2070.0, reasons="0x0", hw="Not Active", hwt="Not Active",
             swt="Not Active", pcap="Not Active"),
        dict(t=2.0, sm=1980.0, sm_max=2070.0, reasons="0x4", hw="Not Active", hwt="Not Active",
             swt="Not Active", pcap="Active"),
        dict(t=9.0, sm=900.0, sm_max=2070.0, reasons="0x8", hw="Active", hwt="Not Active",
             swt="Not Active", pcap="Not Active"),
    ]
    s = c.summary(0.5, 2.5)
    assert s["window"] == "timed" and s["samples"] == 2
    assert s["sm_mhz"] == 2025.0 and s["reasons"] == ["sw_power_cap"]
    s = c.summary(3.0, 4.0)  # nothing inside: falls back to the whole run
    assert s["window"] == "run" and "hw_slowdown" in s["reasons"]


def test_algorithmic_bytes():
    # one row of 7168: 14336 bytes read, 3584 + 448 written (+ 4 for gs)
    assert bench.quantize_bytes(1, 7168) == 14336 + 3584 + 448 + 4
    # router decode T=32: A and B codes + scales, gs, bias, top-8 outputs
    assert bench.gemm_bytes(32, 256, 7168, 8) == (32 + 256) * 4032 + 8 + 1024 + 32 * 8 * 12


def test_rotating_sets_exceed_twice_l2():
    # a rotation reads more than 2.2x L2 per pass, with at least two copies;
    # inputs too small for a bounded number of copies fall back to a flush
    for b in (1 << 20, 29 * (1 << 20), 235 * (1 << 20), 150 * 1024):
        n = bench.rotating_sets(b)
        assert n is not None and n >= 2 and n * b >= bench.ROTATE_BYTES
        assert (n - 1) * b < bench.ROTATE_BYTES or n == 2
    assert bench.rotating_sets(14 * 1024) is None  # 14 KB would need ~20k copies
    assert bench.rotating_sets(bench.ROTATE_BYTES + 1) == 2


SMI_LINE = ("2026/12/02 16:20:01.250, 0, 1965, 2070, 1012.55, 0x0000000000000004, Not Active, Not Active, "
            "Not Active, Active")


def test_smi_line_parser():
    s = bench.parse_smi_line(SMI_LINE)
    assert s["sm"] == 1965.0 and s["sm_max"] == 2070.0 and s["pcap"] == "Active" and s["hw"] == "Not Active"
    assert s["t"] == time.mktime(time.strptime("2026/12/02 16:20:01", "%Y/%m/%d %H:%M:%S")) + 0.25
    assert bench.parse_smi_line("timestamp, index, clocks.current.sm [MHz]") is None  # a header
    assert bench.parse_smi_line("") is None
    assert bench.parse_smi_line("2026/12/02 16:20:01.250, 0, [N/A], 2070, 1, 0x0, a, b, c, d") is None


def test_clock_sampler_reads_samples_until_interrupted(tmp_path, monkeypatch):
    # a stand-in nvidia-smi on PATH: one sample line (current time) every 10 ms, forever
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/bash\nwhile true; do\n"
                    "  printf '%s, 0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active\\n' "
                    "\"$(date '+%Y/%m/%d %H:%M:%S.%N' | cut -c1-23)\"\n  sleep 0.01\ndone\n")
    fake.chmod(fake.stat().st_mode | stat.S_IEXEC)
    monkeypatch.setenv("PATH", f"{tmp_path}:{os.environ['PATH']}")
    with bench.ClockSampler(0, period_ms=10) as clk:
        t0 = time.time()
        time.sleep(0.6)
        t1 = time.time()
    assert len(clk.samples) >= 10
    s = clk.summary(t0 - 1.0, t1 + 1.0)
    assert s["window"] == "timed" and s["sm_mhz"] == 2070.0 and s["reasons"] == []


def test_traffic_record_needs_the_same_source(tmp_path, monkeypatch):
    # a recorded DRAM figure is reported only while the kernel source hashes to the recorded sha
    import hashlib
    import json
    src_dir = tmp_path / "quantize_block_scaled_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = src_dir / "k.cu"
    src.write_text("// kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    rec = {"records": [{"source": "k.cu", "sha": sha, "workload": "w", "dram_bytes_per_launch": 1234}]}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("k.cu", "w") == 1234
    assert bench.load_traffic("k.cu", "other") is None
    src.write_text("// kernel v2\n")  # the kernel changed since the counters were taken
    assert bench.load_traffic("k.cu", "w") is None
