"""Host-side logic of bench.py, on CPU: the cross-rank reduction of the multi-GPU
(replica) path with two gloo ranks, the clock-sample parser, the DRAM-traffic table
lookup and the reference arm (the CPU oracle) on a tiny workload."""

import json
import os
import socket
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks(float(10 * rank + 3), world)
    bench.barrier(world)
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as fh:
        fh.write(repr(got))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    vals = [float(open(tmp_path / f"r{r}.txt").read()) for r in range(2)]
    assert vals == [13.0, 13.0]


def test_single_rank_reduction_is_identity():
    assert bench.max_over_ranks(4.5, 1) == 4.5


def test_clock_parser_keeps_samples_inside_the_window():
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.proc = object()
    t0 = time.time()
    stamp = lambda dt: time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(t0 + dt)) + \
        ".%03d" % int(((t0 + dt) % 1) * 1000)
    cs.lines = [
        f"{stamp(-5)}, 0, 900, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        f"{stamp(0.1)}, 0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Active",
        f"{stamp(0.2)}, 0, 1980, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Active",
    ]
    s = cs.summary(t0, t0 + 0.3)
    assert s["samples_in_timed_region"] == 2
    assert s["sm_mhz"] == pytest.approx(2025.0)
    assert s["reasons"] == ["sw_power_cap"]


def test_traffic_table_lookup():
    v = bench.recorded_traffic("gevm", (1, 8192, 8192), "gevm")
    # present while the kernel source is unchanged since the capture, else None; the
    # one-row product reads B once: traffic within 2 % of its 268.5 MB
    assert v is None or abs(v - 268500992) < 0.02 * 268500992
    assert bench.recorded_traffic("gevm", (2, 3, 4), "gevm") is None


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--shape", "64,96,80", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["cpu_model"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    # the reference arm reports the same workload config as the GPU arm
    assert d["config"] == bench.workload_config((64, 96, 80), "fp32", 1)


def test_cpu_model_string():
    m = bench.cpu_model()
    assert isinstance(m, str) and m and m != "unknown"


def test_vs_baseline_only_for_the_pages_workload():
    r, basis = bench.vs_pages("fp32", bench.HEADLINE, 81.681144)
    assert r == pytest.approx(2.0) and "RTX 4090" in basis
    r, _ = bench.vs_pages("tf32", bench.HEADLINE, 32.528826)
    assert r == pytest.approx(1.0)
    assert bench.vs_pages("fp32", (512, 512, 512), 1.0) == (None, None)


def test_rooflines_use_each_kernels_rate_per_clock():
    """The roofline of each tensor-core kernel uses its own rate: 4096 TF32 flop per clock
    per SM for the TF32 kernels, 8192 for the FP16 one, with three products per term for
    3xTF32 and 3xFP16; the device-clock peak follows the kernel's kind."""
    import dense_fp32_gemm_sgemm_gb300 as sg
    peaks = {"bf16_tflops": 1969.0, "hbm_gbs": 6785.9, "sm_max_mhz": 2070.0}
    M, N, K = 8192, 6144, 4096
    flops = 2.0 * M * N * K
    r3 = bench.roofline_for(sg, sg.KERNEL_TC_3XTF32, M, N, K, 1.0, peaks, 152, 2000.0)
    r16 = bench.roofline_for(sg, sg.KERNEL_TC_3XFP16, M, N, K, 1.0, peaks, 152, 2000.0)
    r1 = bench.roofline_for(sg, sg.KERNEL_TC_1XTF32, M, N, K, 1.0, peaks, 152, 2000.0)
    assert r3["tensor_flop_per_launch"] == r16["tensor_flop_per_launch"] == 3 * flops
    assert r1["tensor_flop_per_launch"] == flops
    assert r16["clock_peak"] == pytest.approx(2 * r3["clock_peak"])
    assert r3["clock_peak"] == pytest.approx(152 * 4096 * 2000e6 / 1e12)
    assert r16["peak"] == pytest.approx(1969.0) and r3["peak"] == pytest.approx(1969.0 / 2)
    for roof, kind, per_clk in ((r3, "tc", 4096), (r16, "tc16", 8192)):
        bench.add_device_clock_peak(roof, 1800.0, 152, kind)
        assert roof["device_clock_peak"] == pytest.approx(152 * per_clk * 1800e6 / 1e12)
    simt = {"achieved": 60.0}
    bench.add_device_clock_peak(simt, 2000.0, 152, "simt")
    assert simt["device_clock_peak"] == pytest.approx(152 * 256 * 2000e6 / 1e12)
