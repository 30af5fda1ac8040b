#!/usr/bin/env python3
"""Benchmark of the FP32 matrix product C = A . B on GB300.

Headline workload: M=8192, N=6144, K=4096 (A 192 MiB, B 96 MiB, C 128 MiB, 2MNK =
412,316,860,416 flop), row-major float32, A and B uniform on [-1, 1) from seed 2 (the
performance shape of "LeetGPU | 02_Matrix_Multiplication", section "Constraints").
One step is one FP32-accurate solve_ex call through the C ABI. Inputs (416 MiB with C)
are larger than the 129 MB L2, so no flush is needed between steps.

Prints one JSON line (rank 0). `value` is TFLOP/s over all ranks with inputs resident
in HBM; `e2e` repeats the measurement through solve_host (host arrays in page-locked
memory, uploads and the download of C inside the timed region); `roofline` describes
the dominant kernel, timed with CUDA events around its own launch inside the timed
steps; `cpu_baseline` times the CPU oracle on a bounded sample of the same product;
`variants` times the other paths (1xTF32, the CUDA-core kernel, the streaming shapes);
`timing_protocols` repeats the step under the pages' own protocols (five warm-ups and ten
individually timed calls; fifty calls back to back; ten calls with L2 flushed by a 512 MiB
write before each); `clocks` carries the nvidia-smi samples and the SM clock the dominant
kernel recorded for itself.

`--impl reference` times the CPU oracle itself on bounded samples of the same workload
(it is the only reference implementation this project has).

Multi-GPU: the product does not shard here; with torchrun each rank runs an independent
replica on its own GPU and `value` sums their work over the slowest rank's time.
"""

from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = (8192, 6144, 4096)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
# TF32 tensor rate per clock relative to BF16: 1:2 (the per-clock rates are 4096 and
# 8192 flop/clk/SM; this library's pair-MMA probes, run at the same clock, measured
# 0.5006 for the TF32 / FP16 ratio).
TF32_PER_BF16 = 0.5
# tcgen05 kind::tf32 rate per SM per clock, as ncu reports it
# (sm__ops_path_tensor_op_utchmma_src_tf32_dst_fp32_sparsity_off peak_sustained).
TF32_FLOP_PER_CLK_SM = 4096


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--mode", default="fp32",
                   help="fp32 (default, FP32-accurate) | tf32 | simt | 3xtf32 | 3xfp16 "
                        "(scaled FP16 pieces: an explicit mode with a weaker bound, not FP32)")
    p.add_argument("--shape", default=None, help="M,N,K (default 8192,6144,4096)")
    p.add_argument("--no-variants", action="store_true", help="skip the other paths")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--no-e2e", action="store_true", help="skip the host round trip")
    p.add_argument("--no-probes", action="store_true", help="skip the peak-rate probes")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target wall time of the CPU oracle sample")
    return p.parse_args(argv)


# ----------------------------------------------------------------------------- peaks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {k: float(d.get(k, FALLBACK_PEAKS[k])) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def fp32_simt_peak_tflops(sm_count: int, mhz: float) -> float:
    # 128 FP32 lanes per SM, one FMA (2 flop) per lane per clock
    return sm_count * 128 * 2 * mhz * 1e6 / 1e12


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, timeout=5.0):
        t0 = time.time()
        while self.proc and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.02)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        if not self.proc:
            return None
        rows = []
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), f[4], f[6:10]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if t0 - 0.06 <= r[0] <= t1 + 0.06]
        used = inside if inside else sorted(rows, key=lambda r: abs(r[0] - (t0 + t1) / 2))[:2]
        reasons = sorted({name for r in used for name, v in zip(self.REASONS, r[4])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in used),
                "sm_max_mhz": max(r[2] for r in used),
                "reasons": reasons, "samples": len(used),
                "samples_in_timed_region": len(inside)}


# ----------------------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def kernel_source_hash(kind: str) -> str:
    files = {"simt": ["simt_gemm.cu"], "gevm": ["skinny.cu"], "gemv": ["skinny.cu"],
             "smalln": ["skinny.cu"], "tc": ["tc_gemm.cu"], "tc16": ["tc_gemm.cu"]}.get(kind, [])
    h = hashlib.sha256()
    for f in files:
        p = os.path.join(ROOT, "dense_fp32_gemm_sgemm_gb300", "csrc", f)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, shape, kind: str):
    """DRAM bytes per launch from the committed ncu summary (profiles/dram_traffic.md),
    only while the kernel's source is unchanged since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    try:
        lines = open(path, encoding="utf-8").read().splitlines()
    except OSError:
        return None
    key = f"{kernel}:{shape[0]}x{shape[1]}x{shape[2]}"
    for line in lines:
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 7 and cells[0] == key:
            if cells[6] != kernel_source_hash(kind):
                return None
            try:
                return int(cells[4])
            except ValueError:
                return None
    return None


# ----------------------------------------------------------------------------- GPU timing
class Runner:
    def __init__(self, torch, sg, M, N, K, seed, dist, device):
        from dense_fp32_gemm_sgemm_gb300.inputs import make_inputs
        self.torch, self.sg = torch, sg
        self.M, self.N, self.K = M, N, K
        A, B = make_inputs(M, N, K, seed, dist)
        self.hA, self.hB = A, B
        self.dA = torch.from_numpy(A).to(device)
        self.dB = torch.from_numpy(B).to(device)
        self.dC = torch.empty((M, K), dtype=torch.float32, device=device)
        self.stream = torch.cuda.current_stream()
        self.handle = int(self.stream.cuda_stream)
        self._args = None
        self._solve = None

    def call(self, mode):
        # the C ABI call with its arguments marshalled once (the buffers never move)
        if self._args is None:
            self._solve = self.sg.lib().solve_ex
            self._args = (self.dA.data_ptr(), self.dB.data_ptr(), self.dC.data_ptr(),
                          self.M, self.N, self.K)
        rc = self._solve(*self._args, mode, self.handle)
        if rc != 0:
            raise RuntimeError(f"solve_ex failed: {self.sg.lib().sgemm_status_string(rc)}")

    def timed(self, mode, steps, warmup, world=1, sampler=None):
        torch = self.torch
        L = self.sg.lib()
        for _ in range(warmup):
            self.call(mode)
        # the kernel's own events bracket every GEMM launch, or every fourth one for
        # products of a few microseconds, whose steps the two event records per call
        # would otherwise lengthen by a fifth
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        self.call(mode)
        e1.record(self.stream)
        torch.cuda.synchronize()
        every = 4 if e0.elapsed_time(e1) < 0.1 and steps >= 8 else 1
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range((steps + every - 1) // every)]
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        for a, b in ev:  # torch creates each CUDA event on its first record
            a.record(self.stream)
            b.record(self.stream)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        launches0 = self.sg.launch_count()
        t0 = time.time()
        start.record(self.stream)
        set_events = L.sgemm_set_kernel_events
        handles = [(a.cuda_event, b.cuda_event) for a, b in ev]
        for i in range(steps):
            if i % every == 0:
                set_events(*handles[i // every])
            self.call(mode)
        end.record(self.stream)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world)
        torch.cuda.synchronize()
        launches = self.sg.launch_count() - launches0
        total_ms = start.elapsed_time(end)
        kern = [a.elapsed_time(b) for a, b in ev]
        return {"ms_per_step": total_ms / steps, "kernel_ms": statistics.mean(kern),
                "kernel_ms_min": min(kern), "kernel_ms_max": max(kern),
                "kernel_ms_median": statistics.median(kern), "kernel_events_every": every,
                "launches": launches, "t0": t0, "t1": t1}

    def protocols(self, mode, flops, clock=None):
        """The pages' other timing protocols on the same operands: five warm-up calls,
        then ten calls each between their own events (mean, min, max, median); fifty calls
        back to back between two events (their mean); and ten calls with L2 cold, a 512 MiB
        scratch buffer written before each (outside its events). `clock`, if given, reads
        the SM clock the last call's kernel recorded, after each protocol."""
        torch = self.torch

        def ev():
            return torch.cuda.Event(enable_timing=True)

        def one_each(before=None):
            pairs = [(ev(), ev()) for _ in range(10)]
            for i, (a, b) in enumerate(pairs):
                if before:
                    before(i)
                a.record(self.stream)
                self.call(mode)
                b.record(self.stream)
            torch.cuda.synchronize()
            t = [a.elapsed_time(b) for a, b in pairs]
            return {"runs": 10, "mean_ms": statistics.mean(t), "min_ms": min(t),
                    "max_ms": max(t), "median_ms": statistics.median(t),
                    "tflops_at_mean": flops / (statistics.mean(t) * 1e-3) / 1e12}

        for _ in range(5):
            self.call(mode)
        p1 = one_each()
        if clock:
            p1["device_sm_mhz"] = clock()
        s, e = ev(), ev()
        s.record(self.stream)
        for _ in range(50):
            self.call(mode)
        e.record(self.stream)
        torch.cuda.synchronize()
        b2b = s.elapsed_time(e) / 50
        b2b_mhz = clock() if clock else None
        scratch = torch.empty(128 << 20, dtype=torch.float32, device=self.dA.device)
        cold = one_each(lambda i: scratch.fill_(float(i)))
        cold["scratch_mib"] = 512
        if clock:
            cold["device_sm_mhz"] = clock()
        del scratch
        return {"five_warmup_ten_timed": p1,
                "fifty_back_to_back": {"mean_ms": b2b, "tflops": flops / (b2b * 1e-3) / 1e12,
                                       "device_sm_mhz": b2b_mhz},
                "l2_cold_ten_timed": cold}

    def e2e(self, mode, steps, warmup):
        """solve_host round trips from page-locked host buffers; seconds per step."""
        torch = self.torch
        hA = torch.from_numpy(self.hA).pin_memory()
        hB = torch.from_numpy(self.hB).pin_memory()
        hC = torch.empty((self.M, self.K), dtype=torch.float32).pin_memory()
        L = self.sg.lib()

        def once():
            rc = L.solve_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), self.M, self.N,
                              self.K, mode, self.handle)
            if rc != 0:
                raise RuntimeError(f"solve_host failed: {L.sgemm_status_string(rc)}")

        for _ in range(warmup):
            once()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            once()
        torch.cuda.synchronize()
        dt = (time.perf_counter() - t0) / steps
        return dt, (self.hA.nbytes + self.hB.nbytes), self.M * self.K * 4


# The pages' own figures for this exact workload, on another GPU (context, not a target):
# "LeetGPU | 02_Matrix_Multiplication", section "Test Result", "NVIDIA GeForce RTX 4090",
# 8192 x 6144 x 4096: the default kernel (FP32, 10.096 ms) and the WMMA kernel (TF32,
# 12.675 ms), in TFLOP/s.
PAGES_HEADLINE_TFLOPS = {
    "fp32": (40.840572, "pages' default FP32 kernel on an RTX 4090, 40.84 TFLOP/s"),
    "tf32": (32.528826, "pages' WMMA TF32 kernel on an RTX 4090, 32.53 TFLOP/s"),
}


def vs_pages(mode_name, shape, value):
    """value / the pages' figure for the same workload and arithmetic (None elsewhere)."""
    if shape != HEADLINE:
        return None, None
    key = "tf32" if mode_name.lower() == "tf32" else "fp32"
    ref, basis = PAGES_HEADLINE_TFLOPS[key]
    return value / ref, basis


KERNEL_OF_PLAN = {1: ("simt_gemm", "simt"), 2: ("gevm", "gevm"), 3: ("gemv", "gemv"),
                  4: ("tc_gemm_1xtf32", "tc"), 5: ("tc_gemm_3xtf32", "tc"),
                  7: ("tc_gemm_3xfp16", "tc16"),
                  6: ("smalln", "smalln")}


def roofline_for(sg, kernel_id, M, N, K, kernel_ms, peaks, sm_count, clock_mhz=None):
    """Roofline of the dominant kernel: algorithmic work per launch / event time."""
    name, kind = KERNEL_OF_PLAN[kernel_id]
    t = kernel_ms * 1e-3
    flops = 2.0 * M * N * K
    if kind == "simt":
        peak = fp32_simt_peak_tflops(sm_count, peaks["sm_max_mhz"])
        ach = flops / t / 1e12
        return {"bound": "alu", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "kernel": name,
                "peak_basis": f"{sm_count} SMs x 128 FP32 lanes x 2 flop x "
                              f"{peaks['sm_max_mhz']:.0f} MHz"}
    if kind in ("gevm", "gemv", "smalln"):
        byts = 4.0 * (M * N + N * K + M * K)
        ach = byts / t / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "kernel": name,
                "peak_basis": "MEASURED_PEAKS hbm_gbs"}
    passes = 3 if kernel_id in (5, 7) else 1
    f16 = kind == "tc16"
    # the 16-bit tensor rate per clock is the BF16 one; TF32's is the nominal ratio of it
    ratio = 1.0 if f16 else TF32_PER_BF16
    per_clk = (2 if f16 else 1) * TF32_FLOP_PER_CLK_SM
    peak = peaks["bf16_tflops"] * ratio
    ach = passes * flops / t / 1e12
    mhz = clock_mhz or peaks["sm_max_mhz"]
    clock_peak = sm_count * per_clk * mhz * 1e6 / 1e12
    extra = {}
    if passes == 3:
        # the FP32-accurate product measured the way an FP32 GEMM is: 2MNK useful flop per
        # launch against the CUDA cores' FP32 FMA peak
        simt = fp32_simt_peak_tflops(sm_count, peaks["sm_max_mhz"])
        extra["vs_fp32_simt_peak"] = {"achieved": flops / t / 1e12, "peak": simt,
                                      "frac": flops / t / 1e12 / simt, "unit": "TFLOP/s",
                                      "basis": "2MNK per launch / FP32 FFMA peak"}
    return {**extra, "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
            "frac": ach / peak, "kernel": name,
            "peak_basis": (f"bf16 burst {peaks['bf16_tflops']:.0f} (FP16 = BF16 rate)" if f16 else
                           f"bf16 burst {peaks['bf16_tflops']:.0f} x {TF32_PER_BF16:.4f} "
                           "(nominal TF32/BF16)"),
            "tensor_flop_per_launch": passes * flops,
            "clock_peak": clock_peak, "frac_of_clock_peak": ach / clock_peak,
            "clock_peak_basis": f"{sm_count} SMs x {per_clk} {'FP16' if f16 else 'TF32'} "
                                f"flop/clk/SM x {mhz:.0f} MHz"}


def device_clock(sg, kind, stream):
    """SM clock (MHz) the last tensor-core (kind "tc", "tc16") or CUDA-core ("simt")
    launch measured for itself; None if no such record is there."""
    try:
        return sg.simt_clock_mhz(stream) if kind == "simt" else sg.tc_clock_mhz(stream)
    except sg.SgemmError:
        return None


def add_device_clock_peak(roof, mhz, sm_count, kind):
    """The roofline at the SM clock the kernel itself measured (sgemm_tc_clock_mhz,
    sgemm_simt_clock_mhz): under the chip's power limit a busy kernel runs below the
    2070 MHz maximum. Tensor: 4096 TF32 flop/clk/SM; CUDA cores: 128 FMA lanes x 2."""
    if not mhz:
        return
    per_clk = {"tc": TF32_FLOP_PER_CLK_SM, "tc16": 2 * TF32_FLOP_PER_CLK_SM}.get(kind, 256)
    peak = sm_count * per_clk * mhz * 1e6 / 1e12
    roof["device_clock_mhz"] = mhz
    roof["device_clock_peak"] = peak
    roof["frac_of_device_clock_peak"] = roof["achieved"] / peak


def run_probes(sg, torch):
    """Peak rates measured on this GPU by the library's probes (best of three runs of
    about 10-20 ms each): register-only FFMA and packed FFMA2 loops on every SM, and the
    pair MMA (kind::tf32, 256 x 256 x 8) issued back to back from shared memory."""
    stream = torch.cuda.current_stream()
    out = {}
    for key, probe, iters in (("ffma", sg.PROBE_FFMA, 1 << 17),
                              ("ffma2", sg.PROBE_FFMA2, 1 << 17),
                              ("tf32_mma", sg.PROBE_TF32_MMA, 1 << 15),
                              ("f16_mma", sg.PROBE_F16_MMA, 1 << 15)):
        sg.peak_probe(probe, 1024 if probe in (sg.PROBE_FFMA, sg.PROBE_FFMA2) else 256, stream)
        best = 0.0
        for _ in range(3):
            flop, ms = sg.peak_probe(probe, iters, stream)
            rate = flop / (ms * 1e-3) / 1e12
            if rate > best:
                out[key + "_sm_mhz"] = device_clock(
                    sg, "simt" if probe in (sg.PROBE_FFMA, sg.PROBE_FFMA2) else "tc", stream)
            best = max(best, rate)
        out[key + "_tflops"] = best
    return out


def add_probe_peak(roof, kind, probes):
    """The dominant kernel's work rate against the matching probe's measured rate."""
    if not probes or kind in ("gevm", "gemv", "smalln"):
        return
    if kind == "simt":
        peak = max(probes["ffma_tflops"], probes["ffma2_tflops"])
        basis = "best of the FFMA and FFMA2 register-only probes"
    elif kind == "tc16":
        peak = probes["f16_mma_tflops"]
        basis = "shared-memory-resident pair MMA probe (tcgen05 kind::f16, 256x256x16)"
    else:
        peak = probes["tf32_mma_tflops"]
        basis = "shared-memory-resident pair MMA probe (tcgen05 kind::tf32, 256x256x8)"
    roof["probe_peak"] = peak
    roof["frac_of_probe_peak"] = roof["achieved"] / peak
    roof["probe_peak_basis"] = basis


def cpu_model() -> str:
    """The host CPU's model, read-only: lscpu's "Model name" (Arm hosts list no model
    name in /proc/cpuinfo), else /proc/cpuinfo's, else the machine type."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            key, _, val = line.partition(":")
            if key.strip() in ("Model name", "Model Name") and val.strip():
                vendor = next((l.partition(":")[2].strip() for l in out.splitlines()
                               if l.partition(":")[0].strip() == "Vendor ID"), "")
                return f"{vendor} {val.strip()}".strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo", encoding="utf-8", errors="replace"):
            key, _, val = line.partition(":")
            if key.strip().lower() in ("model name", "cpu model") and val.strip():
                return val.strip()
    except OSError:
        pass
    return platform.machine() or "unknown"


def cpu_baseline(M, N, K, seed, dist, target_s):
    """The oracle (unchanged) on the first R rows of the product, R sized so that the
    sample takes about target_s seconds on this host's cores."""
    import oracle
    from dense_fp32_gemm_sgemm_gb300.inputs import make_inputs
    A, B = make_inputs(M, N, K, seed, dist)
    threads = oracle.default_threads()
    rows = min(M, threads)
    t0 = time.perf_counter()
    oracle.gemm(A[:rows], B, with_scale=False, threads=threads)
    probe = time.perf_counter() - t0
    per_row = probe / rows
    rows = int(max(threads, min(M, (target_s / max(per_row, 1e-9)) // threads * threads)))
    t0 = time.perf_counter()
    oracle.gemm(A[:rows], B, with_scale=False, threads=threads)
    dt = time.perf_counter() - t0
    return {"value": 2.0 * rows * N * K / dt / 1e12, "unit": "TFLOP/s", "cores": threads,
            "threads": threads, "cpu_model": cpu_model(), "kind": "oracle", "seconds": dt,
            "sample": f"first {rows} of {M} rows of the {M}x{N}x{K} product "
                      f"({rows}x{N}x{K}, C only, double accumulation)"}


# ----------------------------------------------------------------------------- arms
def workload_config(shape, mode_name, world):
    """The `config` object of both arms' lines: the workload, nothing about the arm."""
    M, N, K = shape
    return {"workload": f"sgemm {M}x{N}x{K} row-major fp32, C = A.B reduced over N",
            "M": M, "N": N, "K": K, "seed": 2, "dist": "uniform[-1,1)", "mode": mode_name,
            "parallelism": "replicas" if world > 1 else "single",
            "l2": ("inputs larger than the 129 MB L2; no flush"
                   if 4 * (M * N + N * K + M * K) > 129e6 else "inputs fit in L2; no flush")}


def run_reference(args, shape):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from dense_fp32_gemm_sgemm_gb300.inputs import make_inputs
    M, N, K = shape
    A, B = make_inputs(M, N, K, 2, "uniform")
    threads = oracle.default_threads()
    # rows per step sized for about 2 s of oracle work per step
    rows = min(M, threads)
    t0 = time.perf_counter()
    oracle.gemm(A[:rows], B, with_scale=False, threads=threads)
    per_row = (time.perf_counter() - t0) / rows
    rows = int(max(threads, min(M, (2.0 / max(per_row, 1e-9)) // threads * threads)))
    for i in range(args.warmup):
        oracle.gemm(A[:rows], B, with_scale=False, threads=threads)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.gemm(A[:rows], B, with_scale=False, threads=threads)
    dt = (time.perf_counter() - t0) / args.steps
    value = 2.0 * rows * N * K / dt / 1e12
    sample = (f"first {rows} of {M} rows per step ({rows}x{N}x{K}), C only, double "
              "accumulation; TFLOP/s counts the sample's own 2 x rows x N x K flop")
    line = {"impl": "reference", "metric": "TFLOP/s", "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(shape, args.mode, 1),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                             "threads": threads, "cpu_model": cpu_model(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, shape):
    import torch
    import dense_fp32_gemm_sgemm_gb300 as sg
    from dense_fp32_gemm_sgemm_gb300 import build as sg_build

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: this benchmark needs a GB300")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl")
    if rank == 0:
        sg_build.build()
    barrier(world)
    sg.lib()
    peaks, peak_src = load_peaks()
    props = torch.cuda.get_device_properties(local)
    sm_count = props.multi_processor_count
    mode = sg.MODES[args.mode.lower()]
    M, N, K = shape
    run = Runner(torch, sg, M, N, K, 2, "uniform", f"cuda:{local}")
    kernel_id, tiles = sg.plan(M, N, K, mode)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.wait_first()
    res = run.timed(mode, args.steps, args.warmup, world)
    if sampler:
        time.sleep(0.1)
        sampler.stop()
    clocks = sampler.summary(res["t0"], res["t1"]) if sampler else None

    ms = max_over_ranks(res["ms_per_step"], world)
    kern_ms = max_over_ranks(res["kernel_ms"], world)
    flops = 2.0 * M * N * K
    value = world * flops / (ms * 1e-3) / 1e12
    roof = roofline_for(sg, kernel_id, M, N, K, kern_ms, peaks, sm_count,
                        clocks["sm_mhz"] if clocks else None)
    name, kind = KERNEL_OF_PLAN[kernel_id]
    if kind in ("tc", "tc16", "simt"):
        # the clock the last timed GEMM launch ran at, measured by the kernel itself
        dev_mhz = device_clock(sg, kind, run.stream)
        if clocks is not None:
            clocks["device_sm_mhz"] = dev_mhz
            clocks["device_basis"] = ("clock64 cycles / globaltimer ns on CTA 0 of the last "
                                      "timed GEMM launch" + (", first MMA to last store"
                                                             if kind != "simt" else ""))
        add_device_clock_peak(roof, dev_mhz, sm_count, kind)
    roof["traffic"] = recorded_traffic(name, shape, kind)
    roof["peak_source"] = peak_src
    roof["kernel_ms"] = kern_ms

    protocols = run.protocols(
        mode, flops,
        (lambda: device_clock(sg, kind, run.stream)) if kind in ("tc", "tc16", "simt") else None)

    e2e = None
    if not args.no_e2e:
        dt, h2d, d2h = run.e2e(mode, max(3, min(args.steps, 10)), 2)
        dt = max_over_ranks(dt, world)
        e2e = {"value": world * flops / dt / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": dt * 1e3, "api": "solve_host"}

    variants = {}
    if not args.no_variants and shape == HEADLINE:
        variants = run_variants(torch, sg, mode, run, peaks, sm_count)

    probes = None
    if not args.no_probes:
        probes = run_probes(sg, torch)
        add_probe_peak(roof, kind, probes)
        for v in variants.values():
            if "roofline" in v:
                vkind = {"simt_gemm": "simt", "tc_gemm_3xfp16": "tc16"}.get(
                    v["roofline"]["kernel"], "tc")
                add_probe_peak(v["roofline"], vkind, probes)
    for v in variants.values():
        if "roofline" in v:
            v["roofline"] = compact_roofline(v["roofline"])

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        del run
        torch.cuda.empty_cache()
        cpu = cpu_baseline(M, N, K, 2, "uniform", args.cpu_seconds)

    vs_baseline, vs_basis = vs_pages(args.mode, shape, value)
    line = {"metric": "TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": vs_baseline,
            "vs_baseline_basis": vs_basis,
            "dtype": {sg.MODE_TF32: "tf32", sg.MODE_3XFP16_SCALED: "f16x3"}.get(mode, "f32"),
            "data": "synthetic",
            "config": workload_config(shape, args.mode, world),
            "plan": {"kernel": name, "tiles": tiles},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": res["launches"], "clocks": clocks,
            "kernel_ms": {"mean": res["kernel_ms"], "min": res["kernel_ms_min"],
                          "max": res["kernel_ms_max"], "median": res["kernel_ms_median"],
                          "launches_timed": "every" if res["kernel_events_every"] == 1
                          else f"every {res['kernel_events_every']}th of the timed steps"},
            "probes": probes,
            "timing_protocols": protocols,
            "variants": variants}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def torch_matmul_context(torch, head, steps=10, warmup=3):
    """Another system, for context only: torch.matmul (cuBLAS) on the same device-resident
    operands, FP32 (TF32 disallowed) and TF32. Never part of the library."""
    out = {}
    saved = torch.backends.cuda.matmul.allow_tf32
    try:
        for label, tf32 in (("context_torch_matmul_fp32", False),
                            ("context_torch_matmul_tf32", True)):
            torch.backends.cuda.matmul.allow_tf32 = tf32
            C = torch.empty((head.M, head.K), device=head.dA.device)
            for _ in range(warmup):
                torch.matmul(head.dA, head.dB, out=C)
            torch.cuda.synchronize()
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            start.record()
            for _ in range(steps):
                torch.matmul(head.dA, head.dB, out=C)
            end.record()
            torch.cuda.synchronize()
            ms = start.elapsed_time(end) / steps
            out[label] = {"workload": f"{head.M}x{head.N}x{head.K} uniform seed 2",
                          "system": "torch.matmul (cuBLAS), another system, context only",
                          "ms_per_step": ms, "unit": "TFLOP/s",
                          "value": 2.0 * head.M * head.N * head.K / (ms * 1e-3) / 1e12}
            del C
    finally:
        torch.backends.cuda.matmul.allow_tf32 = saved
    return out


COMPACT_ROOF_KEYS = ("bound", "kernel", "achieved", "peak", "unit", "frac", "kernel_ms",
                     "device_clock_mhz", "frac_of_device_clock_peak", "frac_of_probe_peak")


def compact_roofline(roof):
    """The keys of a variant's roofline that the line keeps (the full form is the main
    path's `roofline`)."""
    return {k: roof[k] for k in COMPACT_ROOF_KEYS if k in roof}


def run_variants(torch, sg, main_mode, head, peaks, sm_count):
    """The other paths on their own workloads, fewer steps each. The explicit 1xTF32
    variant comes last in the line."""
    out = {}

    def gemm_variant(label, mode):
        if mode == main_mode or sg.plan(*HEADLINE, mode)[0] < 0:
            return
        r = head.timed(mode, 10, 3)
        kid = sg.plan(*HEADLINE, mode)[0]
        roof = roofline_for(sg, kid, *HEADLINE, r["kernel_ms"], peaks, sm_count)
        vkind = KERNEL_OF_PLAN[kid][1]
        add_device_clock_peak(roof, device_clock(sg, vkind, head.stream), sm_count, vkind)
        roof["kernel_ms"] = r["kernel_ms"]
        out[label] = {"workload": "8192x6144x4096 uniform seed 2", "ms_per_step": r["ms_per_step"],
                      "value": 2.0 * 8192 * 6144 * 4096 / (r["ms_per_step"] * 1e-3) / 1e12,
                      "unit": "TFLOP/s", "roofline": roof}

    for label, mode in (("fp32_simt", sg.MODE_FP32_SIMT), ("fp32_3xtf32", sg.MODE_FP32_3XTF32),
                        ("3xfp16_scaled", sg.MODE_3XFP16_SCALED)):
        gemm_variant(label, mode)
    out.update(torch_matmul_context(torch, head))
    for label, (M, N, K) in (("gevm_1x8192x8192", (1, 8192, 8192)),
                             ("gemv_8192x8192x1", (8192, 8192, 1)),
                             ("thin_8192x64x8192", (8192, 64, 8192))):
        r_ = Runner(torch, sg, M, N, K, 3, "normal", head.dA.device)
        r = r_.timed(sg.MODE_FP32, 20, 3)
        kid = sg.plan(M, N, K, sg.MODE_FP32)[0]
        byts = 4.0 * (M * N + N * K + M * K)
        ach = byts / (r["kernel_ms"] * 1e-3) / 1e9
        out[label] = {"workload": f"{M}x{N}x{K} normal seed 3",
                      "ms_per_step": r["ms_per_step"], "kernel": KERNEL_OF_PLAN[kid][0],
                      "kernel_ms": r["kernel_ms"],
                      "value": 2.0 * M * N * K / (r["ms_per_step"] * 1e-3) / 1e12,
                      "unit": "TFLOP/s",
                      "hbm": {"achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": ach / peaks["hbm_gbs"], "bytes": byts}}
        del r_
    gemm_variant("tf32_1x", sg.MODE_TF32)
    return out


def main(argv=None):
    args = parse_args(argv)
    shape = tuple(int(x) for x in args.shape.split(",")) if args.shape else HEADLINE
    if args.impl == "reference":
        return run_reference(args, shape)
    return run_ours(args, shape)


if __name__ == "__main__":
    sys.exit(main())
