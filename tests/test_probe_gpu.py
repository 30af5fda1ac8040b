"""Peak-rate probes on the GPU: they run, leave no device error, and report rates in the
range the hardware allows (an FP32 lane does at most one FMA per clock; the tensor
probe must at least beat the CUDA-core FMA rate and stay below the BF16 rate)."""

import pytest

import dense_fp32_gemm_sgemm_gb300 as sg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def device():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    props = torch.cuda.get_device_properties(0)
    return torch, props.multi_processor_count


def rate(probe, iters, torch):
    flop, ms = sg.peak_probe(probe, iters, torch.cuda.current_stream())
    assert flop > 0 and ms > 0
    assert sg.device_error() == sg.OK
    return flop / (ms * 1e-3) / 1e12


def test_ffma_probes(device):
    torch, sms = device
    ceiling = sms * 128 * 2 * 2.2e9 / 1e12  # one FMA per lane per clock at <= 2.2 GHz
    for probe in (sg.PROBE_FFMA, sg.PROBE_FFMA2):
        r = rate(probe, 1 << 14, torch)
        assert 0.3 * ceiling < r < 1.05 * ceiling, (probe, r, ceiling)


def test_tf32_mma_probe(device):
    torch, sms = device
    r = rate(sg.PROBE_TF32_MMA, 1 << 12, torch)
    assert 100.0 < r < 2500.0, r
    # the probe leaves the context usable: a product still works afterwards
    A = torch.ones(256, 64, device="cuda")
    B = torch.ones(64, 256, device="cuda")
    C = sg.matmul(A, B)
    torch.cuda.synchronize()
    assert bool((C == 64.0).all())


def test_tc_clock_record(device):
    """The tensor-core kernels measure their own SM clock: after the TF32 probe and after a
    3xTF32 product the reading lies between 500 MHz and the 2070 MHz maximum (with a
    margin for the two timers' granularity), and the probe's pure-MMA rate matches 4096
    TF32 flop per clock per SM at that clock to within 10 %."""
    torch, sms = device
    flop, ms = sg.peak_probe(sg.PROBE_TF32_MMA, 1 << 14, torch.cuda.current_stream())
    mhz = sg.tc_clock_mhz()
    assert 500.0 < mhz < 2200.0, mhz
    at_clock = 4096.0 * sms * mhz * 1e6
    assert 0.9 < flop / (ms * 1e-3) / at_clock < 1.1, (flop / ms, at_clock)
    A = torch.rand(2048, 1024, device="cuda")
    B = torch.rand(1024, 2048, device="cuda")
    sg.matmul(A, B, mode=sg.MODE_FP32_3XTF32)
    mhz = sg.tc_clock_mhz()
    assert 500.0 < mhz < 2200.0, mhz


def test_simt_clock_record(device):
    """The CUDA-core kernels measure their own SM clock as well: after the FFMA2 probe the
    reading is plausible and the probe's rate is at most one FMA per lane per clock at it;
    after a forced FFMA product the reading is plausible too."""
    torch, sms = device
    flop, ms = sg.peak_probe(sg.PROBE_FFMA2, 1 << 14, torch.cuda.current_stream())
    mhz = sg.simt_clock_mhz()
    assert 500.0 < mhz < 2200.0, mhz
    at_clock = sms * 128 * 2.0 * mhz * 1e6
    assert 0.5 < flop / (ms * 1e-3) / at_clock < 1.05, (flop / ms, at_clock)
    A = torch.rand(1024, 512, device="cuda")
    B = torch.rand(512, 1024, device="cuda")
    sg.matmul(A, B, mode=sg.MODE_FP32_SIMT)
    mhz = sg.simt_clock_mhz()
    assert 500.0 < mhz < 2200.0, mhz

