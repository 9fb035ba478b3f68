"""Host-side logic of bench.py (no GPU): the clock summary and the roofline
terms of a configuration."""
import bench


def test_clock_summary_medians_maxima_and_reasons():
    lines = [
        "0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active, 3996, 3996",
        "0, 1980, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active, 3996, 3996",
        "0, 2010, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active, 3900, 3996",
        "garbage line",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active, 1, 1",
    ]
    c = bench.ClockSampler.summarize(lines)
    assert c["samples"] == 3
    assert c["sm_mhz"] == 2010.0 and c["sm_max_mhz"] == 2070.0
    assert c["mem_mhz"] == 3996.0 and c["mem_max_mhz"] == 3996.0
    assert c["power_w"] == 1000.0
    assert c["reasons"] == ["sw_power_cap"]


def test_clock_summary_of_nothing():
    c = bench.ClockSampler.summarize([])
    assert c["samples"] == 0 and c["sm_mhz"] is None and c["reasons"] == []


def test_roofline_terms_of_the_headline_workload():
    """(2,16,96,128,16,128) with window (3,7,7): 4 * L * NH * HD * 147 useful
    flops and four bf16 tensors of L * NH * HD elements."""
    shape, kernel = bench.WORKLOADS[bench.HEADLINE]
    L = 2 * 16 * 96 * 128
    flops = 4.0 * L * 16 * 128 * 147
    nbytes = 4.0 * L * 16 * 128 * 2
    assert bench.useful_flops(shape, kernel) == flops
    assert bench.min_bytes(shape) == nbytes
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1500.0}
    t = 2000e-6
    r = bench.roofline_terms(shape, kernel, t, peaks)
    assert r["bound"] == "hbm"   # 147 / 2 flop per byte is below the ridge of 333
    assert abs(r["roofline_us"] - nbytes / 6000e9 * 1e6) < 1e-9
    assert abs(r["roofline_frac"] - nbytes / 6000e9 / t) < 1e-12
    assert abs(r["useful_tflops"] - flops / t / 1e12) < 1e-9
    # a large window is bound by the tensor peak
    shape4, kernel4 = (1, 16, 48, 48, 8, 64), (11, 11, 11)
    assert bench.roofline_terms(shape4, kernel4, t, peaks)["bound"] == "tensor"
