"""Host logic of the benchmark's clock record (no GPU): the summary of
sampled SM clocks and throttle reasons, from NVML rows and from nvidia-smi
CSV lines."""
import bench


def test_summary_of_nvml_rows():
    rows = [(2070.0, 2070.0, {"sw_power_cap"}), (1950.0, 2070.0, set()), (2010.0, 2070.0, set())]
    s = bench.clock_summary(rows, "nvml")
    assert s == {"sm_mhz": 2010.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                 "samples": 3, "source": "nvml"}


def test_no_samples_gives_no_record():
    assert bench.clock_summary([], "nvml") is None


def test_nvidia_smi_lines_parse_and_skip_garbage():
    c = bench.ClockSampler(0)
    c.lines = ["2070, 2070, Not Active, Not Active, Not Active, Active",
               "1900, 2070, Active, Not Active, Active, Not Active",
               "[N/A], 2070, Not Active, Not Active, Not Active, Not Active",
               "short line"]
    s = c.summary(0)
    assert s["samples"] == 2 and s["sm_mhz"] == 1985.0 and s["source"] == "nvidia-smi"
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert c.summary(2) is None


def test_nvml_reason_bits_are_distinct():
    bits = list(bench.NVML_REASON_BITS.values())
    assert len(set(bits)) == 4 and all(b & (b - 1) == 0 for b in bits)
    assert set(bench.NVML_REASON_BITS) == set(bench.REASON_NAMES)


def test_roofline_traffic_comes_from_the_committed_profile():
    """The line's roofline traffic is read from the committed ncu summary of
    the dgrad+wgrad launch: the file must keep a parseable per-launch figure
    of the size the step's operands and results imply (67 MB of e4m3
    operands read and up to 67 MB of bf16 results written)."""
    t = bench.profile_traffic("gemm_fp8_pair_dgrad_wgrad_4096.md")
    assert t is not None and 60e6 < t < 160e6
    assert bench.profile_traffic("no_such_profile.md") is None
