"""Host logic of bench.py that needs no GPU: reading the nvidia-smi clock
samples taken during the timed region (median SM clock, its maximum, and
which throttle reasons were active at any sample)."""
import bench


def _line(sm, smax=2070, reasons=("Not Active",) * 4, active="0x0000000000000000"):
    return ", ".join(["0", str(sm), str(smax), "900.00", active] + list(reasons))


def test_clean_run_has_no_reasons_and_the_median_clock():
    text = "\n".join(_line(s) for s in (2070, 2055, 2070, 1980, 2070))
    r = bench.parse_clock_samples(text)
    assert r == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5}


def test_each_reason_column_is_reported_by_name():
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for i, name in enumerate(names):
        reasons = ["Not Active"] * 4
        reasons[i] = "Active"
        text = "\n".join([_line(2070), _line(1900, reasons=reasons), _line(2070)])
        assert bench.parse_clock_samples(text)["reasons"] == [name]


def test_unparsable_lines_are_skipped_and_empty_output_is_none():
    text = "\n".join(["", "0, [N/A], 2070, 900, 0x0, Not Active, Not Active, Not Active, Not Active",
                      "garbage", _line(1500)])
    r = bench.parse_clock_samples(text)
    assert r["samples"] == 1 and r["sm_mhz"] == 1500.0
    assert bench.parse_clock_samples("") is None
    assert bench.parse_clock_samples("0, [N/A], [N/A], 0, 0x0, a, b, c, d") is None


def test_headline_traffic_record_is_used_only_for_the_captured_source(monkeypatch):
    """The DRAM bytes the bench reports for its dominant kernel come from the
    committed ncu record only while the kernel's sources hash to the value
    recorded with the capture; otherwise the bench reports null."""
    import json
    rec = json.load(open(f"{bench.ROOT}/profiles/traffic.json"))["gemv_split_nvfp4_m1"]
    t = bench.ncu_traffic("gemv_split_nvfp4_m1")
    if t is not None:
        # the capture moved at most a few percent more than the algorithmic
        # bytes of one call (150,405,132 B: no re-reads)
        assert 150_405_132 <= t <= 1.05 * 150_405_132
    monkeypatch.setattr(bench, "kernel_src_sha", lambda files: "0" * 16)
    assert bench.ncu_traffic("gemv_split_nvfp4_m1") is None
    monkeypatch.setattr(bench, "kernel_src_sha", lambda files: rec["src_sha"])
    assert bench.ncu_traffic("gemv_split_nvfp4_m1") == rec["dram_bytes_per_launch"]
    assert bench.ncu_traffic("no_such_kernel") is None
