"""The benchmark's clock record: nvidia-smi samples taken during the timed
region are reduced to the median SM clock under load, the maximum clock and
the throttle reasons seen (host logic, fed with recorded-format lines)."""
import bench


def summary(lines):
    cs = bench.ClockSampler(0)
    cs.out = "\n".join(lines)
    return cs.summary()


def row(sm, smax=2070, hw="Not Active", hwt="Not Active", swt="Not Active", pcap="Not Active"):
    return f"0, {sm}, {smax}, 900.00, 0x0000000000000000, {hw}, {hwt}, {swt}, {pcap}"


def test_clean_run():
    s = summary([row(2070)] * 5 + [row(2062)])
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 6}


def test_reasons_are_collected_by_name():
    s = summary([row(2070), row(1900, pcap="Active"), row(2070, hw="Active"), row(2070, swt="Active"),
                 row(2070, hwt="Active")])
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]


def test_idle_samples_do_not_set_the_load_clock():
    s = summary([row(345)] * 2 + [row(2070)] * 4)
    assert s["sm_mhz"] == 2070.0 and s["samples"] == 6


def test_a_clock_stuck_low_is_reported_not_hidden():
    s = summary([row(990)] * 6)                 # every sample well below max: a leftover clock lock
    assert s["sm_mhz"] == 990.0 and s["sm_max_mhz"] == 2070.0 and s["reasons"] == []


def test_malformed_or_missing_samples():
    s = summary(["", "garbage", "0, [N/A], 2070, 1, 0x0, Not Active, Not Active, Not Active, Not Active"])
    assert s == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    s = summary(["garbage", row(2070)])
    assert s["samples"] == 1 and s["sm_mhz"] == 2070.0
