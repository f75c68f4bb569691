"""Host logic of bench.py's clock record: which nvidia-smi samples a window
takes, and what it reports (no GPU, no nvidia-smi: the sampler's rows are set
directly)."""
import bench


def _sampler(rows):
    s = bench.ClockSampler(0)
    s.proc = object()  # as if nvidia-smi had been started
    s.rows = rows
    return s


def _row(t, mhz, power, cap=False, thermal=False):
    flags = ["0x0", "Not Active", "Not Active", "Active" if thermal else "Not Active",
             "Active" if cap else "Not Active"]
    return (t, float(mhz), 2070.0, str(power), flags)


def _load_rows():
    # idle at both ends, power-capped load in between
    rows = [_row(0.0, 2070, 190)]
    rows += [_row(0.1 * i, 1800 + i, 1300, cap=True) for i in range(1, 10)]
    rows.append(_row(1.0, 2070, 190))
    return rows


def test_trimmed_window_takes_only_the_load():
    c = _sampler(_load_rows()).window(0.0, 1.0, margin=-0.05, label="back to back")
    assert c["samples"] == 9
    assert c["sm_mhz"] == 1805.0  # median of 1801..1809
    assert c["power_w_max"] == 1300.0
    assert c["reasons"] == ["sw_power_cap"]
    assert c["window"] == "back to back"


def test_default_window_widens_by_the_margin():
    c = _sampler(_load_rows()).window(0.05, 0.95)
    assert c["samples"] == 11  # the idle samples at 0.0 and 1.0 fall within 50 ms
    assert c["sm_max_mhz"] == 2070.0
    assert c["window"] == "timed"


def test_thermal_reason_is_reported():
    rows = [_row(0.1 * i, 1500, 1400, thermal=True) for i in range(5)]
    c = _sampler(rows).window(0.0, 0.4)
    assert "sw_thermal_slowdown" in c["reasons"]


def test_short_region_falls_back_to_adjacent_samples():
    c = _sampler(_load_rows()).window(0.31, 0.32, margin=-0.05)
    assert c["window"].startswith("adjacent")
    assert c["samples"] == 3


def test_no_sampler_process():
    s = bench.ClockSampler(0)
    assert s.window(0.0, 1.0)["reasons"] == ["nvidia-smi unavailable"]
