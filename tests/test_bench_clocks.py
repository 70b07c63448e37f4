"""The benchmark's clock record: the SM clock median under load, the maximum,
and the throttle reasons that were active at any sample, parsed from the
nvidia-smi CSV the sampler writes during the timed region."""
import bench


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _record(tmp_path, lines):
    p = tmp_path / "clocks.csv"
    p.write_text("\n".join(lines) + "\n")
    s = bench.ClockSampler(0)
    s.proc, s.path = _Done(), str(p)
    return s.stop()


def test_median_max_and_no_reasons(tmp_path):
    rec = _record(tmp_path, [
        "0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 980.2, 0x0, Not Active, Not Active, Not Active, Not Active",
    ])
    assert rec["sm_mhz"] == 2070.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == [] and rec["samples"] == 3


def test_reasons_active_in_any_sample_are_reported(tmp_path):
    rec = _record(tmp_path, [
        "0, 1900, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1800, 2070, 1400.0, 0x48, Not Active, Active, Not Active, Active",
        "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ])
    assert rec["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert rec["sm_mhz"] == 1900.0


def test_malformed_lines_are_skipped(tmp_path):
    rec = _record(tmp_path, ["", "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
                             "garbage", "0, 2070, 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active"])
    assert rec["samples"] == 1 and rec["sm_mhz"] == 2070.0


def test_no_sampler_is_reported_as_such():
    s = bench.ClockSampler(0)
    s.proc = None
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]
