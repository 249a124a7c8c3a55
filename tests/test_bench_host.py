"""Host-side logic of bench.py that needs no GPU: the clock-record checks of the measurement rules,
the clock summaries over a timed window, and the algorithmic flop counts of the workloads."""
import bench


def test_clocks_rejected_rules():
    ok = {"sm_mhz": 2070, "sm_max_mhz": 2070, "reasons": []}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected(dict(ok, reasons=["sw_power_cap"], sm_mhz=1500))   # kept and noted
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected(dict(ok, reasons=[r]))
    assert bench.clocks_rejected(dict(ok, sm_mhz=1200))                                # locked low, no reason
    assert not bench.clocks_rejected(None)
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]})


def test_nvml_summary_window_and_reasons():
    s = bench.NvmlSampler.__new__(bench.NvmlSampler)   # no NVML: only the summary logic
    s.samples = [(0.5, 1000, 2070, 100.0, 0x0),          # before the window
                 (1.0, 2070, 2070, 300.0, 0x4),
                 (1.5, 2000, 2070, 350.0, 0x0),
                 (2.0, 1990, 2070, 320.0, 0x8),
                 (3.0, 500, 2070, 50.0, 0x40)]           # after the window
    c = s.summary(1.0, 2.0)
    assert c["samples"] == 3 and c["sm_mhz"] == 2000 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"] and c["power_w_max"] == 350.0
    assert bench.clocks_rejected(c)
    assert s.summary(10.0, 11.0) is None


def test_smi_summary_parses_and_falls_back_to_whole_run():
    s = bench.ClockSampler(0)
    row = lambda mhz, act: [str(mhz), "2070", "250.5", "0x0", "Not Active", "Not Active", "Not Active", act]  # noqa: E731
    s.samples = [(1.0, row(2070, "Not Active")), (1.1, row(2060, "Active")), (5.0, row(2070, "Not Active"))]
    c = s.summary(1.0, 1.2)   # two samples: shorter than the sampling period allows, whole run used
    assert c["window"].startswith("whole run") and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"] and c["sm_mhz"] == 2070


def test_flop_counts():
    # forward X W0^T + (X A^T) B^T: 2M(out in + r in + out r); backward adds dX and the two
    # adapter gradients plus the rank-r passes
    f, b = bench.lora_flops(8, 32, 16, 4)
    assert f == 2 * 8 * (16 * 32 + 4 * 32 + 16 * 4)
    assert b > f
    fm, bm = bench.mlp_flops(8, 32, 64, 4)
    assert fm > 0 and bm > fm
