"""Host logic of bench.py that needs no GPU: the clock summary taken from
nvidia-smi samples during the timed region (median SM clock, the throttle
reasons seen, the fallback window for a region shorter than the sampling
period, unreadable fields), and the kernel name a launch is reported under."""
import bench


def sampler_with(rows):
    s = object.__new__(bench.ClockSampler)
    s.proc = None
    s.samples = rows
    return s


def row(t, sm, smax=2070, power=700.0, hw="Not Active", hwt="Not Active", swt="Not Active",
        cap="Not Active"):
    return (t, ["0", str(sm), str(smax), str(power), "0x0", hw, hwt, swt, cap])


def test_median_clock_and_reasons_inside_the_region():
    rows = [row(0.5, 1000), row(1.0, 2070), row(1.1, 2040), row(1.2, 2070, cap="Active"),
            row(1.3, 2055, power=1390.5), row(5.0, 900, hw="Active")]
    s = sampler_with(rows).summary(0.9, 1.4)
    assert s["samples"] == 4 and s["sm_mhz"] == 2062.5 and s["sm_max_mhz"] == 2070.0
    assert s["power_w_max"] == 1390.5
    assert s["reasons"] == ["sw_power_cap"]  # the hw_slowdown sample lies outside the region
    assert s["note"] == "samples inside the timed region"


def test_short_region_takes_the_samples_around_it():
    rows = [row(0.8, 2070), row(1.6, 2070, hwt="Active"), row(3.0, 1500)]
    s = sampler_with(rows).summary(1.0, 1.2)
    assert s["samples"] == 2 and s["reasons"] == ["hw_thermal_slowdown"]
    assert "shorter than the sampling period" in s["note"]


def test_unreadable_fields_are_skipped():
    rows = [(1.0, ["0", "[N/A]", "2070", "[N/A]", "0x0", "Not Active", "Active", "Active",
                   "Not Active"]), row(1.1, 2070)]
    s = sampler_with(rows).summary(0.9, 1.2)
    assert s["sm_mhz"] == 2070.0 and s["power_w_max"] == 700.0
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_no_samples():
    s = sampler_with([]).summary(0.0, 1.0)
    assert s["sm_mhz"] is None and s["samples"] == 0 and s["reasons"] == []


def test_hop1_kernel_label_follows_the_launcher():
    """The bench names the kernel hop 1 runs on a workload by the launcher's
    rules: int4 with eight sources a node on whole warp units takes the staged
    kernel, other widths and source counts that are multiples of four the
    register-chunk kernel, other whole-unit rows the tiled hop kernel and
    ragged rows the general one."""
    import dataclasses
    from synth import workloads as W
    assert bench.kernel_label("qgz_hop1", W.WORKLOADS["7b"]) == "hop1_staged_kernel<LOGB>"
    assert bench.kernel_label("qgz_hop1", W.WORKLOADS["two_hop"]) == "hop1_staged_kernel<LOGB>"
    wl = W.WORKLOADS["two_hop"]
    g = wl.qgz
    int8 = dataclasses.replace(wl, qgz=dataclasses.replace(g, bits=8))
    assert bench.kernel_label("qgz_hop1", int8) == "hop1_kernel<BITS, LOGB, SCH>"
    g4 = dataclasses.replace(wl, qgz=dataclasses.replace(g, gpus_per_node=4))
    assert bench.kernel_label("qgz_hop1", g4) == "hop1_kernel<BITS, LOGB, SCH>"
    assert bench.kernel_label("qgz_hop1", W.WORKLOADS["tiny"]).startswith("hop_tiled_kernel")
    # 2 x 8 ranks with 3 * 256-element slices: rows of 1536 elements, not whole 1024-element units
    ragged = dataclasses.replace(wl, qgz=dataclasses.replace(g, bucket=16 * 3 * 256))
    assert bench.kernel_label("qgz_hop1", ragged).startswith("hop_kernel")
    assert bench.kernel_label("qwz_quant", wl) == bench.KERNEL_OF["qwz_quant"]
