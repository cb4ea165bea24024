"""The bench's clock record on CPU: nvidia-smi lines (faked here) are kept with their arrival times, and each timed
region's figures come from the samples printed while it ran -- the device-timed steps and the end-to-end steps each
get their own median clock and throttle reasons."""
import bench


def _line(sm, power_cap=False, thermal=False):
    act = lambda b: "Active" if b else "Not Active"
    return (f"0, {sm}, 2070, 900.00, 0x0000000000000004, Not Active, {act(thermal)}, Not Active, {act(power_cap)}")


class _Done:
    stdout = []

    def poll(self):
        return None

    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.proc = _Done()
    s.lines = list(lines)
    return s


def test_each_region_takes_its_own_samples():
    lines = [(0.9, _line(2070)), (1.0, _line(2070)), (1.5, _line(2070)), (2.0, _line(2070)),
             (3.0, _line(1800, power_cap=True)), (3.5, _line(1810, power_cap=True)), (4.0, _line(1820, True))]
    s = _sampler(lines)
    timed = s.summary(1.0, 2.0)
    assert timed["sm_mhz"] == 2070 and timed["reasons"] == [] and timed["samples"] == 3
    assert timed["samples_from"] == "the timed region"
    e2e = s.stop(3.0, 4.0)
    assert e2e["sm_mhz"] == 1810 and e2e["reasons"] == ["sw_power_cap"] and e2e["samples"] == 3


def test_a_region_without_samples_falls_back_to_the_window():
    s = _sampler([(0.0, _line(2000)), (10.0, _line(2070, thermal=True))])
    out = s.summary(4.0, 5.0)
    assert out["samples_from"] == "the sampling window around it"
    assert out["samples"] == 2 and out["reasons"] == ["hw_thermal_slowdown"]


def test_no_nvidia_smi():
    s = bench.ClockSampler(0)
    assert s.stop(0.0, 1.0)["reasons"] == ["nvidia-smi unavailable"]
