"""bench.py's clock record: nvidia-smi samples are kept only when their own timestamps fall
inside the timed region, and throttle reasons seen there are reported (no GPU needed)."""
import datetime
import time

import bench


def _line(ts, sm, smax=2070, reasons=("Not Active",) * 4):
    stamp = datetime.datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([stamp, "0", str(sm), str(smax), "812.3", "0x0000000000000000"] + list(reasons))


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler(lines, region):
    s = bench.ClockSampler(0)
    s.proc = _Done()
    s.lines = lines
    s.mark(*region)
    return s


def test_samples_outside_the_region_are_dropped():
    t0 = time.time()
    lines = [_line(t0 - 1.0, 1200),  # before: a leftover idle clock
             _line(t0 + 0.10, 2070), _line(t0 + 0.15, 2055), _line(t0 + 0.20, 2070),
             _line(t0 + 5.0, 900)]  # after
    rec = _sampler(lines, (t0, t0 + 0.3)).stop()
    assert rec["samples"] == 3
    assert rec["sm_mhz"] == 2070.0
    assert rec["sm_mhz_min"] == 2055.0
    assert rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == []


def test_throttle_reasons_inside_the_region_are_reported():
    t0 = time.time()
    hot = ("Not Active", "Active", "Not Active", "Active")  # hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    lines = [_line(t0 - 2.0, 1500, reasons=("Active",) * 4), _line(t0 + 0.1, 1900, reasons=hot)]
    rec = _sampler(lines, (t0, t0 + 0.2)).stop()
    assert rec["samples"] == 1
    assert rec["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_malformed_lines_are_ignored():
    t0 = time.time()
    lines = ["", "garbage", "a, b, c", _line(t0 + 0.1, 2070)]
    rec = _sampler(lines, (t0, t0 + 0.2)).stop()
    assert rec["samples"] == 1


def test_plan_times_cover_every_plan_of_the_step(lib):
    # the plans a workload holds directly or through its EinGraph object are timed apart from
    # the step (no GPU needed: ein_plan is host code)
    class Graph:
        pass

    Graph.__module__ = "tensor_relational_algebra_gb300.eingraph"

    class Workload:
        pass

    wl = Workload()
    wl.p = lib.Plan("ij,jk->ik:add:max", [256, 64, 256], [2, 1, 1, 2])
    wl.g = Graph()
    wl.g.p_proj = lib.Plan("sa,ahd->shd:mul:sum:in=bf16:out=bf16", [256, 256, 2, 128], [1, 1, 1, 2, 1])
    t = bench.plan_times(lib, wl, reps=3)
    assert set(t) == {"ij,jk->ik:add:max d=[2, 1, 1, 2]", "sa,ahd->shd:mul:sum:in=bf16:out=bf16 d=[1, 1, 1, 2, 1]"}
    assert all(v >= 0 for v in t.values())
