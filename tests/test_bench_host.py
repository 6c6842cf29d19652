"""The bench's host-side helpers that need no GPU: the clock / throttle summary
of nvidia-smi samples taken during the timed region, and the node list of each
workload's mask program."""
import bench


def test_clock_summary_median_max_and_reasons():
    lines = ["2070, 2070, 900.5, Not Active, Not Active, Not Active, Not Active"] * 3 + [
        "1500, 2070, 1390.1, Active, Not Active, Not Active, Active",
        "garbage",                                                   # skipped: too few fields
        "[N/A], 2070, 800, Not Active, Not Active, Not Active, Not Active",  # skipped: no clock
        "2040, 2070, [N/A], Not Active, Not Active, Active, Not Active",     # power unreadable: kept
    ]
    r = bench.ClockSampler.summarise(lines)
    assert r["samples"] == 5
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    r = bench.ClockSampler.summarise([])
    assert r["sm_mhz"] is None and r["sm_max_mhz"] is None and r["reasons"] == [] and r["samples"] == 0


def test_mask_nodes_of_the_workloads():
    docs, W = object(), object()                        # stand-ins for the device tensors
    n2 = bench.mask_nodes(bench.WORKLOADS[2], docs, W)
    assert ("same_doc", docs) in n2 and ("causal",) in n2
    assert any(x[0] == "window" and x[1] == 1024 for x in n2)   # fixed window: an int
    n5 = bench.mask_nodes(bench.WORKLOADS[5], docs, W)
    assert ("window", W) in n5                           # the sweep: the device scalar
    n3 = bench.mask_nodes(bench.WORKLOADS[3], None, W)
    assert ("sink", 4) in n3
    for w in bench.WORKLOADS.values():                   # postfix programs keep their length
        assert len(bench.mask_nodes(w, docs, W)) == len(w.mask.nodes)


def test_clock_sampler_stop_summarises_its_lines(monkeypatch):
    class _Proc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    cs = bench.ClockSampler(0)
    cs.proc = _Proc()
    cs.lines = ["2070, 2070, 900, Not Active, Not Active, Not Active, Not Active"] * 2
    assert cs.stop() == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 2}
    cs2 = bench.ClockSampler(0)                           # nvidia-smi could not start
    assert cs2.stop()["reasons"] == ["nvidia-smi unavailable"]
