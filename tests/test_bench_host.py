"""Host-side arithmetic of bench.py, without a GPU."""

import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_steps_binned_by_clock():
    """Steps are paired with the clock samples taken while they ran and
    grouped by clock; the rate per clock follows from the step times."""
    b = _bench()
    s = b.NvmlClockSampler.__new__(b.NvmlClockSampler)
    t0 = 1000.0
    # 2,070 MHz for the first 10.5 ms, then 1,620 MHz
    s.samples = [(t0 + 0.00025 * i, 2070.0 if i < 42 else 1620.0, 0) for i in range(120)]
    # ten 1 ms steps
    spans = [(0.001 * i, 0.001 * i + 0.001) for i in range(10)]
    # later steps only in the second clock range
    spans += [(0.012 + 0.001 * i, 0.013 + 0.001 * i) for i in range(10)]
    flops = 2.0e12
    out = s.by_clock(t0, spans, flops, sms=152)
    assert [o["sm_mhz"] for o in out] == [1620, 2070]
    assert [o["steps"] for o in out] == [10, 10]
    for o in out:
        assert abs(o["kernel_ms"] - 1.0) < 1e-9
        assert abs(o["tflops"] - 2000.0) < 1e-6
        assert o["flop_per_clk_per_sm"] == round(flops / 1e-3 / (152 * o["sm_mhz"] * 1e6))


def test_step_without_a_sample_takes_the_nearest():
    b = _bench()
    s = b.NvmlClockSampler.__new__(b.NvmlClockSampler)
    s.samples = [(10.0, 1800.0, 0), (10.010, 1900.0, 0)]
    out = s.by_clock(10.0, [(0.0041, 0.0042)], 1e9, sms=1)
    assert len(out) == 1 and out[0]["steps"] == 1
