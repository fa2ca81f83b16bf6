"""The unit-rate probe behind the benchmark's FP32/SFU roofline denominators:
rates are positive, no FP32 rate exceeds the 128 lanes an SM of this family
has, and a repeat measures the same rates within a few percent."""
import pytest

pytestmark = pytest.mark.gpu


def test_probe_unit_rates_are_plausible_and_repeatable():
    import selective_state_space_147_b300 as L
    r1 = L.probe_unit_rates()
    r2 = L.probe_unit_rates()
    for k in ("fp32_lanes_per_sm_clock", "f32x2_lanes_per_sm_clock"):
        assert 32.0 <= r1[k] <= 128.0 * 1.02, (k, r1[k])
    assert 4.0 <= r1["ex2_per_sm_clock"] <= 64.0, r1["ex2_per_sm_clock"]
    for k in r1:
        assert abs(r1[k] - r2[k]) <= 0.05 * r1[k], (k, r1[k], r2[k])
