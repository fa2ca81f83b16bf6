"""Host-side logic of the benchmark (CPU only): the algorithmic work model, the
roofline arithmetic, the traffic table keyed by the kernel sources, and the
unit-rate probe hand-off with a stand-in library object."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_work_model_bytes_per_channel_token():
    b, d, L, N = 8, 4096, 16384, 16
    ct = b * d * L
    fw = bench.fwd_work(b, d, L, N)
    # u, delta, z in and out: 4 bf16 values per channel-token, plus B and C once per (b, t)
    assert fw["bytes"] == 8 * ct + 2 * N * 2 * b * L
    assert fw["fp32"] == ct * (6 * N + 3) and fw["sfu"] == ct * (N + 4)
    assert bench.fwd_ckpt_bytes(b, d, L, N) == 16 * ct          # N floats every 4 steps
    bw = bench.bwd_work(b, d, L, N)
    assert bw["bytes"] == 14 * ct + 16 * ct + 2 * N * 2 * b * L + 2 * N * 4 * b * L
    assert bench.conv_work(b, d, L)["bytes"] == 4 * ct
    assert bench.conv_bwd_work(b, d, L)["bytes"] == 6 * ct


def test_roofline_picks_the_slowest_unit_and_reports_the_fraction():
    saved = dict(bench.UNIT_RATES)
    try:
        bench.UNIT_RATES.update(fp32=128.0, ex2=32.0, source="nominal")
        sms, mhz, hbm = 148, 2000.0, 6000.0
        # FP32-bound work: 1e12 lane-ops at 148 * 128 * 2e9 per second
        w = dict(bytes=1e6, fp32=1e12, sfu=1e9)
        t_fp32 = 1e12 / (sms * 128 * mhz * 1e6)
        r = bench.roofline(w, 2 * t_fp32, hbm, sms, mhz, "measured", "sampled")
        assert r["bound"] == "alu" and r["unit"] == "TFP32op/s"
        assert r["frac"] == pytest.approx(0.5, rel=1e-3)
        # HBM-bound work
        w = dict(bytes=6e12, fp32=1e6, sfu=1e6)
        r = bench.roofline(w, 4.0, hbm, sms, mhz, "measured", "sampled")
        assert r["bound"] == "hbm" and r["achieved"] == pytest.approx(1500.0) and r["frac"] == pytest.approx(0.25)
    finally:
        bench.UNIT_RATES.clear()
        bench.UNIT_RATES.update(saved)


def test_traffic_is_scaled_and_tied_to_the_sources(monkeypatch):
    ct = 8 * 4096 * 16384
    monkeypatch.setattr(bench, "TRAFFIC_SOURCES_SHA", bench.kernel_sources_sha())
    t = bench.traffic_bytes("ssm_scan_bwd", ct)
    assert t == int(bench.TRAFFIC_PER_CT["ssm_scan_bwd"] * ct)
    assert bench.traffic_bytes("ssm_scan_bwd", 2 * ct) == pytest.approx(2 * t, rel=1e-9, abs=2)
    monkeypatch.setattr(bench, "TRAFFIC_SOURCES_SHA", "0" * 16)
    assert bench.traffic_bytes("ssm_scan_bwd", ct) is None
    assert bench.traffic_bytes("not_a_kernel", ct) is None


def test_unit_rates_from_the_probe_and_the_nominal_fallback():
    saved = dict(bench.UNIT_RATES)

    class Fake:
        def __init__(self, fail):
            self.fail = fail

        def probe_unit_rates(self):
            if self.fail:
                raise RuntimeError("no device")
            return {"fp32_lanes_per_sm_clock": 120.0, "f32x2_lanes_per_sm_clock": 124.0, "ex2_per_sm_clock": 30.0}

    try:
        out = bench.measure_unit_rates(Fake(fail=True))
        assert "error" in out and bench.UNIT_RATES["source"] == "nominal"
        out = bench.measure_unit_rates(Fake(fail=False))
        assert out["ex2_per_sm_clock"] == 30.0
        assert bench.UNIT_RATES["fp32"] == 124.0 and bench.UNIT_RATES["ex2"] == 30.0
        assert bench.UNIT_RATES["source"].startswith("measured")
    finally:
        bench.UNIT_RATES.clear()
        bench.UNIT_RATES.update(saved)


def _chunk_products(b, T, H, P, N, Q, shapes):
    """FLOPs of products (m, n, k) per chunk, summed over every (b, h, chunk) of full blocks."""
    chunks = b * H * (T // Q)
    return chunks * sum(2 * m * n * k for m, n, k in shapes)


def test_ssd_work_counts_the_chunked_products():
    cfg = dict(bench.SSD)
    b, T, H, P, N, G, Q = (cfg[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate", "ngroups", "chunk"))
    # C B^T (Q x Q, k N), M x (Q x P, k Q), C H (Q x P, k N), state update B^T (w x) (N x P, k Q)
    assert bench.ssd_work(cfg)["flops"] == _chunk_products(b, T, H, P, N, Q,
                                                           [(Q, Q, N), (Q, P, Q), (Q, P, N), (N, P, Q)])
    assert bench.ssd_work(cfg)["bytes"] == 346_554_368                 # x, dt, y, B, C at the 2.7B shape


def test_ssd_bwd_work_counts_the_chunked_adjoint_products():
    cfg = dict(bench.SSD)
    b, T, H, P, N = (cfg[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate"))
    Q = 64
    shapes = [(Q, Q, N),                     # C B^T
              (Q, Q, P),                     # dY X^T
              (Q, P, Q),                     # Z = K^T dY
              (Q, P, N),                     # B G
              (Q, N, Q), (Q, N, P),          # dC: intra, state
              (Q, N, Q), (Q, N, P),          # dB: intra, state
              (N, P, Q), (N, P, Q)]          # the two state passes
    assert bench.ssd_bwd_work(cfg, Q)["flops"] == _chunk_products(b, T, H, P, N, Q, shapes)
    # x, dout, dx (bf16) and dt, ddt (bf16) per (b, t, h); B, C in bf16 and dB, dC in fp32 per (b, t)
    assert bench.ssd_bwd_work(cfg, Q)["bytes"] == b * T * (H * (3 * 2 * P + 2 * 2) + N * (2 * 2 + 2 * 4))
