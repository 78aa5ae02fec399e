"""Host logic of the benchmark (CPU): the captured-traffic figure is reported
only for the GEMM sources it was captured on, the roofline object's
arithmetic (achieved = FLOP / time, the burst peak for short timed regions
and the sustained one for long ones, twice the BF16 peak for MXFP8, the HBM
bound when weights dominate), and the clock record's choice of samples."""
import types

import pytest

import bench
from combine_router_top_expert_gb300 import mok, synth


def _args(**kw):
    d = dict(gemm_pairs=False, swapped_tiles=False, single_cta=False)
    d.update(kw)
    return types.SimpleNamespace(**d)


def _m(wl, dtype, gemm_ms, total_ms):
    return dict(wl=wl, dtype=dtype, flops=6.0 * wl.H * wl.I * wl.T * wl.k, gemm_ms=gemm_ms,
                rank_total_ms=total_ms, staged=True, batches=1, kern="gemm pair")


def test_captured_traffic_follows_the_gemm_sources(monkeypatch):
    sha = bench.gemm_sources_sha1()
    monkeypatch.setattr(bench, "GEMM_PAIR_TRAFFIC", {"w": {"bytes": 123.0, "gemm_sources_sha1": sha}})
    assert bench.captured_traffic("w") == (123.0, "ncu capture on GEMM sources " + sha)
    monkeypatch.setattr(bench, "GEMM_PAIR_TRAFFIC", {"w": {"bytes": 123.0, "gemm_sources_sha1": "0" * 16}})
    b, why = bench.captured_traffic("w")
    assert b is None and why.startswith("stale")
    assert bench.captured_traffic("other")[0] is None


def test_roofline_tensor_bound_burst_and_sustained(monkeypatch):
    monkeypatch.setattr(bench, "load_peaks", lambda: dict(hbm=6000.0, bf16=2000.0, bf16_sus=1600.0, source="t"))
    wl = synth.WORKLOADS["bf16_fwd_T2560"]
    m = _m(wl, mok.BF16, [1.0, 1.0], 100.0)
    r = bench.roofline(m, _args())
    assert r["bound"] == "tensor"
    assert r["achieved"] == pytest.approx(m["flops"] / 1e-3 / 1e12)
    assert r["peak"] == 2000.0 and r["frac"] == pytest.approx(r["achieved"] / 2000.0)
    assert "burst" in r["peak_source"]
    r2 = bench.roofline(_m(wl, mok.BF16, [1.0], 5000.0), _args())
    assert r2["peak"] == 1600.0 and "sustained" in r2["peak_source"]
    # traffic only for the default stage kernels
    assert bench.roofline(m, _args(single_cta=True))["traffic"] is None


def test_roofline_mxfp8_peak_and_hbm_bound(monkeypatch):
    monkeypatch.setattr(bench, "load_peaks", lambda: dict(hbm=6000.0, bf16=2000.0, bf16_sus=1600.0, source="t"))
    wl = synth.WORKLOADS["mxfp8_zipf_T2560"]
    r = bench.roofline(_m(wl, mok.MXFP8, [1.0], 100.0), _args())
    assert r["peak"] == 4000.0 and "x2" in r["peak_source"]
    # 512 tokens: the 1.45 GB of E4M3 weights take longer at the HBM rate than the FLOPs at the FP8 rate
    small = synth.WORKLOADS["mxfp8_zipf_T512"]
    r3 = bench.roofline(_m(small, mok.MXFP8, [0.3], 100.0), _args())
    assert r3["bound"] == "hbm" and r3["unit"] == "GB/s"
    assert r3["frac"] == pytest.approx(r3["bytes_per_step"] / 0.3e-3 / 1e9 / 6000.0)


def test_clock_record_summarises_the_timed_region():
    """Samples stamped inside the timed region decide the clock record; the
    utilisation filter and then all samples are the fallbacks."""
    import datetime
    import bench

    def line(t, mhz, util, power_cap):
        ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        cap = "Active" if power_cap else "Not Active"
        return (f"{ts}, 0, {mhz}, 2070, 500.0, {util}, 0x0, Not Active, Not Active, Not Active, {cap}")
    t0 = 1_800_000_000.0
    lines = [line(t0 + 0.00, 2070, 0, False),     # warm-up, before the window
             line(t0 + 0.10, 1700, 10, True),     # inside the window (utilisation still lagging)
             line(t0 + 0.12, 1650, 20, True),
             line(t0 + 0.30, 2070, 90, False)]    # after it
    r = bench.ClockSampler.summarise(lines, (t0 + 0.05, t0 + 0.20))
    assert r["samples"] == 4 and r["samples_in_timed_region"] == 2 and r["summarised"] == "timed region"
    assert r["sm_mhz"] == 1675.0 and r["sm_max_mhz"] == 2070.0 and r["reasons"] == ["sw_power_cap"]
    r = bench.ClockSampler.summarise(lines, (t0 + 0.50, t0 + 0.60))   # no sample inside
    assert r["summarised"] == "under load" and r["sm_mhz"] == 2070.0 and r["reasons"] == []
    r = bench.ClockSampler.summarise(lines[:3])
    assert r["summarised"] == "all samples" and r["samples_in_timed_region"] == 0
    assert bench.ClockSampler.summarise([]) is None
