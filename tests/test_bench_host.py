"""Host-side arithmetic of bench.py's roofline objects (no GPU): the
whole-evaluation roofline adds each stage's ideal time (algorithmic work over
its peak) and divides by the measured evaluation time."""
import math
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from body_forces_morton_b300 import workloads as W  # noqa: E402


def fake_result(n, pairs, m2l):
    return {"n": n, "stats": {"n_p2p_interactions": pairs + n, "n_m2l": m2l}, "stage_ms": {}}


def test_reduced_m2l_flop_count():
    # 155 contraction terms at p = 4 (2 flop each), 25 derivatives at ~10 flop, 6 traces at one add
    assert bench.m2l_flops_per_pair(4) == 2 * 155 + 10 * 25 + 6 == 566
    assert bench.m2l_flops_per_pair(0) == 2 + 10


def test_hbm_bytes_per_particle():
    f32 = bench.hbm_bytes_per_particle(4)
    f64 = bench.hbm_bytes_per_particle(8)
    assert sum(f32.values()) == 336
    assert sum(f64.values()) == 456
    assert f32["sort"] == f64["sort"] == 192  # the keys do not depend on the dtype


def test_eval_roofline_sums_the_stage_terms():
    w = W.WORKLOADS[4]
    res = fake_result(1 << 20, 1_274_776_446, 9_694_118)
    r = bench.eval_roofline(res, w, 2.45, 6500.0, "measured")
    t = r["terms_ms"]
    assert math.isclose(r["ideal_ms"], t["p2p_alu"] + t["m2l_alu"] + t["hbm"], rel_tol=1e-12)
    assert math.isclose(r["frac"], r["ideal_ms"] / 2.45, rel_tol=1e-12)
    # P2P: 20 flop per pair at 148 x 128 x 2 x 2.032e9 flop/s
    assert math.isclose(t["p2p_alu"], 1_274_776_446 * 20 / (148 * 128 * 2 * 2.032e9) * 1e3, rel_tol=1e-12)
    assert math.isclose(t["hbm"], 336 * (1 << 20) / 6.5e12 * 1e3, rel_tol=1e-12)
    assert 0.1 < r["frac"] < 0.3


def test_eval_roofline_fp64_peaks_follow_the_pipe():
    w = W.WORKLOADS[3]
    res = fake_result(100_000, 48_723_340, 1_000_000)
    # double-float stages run on the FP32 pipe
    r = bench.eval_roofline(res, w, 2.14, 6500.0, "measured")
    assert r["peaks"]["alu_tflops"] == bench.FP32_PEAK_TFLOPS
    # IEEE fp64: the FP64 pipe, 148 SMs x 2 FMA per clock x 2 flop x 2.032 GHz
    r = bench.eval_roofline(res, w, 2.14, 6500.0, "measured", dtype="f64", f64_ieee=True)
    assert math.isclose(r["peaks"]["alu_tflops"], 148 * 2 * 2 * 2.032e9 / 1e12, rel_tol=1e-12)
    assert math.isclose(r["terms_ms"]["p2p_alu"], 48_723_340 * 20 / (148 * 4 * 2.032e9) * 1e3, rel_tol=1e-12)


def test_df_roofline_uses_the_fp32_pipe_and_counted_operations():
    res = {"n": 100_000, "stats": {"n_p2p_interactions": 48_823_340, "n_m2l": 1_833_964},
           "stage_ms": {"p2p": 0.5, "m2l": 0.4}}
    w = W.WORKLOADS[3]
    key = ("k_p2p_df", bench.kernel_source_hash(bench.DF_SOURCES["k_p2p_df"]))
    saved = dict(bench.DF_FMA_OPS_PER_PAIR)
    try:
        bench.DF_FMA_OPS_PER_PAIR.clear()
        r = bench.p2p_roofline(res, w)
        assert r["frac"] is None and r["unit"] == "FP32 lane-ops/s"
        bench.DF_FMA_OPS_PER_PAIR[key] = 100.0
        r = bench.p2p_roofline(res, w)
        assert math.isclose(r["achieved"], 100.0 * 48_723_340 / 0.5e-3, rel_tol=1e-12)
        assert math.isclose(r["frac"], r["achieved"] / (148 * 128 * 2.032e9), rel_tol=1e-12)
        assert math.isclose(r["fp64_equivalent_tflops"], 20 * 48_723_340 / 0.5e-3 / 1e12, rel_tol=1e-12)
    finally:
        bench.DF_FMA_OPS_PER_PAIR.clear()
        bench.DF_FMA_OPS_PER_PAIR.update(saved)


def test_hbm_peak_reads_the_measured_file():
    v, src = bench.hbm_peak_gbs()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert src == "measured" and v > 1000
    else:
        assert (v, src) == (6400.0, "fallback")
