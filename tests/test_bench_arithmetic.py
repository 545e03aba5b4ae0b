"""The benchmark's roofline arithmetic and step bookkeeping, on the CPU.

The per-sample figures are the ones worked out by hand from the method's block geometry (step 2
of the claim: N = L + M - 1; an output sample costs the s bytes of its input, the (M-1)/L overlap
re-read and the s bytes of its store; the transforms cost 2 * 5 N log2 N + 6 N flops per block of
L outputs, halved for pair-packed real data), not retyped from bench.py's formulas.
"""
import io
import json
import math
from contextlib import redirect_stdout

import pytest

import bench
import workloads as W

# (bytes per output sample, nominal flops per output sample), to the precision printed in the
# workload table the measurement plan was written against
HAND = {"C1": (18.61, 114.1), "C2": (18.66, 167.9), "C3": (18.67, 208.0), "C4": (9.32, 70.5),
        "C5": (18.67, 221.3)}


@pytest.mark.parametrize("name", sorted(HAND))
def test_bytes_and_flops_per_output(name):
    w = W.WORKLOADS[name]
    b, f = HAND[name]
    assert bench.bytes_per_output(w) == pytest.approx(b, abs=0.006)
    assert bench.flops_per_output(w) == pytest.approx(f, abs=0.06)


def test_c5_bounds_order():
    # at the measured 6689.1 GB/s and a 77.5 TFLOP/s FP32 peak, C5's flop bound is the slower one
    w = W.WORKLOADS["C5"]
    t_hbm = w.n * bench.bytes_per_output(w) / 6689.1e9
    t_fp32 = w.n * bench.flops_per_output(w) / 77.5e12
    assert t_fp32 > t_hbm
    assert t_hbm * 1e6 == pytest.approx(281, abs=1)
    assert t_fp32 * 1e6 == pytest.approx(287.5, abs=1)


def test_roofline_block_picks_the_slower_bound():
    r = bench.roofline_block(achieved_gbs=3000.0, peak_gbs=6000.0, peak_kind="measured", traffic=None,
                             bytes_launch=1e9, flops_launch=2e10, launch_ms=1.0, fp32_peak=80.0,
                             t_hbm=1e9 / 6000e9, t_fp32=2e10 / 80e12)
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(20.0) and r["frac"] == pytest.approx(0.25)
    assert r["hbm_frac"] == pytest.approx(0.5)
    r = bench.roofline_block(achieved_gbs=3000.0, peak_gbs=6000.0, peak_kind="measured", traffic=123.0,
                             bytes_launch=1e9, flops_launch=1e9, launch_ms=1.0, fp32_peak=80.0,
                             t_hbm=1e9 / 6000e9, t_fp32=1e9 / 80e12)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["frac"] == pytest.approx(0.5)
    assert r["traffic"] == 123.0


@pytest.mark.parametrize("per_set", [1 << 20, 50 << 20, 403 << 20, 3 << 30])
def test_buffer_sets_exceed_l2(per_set):
    sets = bench.buffer_sets(per_set)
    assert 2 <= sets <= 1024
    assert sets * per_set >= 1.25 * bench.L2_BYTES or sets == 1024


@pytest.mark.parametrize("sets,launches,K", [(2, 1, 20), (836, 1, 2000), (2, 64, 20), (32, 2, 7)])
def test_graph_replays_cover_exactly_k_steps(sets, launches, K):
    R = bench.steps_per_graph(sets, launches)
    assert R % sets == 0 and R >= sets
    runs = bench.graph_replays(K, R)
    assert sum(runs) == K and all(0 < n <= R for n in runs)


def test_shortened_workload():
    w = bench.workload("C5", 512)
    assert w.n == 512 * w.L and "shortened to k=512" in w.description
    assert bench.workload("C4", 10).n == W.WORKLOADS["C4"].n  # multi-call workloads stay whole


def test_reference_arm_prints_one_line():
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--config", "C1", "--steps", "3", "--warmup", "3"])
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GS/s"
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and math.isfinite(d["ms_per_step"])
