"""Host-side accounting of bench.py (no GPU): the per-group roofline of the grouped products
and the algorithmic work per phase, against values worked out by hand."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

PEAKS = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0, "bf16_tflops_sustained": 100.0, "source": "test"}
CFG = {"T": 64, "d": 128, "E": 2, "k": 2, "f": 64, "S": 1, "f_s": 64, "dtype": "bf16"}


def test_group_roofline_by_hand():
    # P = 1e14 flop/s, BW = 1e12 B/s. FWD1 of a group with n rows and width w:
    # flops 4 d w n, bytes 2 d w 2 + 2 n (d + 3 w).
    counts = [100, 28]
    r = bench.group_roofline(CFG, counts, PEAKS)
    d, w, T = 128, 64, 64

    def fwd1(n):
        return max(4.0 * d * w * n / 1e14, (2 * d * w * 2 + 2 * n * (d + 3 * w)) / 1e12)

    want = sum(fwd1(n) for n in counts + [T]) * 1e3
    assert r["gemm_fwd1"]["per_group_ms"] == pytest.approx(want, rel=1e-12)
    # every group here is below the ridge (n < P / BW = 100 flop per byte at these sizes),
    # so the per-group bound is the byte total
    by = sum(2 * d * w * 2 + 2 * n * (d + 3 * w) for n in counts + [T])
    assert r["gemm_fwd1"]["bytes"] == by
    assert r["gemm_fwd1"]["whole_launch_ms"] == pytest.approx(by / 1e12 * 1e3, rel=1e-12)


def test_group_roofline_bounds_ordered():
    # the whole-launch bound never exceeds the per-group one (max of sums <= sum of maxes)
    for counts in ([0, 128], [4000, 1], [7, 7]):
        r = bench.group_roofline(CFG, counts, PEAKS)
        for ph, v in r.items():
            assert v["whole_launch_ms"] <= v["per_group_ms"] * (1 + 1e-12), ph


def test_group_roofline_compute_bound_group():
    # one huge group: compute-bound, so its term is its flops over P
    counts = [10 ** 6, 0]
    r = bench.group_roofline(CFG, counts, PEAKS)
    d, w = 128, 64
    n = 10 ** 6
    dw13 = 4.0 * d * w * n / 1e14
    assert r["gemm_dw13"]["per_group_ms"] >= dw13 * 1e3


def test_algorithmic_work_totals():
    flops, bytes_ = bench.algorithmic_work(CFG)
    T, d, k, f, S, fs = 64, 128, 2, 64, 1, 64
    rows_f = T * k * f + S * T * fs
    assert flops["gemm_fwd1"] == 4.0 * d * rows_f
    assert flops["gemm_dw2"] == 2.0 * d * rows_f
    assert bytes_["permute_scatter"] == (1 + k) * T * d * 2 + 24.0 * T * k
    assert bytes_["combine"] == (k + 2) * T * d * 2 + 8.0 * T * k


def test_dw_write_bytes():
    w = bench.dw_write_bytes(CFG)
    assert w["gemm_dw13"] == 2 * (2 * 64 * 128 * 2 + 2 * 64 * 128 * 1)
    assert w["gemm_dw2"] == w["gemm_dw13"] // 2


def test_oracle_scale_keeps_twice_k_experts():
    assert bench.oracle_scale({"E": 256, "k": 8}) == 16       # 16 experts, 256 copies each
    assert bench.oracle_scale({"E": 64, "k": 6}) == 4         # 16 >= 12 experts
    assert bench.oracle_scale({"E": 8, "k": 2}) == 2
    assert bench.oracle_scale({"E": 2, "k": 2}) == 1


def test_oracle_sample_runs_a_sub_layer_on_cpu():
    import numpy as np
    import oracle as O
    from synth import make_workload, shrink
    w = make_workload(shrink("pangu_bf16", T=64, d=64, E=32, k=4, f=64, f_s=64))
    s = bench.oracle_scale(w.cfg)
    assert s == 4
    logits32 = O.router_logits(O.as_f64(w.x), O.as_f64(w.w_r)).astype(np.float32)
    dt, Ts, Es = bench.oracle_sample(w, logits32, s)
    assert (Ts, Es) == (16, 8) and dt > 0
    text = bench.sample_text(w.cfg, s, Ts, Es)
    assert "16 tokens" in text and "8 of its 32 experts" in text and "8 copies per expert" in text


def test_summarize_grouped_totals_and_dominant():
    steps = 2
    trace = {"gemm_fwd1": (2, 8.0), "gemm_dw13": (2, 10.0), "combine": (2, 1.0)}
    counts = [100, 28]
    r = bench.summarize(CFG, trace, steps, counts, PEAKS)
    flops, bytes_ = bench.algorithmic_work(CFG)
    assert r["dominant"] == "gemm_dw13" and r["launches"] == 6
    tf = (flops["gemm_fwd1"] + flops["gemm_dw13"]) / (9.0 / 1e3) / 1e12
    assert r["grouped_gemm"]["tflops"] == pytest.approx(tf, abs=0.06)
    assert r["grouped_gemm"]["frac_of_burst_peak"] == pytest.approx(tf / 100.0, abs=1e-3)
    assert r["kernels"]["combine"]["unit"] == "GB/s"
    # executed rows: 100 in a 128-row tile, 28 and 64 in 64-row tiles; all in 128-row tiles: 384
    assert r["routing"]["m_tile_fill"] == pytest.approx(192 / 256, abs=1e-4)
    assert r["routing"]["m_tile_fill_128"] == pytest.approx(192 / 384, abs=1e-4)
    assert [bench.executed_rows(c) for c in (0, 1, 64, 65, 128, 129, 192, 193)] == [0, 64, 64, 128, 128, 192, 192, 256]
