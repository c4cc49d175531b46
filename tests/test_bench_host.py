"""Host-side arithmetic of the benchmark (no GPU): the algorithmic work it
divides by each stage's time, the roofline fractions, the committed traffic
figure it reports, the clock-record parsing and the workload description.
The counts are the ones the kernels' rooflines are stated in: a
multiply-add is two flops, a symmetric Gram counts its distinct entries, the
inversions count a factorisation of the t x t system (t^3 / 3)."""
import os

import numpy as np
import pytest

import bench
from workloads import WORKLOADS, budgets


def test_stage_work_of_the_32_layer_cache():
    w = WORKLOADS[3]
    b = budgets(w)
    work = bench.stage_work(w, b)
    H, n, T, d, t = w.H, w.n, w.T, w.d, 655
    assert np.all(b == t) and len(b) == H == 256
    assert work["attn_fwd"] == ("flops", 4.0 * n * T * d * H)          # Q K^T and P V
    assert work["colscore"] == ("flops", 2.0 * n * T * d * H)          # K Q^T again
    assert work["masslogits"] == ("flops", 2.0 * n * d * t * H)
    assert work["gram_a"] == ("flops", float(H * n * t * (t + 1)))     # distinct entries of A'^T A'
    assert work["xto"] == ("flops", 2.0 * n * d * t * H)
    assert work["inv_h"][1] == pytest.approx(H * t ** 3 / 3.0)
    assert work["apply_minv"][1] == pytest.approx(H * 2.0 * t * t * d)
    assert work["v_f16"] == ("bytes", 4.0 * T * d * H)                  # bf16 read, fp16 written


def test_stage_work_sums_nonuniform_budgets():
    w = WORKLOADS[4]
    b = budgets(w)
    work = bench.stage_work(w, b)
    assert work["inv_m"][1] == pytest.approx(sum(float(x) ** 3 / 3.0 for x in b))
    assert work["gram_x"][1] == pytest.approx(sum(w.n * float(x) * (x + 1) for x in b))


def test_roofline_fractions():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 1500.0, "bf16_tflops_sustained": 1300.0}
    r = bench.roofline_for("v_f16", 1.0, ("bytes", 3.0e9), peaks, "measured", None)
    assert r["bound"] == "hbm" and r["achieved"] == pytest.approx(3000.0) and r["frac"] == pytest.approx(0.5)
    bench.TENSOR_STAGES.clear()
    bench.TENSOR_STAGES.update({"attn_fwd"})
    try:
        r = bench.roofline_for("attn_fwd", 2.0, ("flops", 1.5e12), peaks, "measured", 123)
        assert r["bound"] == "tensor" and r["achieved"] == pytest.approx(750.0)
        assert r["frac"] == pytest.approx(0.5) and r["traffic"] == 123 and r["peak"] == 1500.0
        r = bench.roofline_for("inv_h", 1.0, ("flops", 1.0e10), peaks, "measured", None)
        assert r["bound"] == "alu" and r["achieved"] == pytest.approx(10.0)
        assert r["frac"] == pytest.approx(10.0 / bench.SIMT_F32_PEAK_TFLOPS, abs=1e-4)
    finally:
        bench.TENSOR_STAGES.clear()


def test_tensor_stages_follow_the_input_type():
    assert {"attn_fwd", "colscore", "masslogits", "gram_a"} <= bench.tensor_stages(WORKLOADS[3])
    fp32 = bench.tensor_stages(WORKLOADS[1])
    assert "attn_fwd" not in fp32 and "gram_a" in fp32


def test_committed_traffic_is_read_for_its_stage_only():
    path = os.path.join(bench.ROOT, "profiles", "traffic_attn_fwd_llama3-8b-32layer-cache-T32768.txt")
    with open(path) as fh:
        rows = [ln.split() for ln in fh if not ln.startswith("#") and ln.strip()]
    assert rows == [["attn_fwd", "config3", str(bench._traffic_for("attn_fwd", 3))]]
    assert bench._traffic_for("colscore", 3) is None
    assert bench._traffic_for("attn_fwd", 2) is None


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_record_parsing():
    s = bench.ClockSampler(0)
    s.proc = _Done()
    s.lines = [
        "0, 1950, 2032, 905.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1940, 2032, 910.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2032, 2032, 400.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbled line",
    ]
    rec = s.stop()
    assert rec["sm_mhz"] == 1950.0 and rec["sm_max_mhz"] == 2032.0
    assert rec["reasons"] == ["sw_power_cap"] and rec["samples"] == 3
    assert bench.ClockSampler(0).stop()["reasons"] == ["nvidia-smi unavailable"]


def test_workload_description_names_the_config():
    w = WORKLOADS[3]
    c = bench.config_dict(w, budgets(w), 1)
    assert c["workload"] == "llama3-8b-32layer-cache-T32768" and c["heads_per_gpu"] == 256 and c["t"] == 655
    w4 = WORKLOADS[4]
    assert str(bench.config_dict(w4, budgets(w4), 1)["t"]).startswith("nonuniform mean 1638.4")
    two = bench.limit_layers(w, 2)
    assert two.H == 16 and two.name.endswith("first2layers")
    assert bench.rank_workload(w, 1, 2).seq_offset != w.seq_offset
