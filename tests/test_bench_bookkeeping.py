"""The benchmark's bookkeeping on CPU: the algorithmic work it credits per step, the
roofline it reports for the dominant kernel, and the peaks it divides by. These numbers
are what the JSON line's fractions rest on, so they are checked against closed forms."""
import json
import os

import numpy as np
import pytest

import bench
import moe_inputs as mi


class _LI:
    def __init__(self, wl):
        self.wl = wl


def test_algorithmic_work_prefill_closed_form():
    wl = mi.QWEN3_PREFILL
    M, K, N, topk, E = wl.M, wl.K, wl.N, wl.topk, wl.E
    # every slot kept (no expert map): R = M * topk, spread over all experts
    counts = [np.full(E, M * topk // E, np.int64)]
    a = bench.algorithmic(_LI(wl), counts)
    R = M * topk
    assert a["R"] == R == 65536
    assert a["gemm1_flops"] == pytest.approx(4.12e11, rel=1e-3)      # 2 R (2N) K
    assert a["gemm2_flops"] == pytest.approx(2.06e11, rel=1e-3)      # 2 R K N
    assert a["gemm1_flops"] == 2 * a["gemm2_flops"]
    assert a["scatter_bytes"] == 2 * M * K + R * K + R * (K // 128) * 4 + 8 * M * topk
    assert a["gather_bytes"] == 2 * R * K + 2 * M * K + 8 * M * topk
    # weights: each touched expert's w13 + w2 codes (3NK bytes) and their fp32 block scales
    per_expert = 3 * N * K + (2 * N // 128) * (K // 128) * 4 + (K // 128) * (N // 128) * 4
    assert a["weight_bytes"] == E * per_expert


def test_algorithmic_work_counts_only_kept_rows_and_touched_experts():
    wl = mi.QWEN3_CHUNKED
    c1 = np.zeros(wl.El, np.int64)
    c1[[0, 5, 9]] = [3, 1, 100]
    c2 = np.zeros(wl.El, np.int64)
    c2[[5]] = [7]
    a = bench.algorithmic(_LI(wl), [c1, c2])
    assert a["R"] == 111
    assert a["gemm2_flops"] == 2.0 * 111 * wl.K * wl.N
    per_expert = a["weight_bytes"] / 4  # 3 experts touched in chunk 1, 1 in chunk 2
    assert per_expert == 3 * wl.N * wl.K + (2 * wl.N // 128) * (wl.K // 128) * 4 + (wl.K // 128) * (wl.N // 128) * 4


def _kern(us):
    t = {k: {"us_per_step": v, "launches_per_step": 1} for k, v in us.items()}
    return {"table": t}


def test_roofline_reports_the_dominant_kernel_against_the_right_peak():
    wl = mi.QWEN3_PREFILL
    counts = [np.full(wl.E, wl.M * wl.topk // wl.E, np.int64)]
    work = bench.algorithmic(_LI(wl), counts)
    pk = {"hbm": 6800.0, "bf16": 1900.0, "src": "test"}
    kern = _kern({"scatter": 40.0, "gemm1": 240.0, "gemm2": 150.0, "gather": 50.0})
    roof = bench.roofline(kern, work, pk, wl)
    assert roof["kernel"] == "gemm1" and roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert roof["peak"] == pytest.approx(3800.0)                    # dense FP8 = 2 x bf16
    assert roof["achieved"] == pytest.approx(work["gemm1_flops"] / 240e-6 / 1e12, rel=1e-3)
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], rel=1e-3)
    t = kern["table"]
    assert t["gather"]["GB/s"] == pytest.approx(work["gather_bytes"] / 50e-6 / 1e9, rel=1e-3)
    assert t["gather"]["hbm_frac"] == pytest.approx(t["gather"]["GB/s"] / 6800.0, rel=1e-3)
    # an HBM-bound workload reports GB/s against the copy bandwidth
    wl2 = mi.PERMUTE_ONLY
    work2 = bench.algorithmic(_LI(wl2), [np.full(wl2.E, wl2.M * wl2.topk // wl2.E, np.int64)])
    roof2 = bench.roofline(_kern({"scatter": 28.0, "gather": 30.0}), work2, pk, wl2)
    assert roof2["kernel"] == "gather" and roof2["bound"] == "hbm" and roof2["unit"] == "GB/s"
    assert roof2["peak"] == 6800.0
    assert roof2["frac"] == pytest.approx(work2["gather_bytes"] / 30e-6 / 1e9 / 6800.0, rel=1e-3)


def test_peaks_come_from_the_measured_file():
    pk = bench.peaks()
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        assert pk["src"] == "measured"
        assert pk["hbm"] == float(p["hbm_gbs"]) and pk["bf16"] == float(p["bf16_tflops"])
    else:
        assert pk["src"] == "fallback"


def test_recorded_traffic_matches_only_the_source_it_was_taken_on():
    wl = mi.QWEN3_PREFILL
    got = bench.recorded_traffic("gemm1", wl.name)
    with open(os.path.join(bench.PROFILES, "dram_traffic.json")) as f:
        rec = json.load(f)[wl.name]["gemm1"]
    if rec["src_sha"] == bench.src_hash(rec["src"]):
        assert got == float(rec["bytes_per_launch"])
    else:
        assert got is None
    assert bench.recorded_traffic("gemm1", "no_such_workload") is None
