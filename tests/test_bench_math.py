"""The bench's algorithmic work and roofline arithmetic, host only: the bytes
and flops that every reported GB/s, TFLOP/s and roofline fraction divides
by, checked against values worked out by hand from the shard shapes."""

import numpy as np
import pytest

import bench
from w4a16_int4_moe_gb300 import workloads as wl

B_W = 0.5 + 2.0 / 32          # uint4 code + a BF16 scale per 32 elements


def test_weight_bytes_per_element():
    assert bench.WEIGHT_BYTES == pytest.approx(0.5625)


def test_ep8_decode_work():
    p = wl.ep8_decode(weights=False)
    w = bench.algorithmic_work(p)
    assert w["active_experts"] == 48 and w["rows"] == 576
    # 48 experts x gate_up [4096 x 7168]: 792.7 MB of weights
    gu_weights = 48 * 4096 * 7168 * B_W
    assert gu_weights == pytest.approx(792.72e6, rel=1e-4)
    used = int(np.any(p.topk_ids >= 0, axis=1).sum())
    assert w["gate_up"]["bytes"] == pytest.approx(gu_weights + used * 7168 * 2 + 576 * 4096 * 2)
    # down: 48 x [7168 x 2048] weights, the 576 activation rows, the FP32 output once
    assert w["down"]["bytes"] == pytest.approx(48 * 7168 * 2048 * B_W + 576 * 2048 * 2
                                               + 576 * 7168 * 4)
    # 2 * rows * n * k per GEMM: 33.8 + 16.9 GF
    assert w["gate_up"]["flops"] == pytest.approx(2 * 576 * 4096 * 7168)
    assert w["down"]["flops"] == pytest.approx(2 * 576 * 7168 * 2048)
    assert (w["gate_up"]["flops"] + w["down"]["flops"]) / 1e9 == pytest.approx(50.7, abs=0.05)


def test_ep8_prefill_work():
    p = wl.ep8_prefill(weights=False)
    w = bench.algorithmic_work(p)
    assert w["rows"] == 3904 and w["active_experts"] == 48
    total = w["gate_up"]["flops"] + w["down"]["flops"]
    assert total == pytest.approx(2 * 3904 * (4096 * 7168 + 7168 * 2048))
    assert total / 1e9 == pytest.approx(344.0, abs=0.5)


def test_tp8_work_counts_only_experts_with_rows():
    p = wl.tp8(16, weights=False)
    w = bench.algorithmic_work(p)
    active = np.unique(p.topk_ids[p.topk_ids >= 0]).size
    assert w["active_experts"] == active < 384
    assert w["gate_up"]["bytes"] >= active * 512 * 7168 * B_W
    assert w["rows"] == 16 * 8


def test_grouped_work():
    # contiguous, 128 rows for each of 48 experts: 6144 rows
    w = bench.grouped_work(6144, 48)
    assert w["gate_up"]["flops"] + w["down"]["flops"] == 2 * 6144 * 44040192   # 4096*7168 + 7168*2048
    assert (w["gate_up"]["flops"] + w["down"]["flops"]) / 1e9 == pytest.approx(541.17, abs=0.01)
    # masked, budget 32: all 48 experts' weights (1.189 GB) plus the rows in and out
    counts = wl.masked_counts(48, 32, seed=1)
    rows = int(counts.sum())
    w = bench.grouped_work(rows, 48)
    weights = 48 * (4096 * 7168 + 7168 * 2048) * B_W
    assert weights / 1e9 == pytest.approx(1.189, abs=0.001)
    assert w["gate_up"]["bytes"] + w["down"]["bytes"] == pytest.approx(
        weights + rows * (7168 + 4096) * 2 + rows * (2048 + 7168) * 2)


def test_roofline_entry_fractions():
    r = bench.roofline_entry("hbm", "k", 3400.0, 6800.0, 8000.0, "measured hbm_gbs",
                             {"traffic": None})
    assert r["unit"] == "GB/s" and r["frac"] == pytest.approx(0.5)
    assert r["frac_of_nominal"] == pytest.approx(0.425)
    assert r["traffic"] is None
    t = bench.roofline_entry("tensor", "k", 950.0, 1900.0, 2250.0, "measured bf16_tflops")
    assert t["unit"] == "TFLOP/s" and t["frac"] == pytest.approx(0.5)
