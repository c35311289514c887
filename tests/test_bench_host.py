"""Host-side checks of bench.py: the algorithmic byte and flop formulas behind every roofline
fraction, the per-workload traffic table (dropped once the kernel changes), and the JSON line of the reference (oracle) arm."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


# drafter shape: G = 16 rows per block, H = 5120, group 16 (320 groups), V = 248320, R = 64, K = 16
G, H, GROUPS, V, R, K = 16, 5120, 320, 248320, 64, 16


def test_head_flops_count_every_multiply_add_once():
    # 960 rows (64 blocks x 15 draft rows) against the vocabulary and the 64 projection rows
    assert bench.head_flops(960, V, R, H) == 2 * 960 * (V + R) * H
    assert bench.head_flops(960, V, R, H) == pytest.approx(2.4417e12, rel=1e-4)


def test_head_bytes_are_the_weight_stream_plus_rows_and_outputs():
    b = bench.head_bytes(15, V, R, H, K)
    weights = 2 * (V + R) * H  # bf16 head weight and hidden projection, read once
    assert weights == 2_543_452_160
    # the rows, the bias and the outputs (16 ids + 16 values and z per row) on top of the weights
    assert b - weights == 2 * 15 * H + 4 * V + 15 * (8 * K + 4 * R)


def test_prepare_and_finish_bytes_at_64_blocks():
    rows = 64 * G
    # prepare: normed rows in, W_kp in, side-0 output out, side-1 coefficients out (all bf16)
    assert bench.prepare_call_bytes(rows, H, GROUPS) == 35_389_440
    # finish with the next norm: y, residual, coefficients in; x and the normed rows out;
    # the fp32 base kernel's side-1 taps and the bf16 norm weight
    assert bench.finish_call_bytes(rows, H, GROUPS, rows) == 43_304_960


def test_edge_score_bytes_per_slot():
    per_slot = bench.edges_call_bytes(1, 1, K, R)
    # cand and unary (K each, 4 bytes), z (R floats), 2K gathered bf16 codebook rows, S (K x K
    # floats) and one path entry
    assert per_slot == 4 * K + 4 * K + 4 * R + 2 * K * R * 2 + 4 * K * K + 4
    assert bench.edges_call_bytes(64, 15, K, R) == 64 * 15 * per_slot


def test_traffic_table_names_only_known_workloads_and_is_dropped_when_the_kernel_changes():
    assert set(bench.HEAD_TRAFFIC) <= set(bench.WORKLOADS)
    for name, t in bench.HEAD_TRAFFIC.items():
        # every measured launch read at least the head weight once
        assert t["bytes"] >= 2 * (V + R) * H, name
        assert t["date"] and len(t["gemm_sha"]) == 16
    saved = dict(bench.HEAD_TRAFFIC)
    try:
        bench.HEAD_TRAFFIC["full-tail-B64"] = {"bytes": 3e9, "date": "then", "gemm_sha": "0" * 16}
        assert bench.head_traffic("full-tail-B64")["traffic"] is None
        bench.HEAD_TRAFFIC["full-tail-B64"]["gemm_sha"] = bench.kernel_source_sha("gemm.cu")
        assert bench.head_traffic("full-tail-B64")["traffic"] == 3e9
    finally:
        bench.HEAD_TRAFFIC.clear()
        bench.HEAD_TRAFFIC.update(saved)


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "conv-chain-B1",
                          "--steps", "1", "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["unit"] == "blocks/s" and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["n_gpus"] == 1 and line["value"] > 0
    assert line["config"]["workload"] == "conv-chain-B1"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
