"""bench.py's algorithmic work per phase and its roofline arithmetic, on the
CPU with hand-computed values (no GPU)."""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from dispatch_ffn_combine_gb300.workloads import CONFIGS  # noqa: E402

PEAKS = {"hbm_gbs": 6793.1, "bf16_tflops": 1939.5, "bf16_tflops_sustained": 1721.2, "source": "measured"}


def test_flops_bytes_large_hand_computed():
    cfg = CONFIGS["large"]  # T 32768, d 7168, E 256, k 8, f 2048
    offsets = np.arange(0, 257, dtype=np.int64) * 1024  # every expert touched, 1024 rows each
    fb = bench.flops_bytes(cfg, offsets)
    S = 32768 * 8
    assert fb["gemm1"]["flops"] == 4 * S * 7168 * 2048 == 15_393_162_788_864
    # W1 and W3 of 256 experts + x_perm read + h written
    assert fb["gemm1"]["bytes"] == 2 * 256 * 2048 * 7168 * 2 + S * 7168 * 2 + S * 2048 * 2
    assert fb["gemm2"]["flops"] == 2 * S * 7168 * 2048
    assert fb["layer"]["flops"] == 6 * S * 7168 * 2048
    assert fb["combine"] == {"flops": 0, "bytes": S * 7168 * 2 + 32768 * 7168 * 2}
    assert fb["touched_experts"] == 256


def test_flops_bytes_counts_only_touched_experts():
    cfg = CONFIGS["decode"]  # T 128, d 7168, E 256, k 8, f 2048
    counts = np.zeros(256, dtype=np.int64)
    counts[:128] = 8  # 128 experts hold all 1024 rows
    offsets = np.concatenate([[0], np.cumsum(counts)])
    fb = bench.flops_bytes(cfg, offsets)
    assert fb["touched_experts"] == 128
    assert fb["gemm1"]["bytes"] == 2 * 128 * 2048 * 7168 * 2 + 1024 * 7168 * 2 + 1024 * 2048 * 2


def test_roofline_tensor_bound_with_hbm_beside():
    work = {"flops": 15.4e12, "bytes": 20.0e9}  # 770 FLOP/B, above the ridge (253 FLOP/B)
    r = bench.roofline(work, 9.0, PEAKS)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 1939.5
    assert r["achieved"] == pytest.approx(15.4e12 / 9.0e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 1939.5)
    assert r["sustained"]["frac"] == pytest.approx(r["achieved"] / 1721.2)
    assert r["other"]["bound"] == "hbm"
    assert r["other"]["achieved"] == pytest.approx(20.0e9 / 9.0e-3 / 1e9)
    assert r["other"]["frac"] == pytest.approx(r["other"]["achieved"] / 6793.1)
    assert r["peak_source"].endswith("(bf16 burst)")


def test_roofline_hbm_bound_and_copy_kernels():
    r = bench.roofline({"flops": 60e9, "bytes": 14.9e9}, 2.14, PEAKS)  # decode's gemm1: 4 FLOP/B
    assert r["bound"] == "hbm" and r["frac"] == pytest.approx(14.9e9 / 2.14e-3 / 1e9 / 6793.1)
    assert r["other"]["bound"] == "tensor"
    c = bench.roofline({"flops": 0, "bytes": 4.2e9}, 0.65, PEAKS)  # the combine: no arithmetic
    assert c["bound"] == "hbm" and "other" not in c


def test_roofline_without_a_sustained_figure():
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}
    r = bench.roofline({"flops": 1e12, "bytes": 1e9}, 1.0, peaks)
    assert r["bound"] == "tensor" and r["peak"] == 1900.0 and "sustained" not in r


def test_traffic_record_needs_every_source_unchanged(tmp_path):
    # The record is used only while the digest over all of its source files
    # matches; a record naming one file too few, or a changed file, reads None.
    import json

    srcs = ["gemm_pair.cu", "gemm_impl.cuh", "mk_device.cuh", "mk_internal.h"]
    rec = {"sources": srcs, "sha256_16": bench.sources_digest(srcs), "dram_bytes_per_launch": 123}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps({"gemm1": {"large": rec}}))
    assert bench.traffic_record("gemm1", "large", str(path)) == 123
    assert bench.traffic_record("gemm2", "large", str(path)) is None
    stale = dict(rec, sha256_16=bench.sources_digest(srcs[:1]))
    path.write_text(json.dumps({"gemm1": {"large": stale}}))
    assert bench.traffic_record("gemm1", "large", str(path)) is None
    legacy = {"source": "gemm_pair.cu", "sha256_16": "0" * 16, "dram_bytes_per_launch": 1}
    path.write_text(json.dumps({"gemm1": {"large": legacy}}))
    assert bench.traffic_record("gemm1", "large", str(path)) is None


def test_phase_rooflines_per_step():
    cfg = CONFIGS["large"]
    offsets = np.arange(0, 257, dtype=np.int64) * 1024
    fb = bench.flops_bytes(cfg, offsets)
    phase = {"route_logits": 0.25, "topk": 0.75, "count": 0.01, "scan": 0.01, "scatter": 0.65,
             "gemm1": 8.9, "gemm2": 4.5, "combine": 0.68}
    pr = bench.phase_rooflines(fb, phase, PEAKS)
    assert set(pr) == {"gemm1", "gemm2", "scatter", "combine", "route"}
    assert pr["gemm1"]["bound"] == "tensor" and pr["gemm1"]["ms"] == 8.9
    # the scatter reads x once and writes the k copies: 32768*7168*2*(1+8) bytes in 0.65 ms
    assert pr["scatter"]["bound"] == "hbm"
    assert pr["scatter"]["achieved"] == pytest.approx(32768 * 7168 * 2 * 9 / 0.65e-3 / 1e9)
    # the router's kernels together, against HBM at its intensity (x read once)
    assert pr["route"]["ms"] == pytest.approx(1.0) and pr["route"]["bound"] == "hbm"
    assert pr["route"]["achieved"] == pytest.approx(
        (32768 * 7168 * 2 + 256 * 7168 * 4 + 32768 * 256 * 4) / 1.0e-3 / 1e9)


def test_launches_per_step_by_path_and_router():
    import dispatch_ffn_combine_gb300 as mk
    # large: the candidate-filter router (prep, approximate logits, select), then
    # count, scan, scatter, gemm1, gemm2, combine
    assert bench.launches_per_step(CONFIGS["large"], mk.MK_PATH_STEPS) == 9
    assert bench.launches_per_step(CONFIGS["large"], mk.MK_PATH_TILES) == 9
    # the fused path: the filter's three kernels, count and scan, then the persistent kernel
    assert bench.launches_per_step(CONFIGS["large"], mk.MK_PATH_FUSED) == 6
    # tiny: the plain router (logits, top-k) and the same six; fused: one kernel
    assert bench.launches_per_step(CONFIGS["tiny"], mk.MK_PATH_STEPS) == 8
    assert bench.launches_per_step(CONFIGS["tiny"], mk.MK_PATH_FUSED) == 1
