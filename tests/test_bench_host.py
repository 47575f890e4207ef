"""Host-side pieces of bench.py (CPU): the algorithmic work per stage, the launch counts it
claims, the kernel choice it reports, and the reading of committed ncu traffic summaries."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mixture_experts_layer_84_b300 import workloads as W  # noqa: E402


def test_stage_work_mixtral_closed_forms():
    """Mixtral shape, no drops (A = T k): the GEMM is 6 A h d_e FLOPs over 3 E h d_e weights plus
    X, act (out and in) and Y; dispatch reads U once and writes X."""
    w = W.MIXTRAL
    A = w.T * w.k
    work = bench.stage_work(w, A, w.E)
    assert work["ffn"]["flops"] == 6 * A * w.h * w.d_e
    assert work["ffn"]["bytes"] == 3 * w.E * w.h * w.d_e * 2 + 2 * A * w.h * 2 + 2 * A * w.d_e * 2
    assert work["dispatch"]["bytes"] == w.T * w.h * 2 + A * w.h * 2 + w.T * w.k * 12
    assert work["combine"]["bytes"] == A * w.h * 2 + 2 * w.T * w.h * 2 + w.T * w.k * 8
    assert work["route"]["flops"] == 2 * w.T * w.h * w.E


def test_stage_work_fp8_and_gather_variants():
    w = W.MIXTRAL
    A = w.T * w.k
    base = bench.stage_work(w, A, w.E)
    f8 = bench.stage_work(w, A, w.E, fp8=True)
    # gate/up weights and the dispatched rows at one byte, plus a float32 scale per row
    assert base["ffn"]["bytes"] - f8["ffn"]["bytes"] == 2 * w.E * w.h * w.d_e + A * w.h
    assert base["dispatch"]["bytes"] - f8["dispatch"]["bytes"] == A * w.h - 4 * A
    assert f8["ffn"]["flops"] == base["ffn"]["flops"]
    g = bench.stage_work(w, A, w.E, gather=True)
    assert g["dispatch"]["bytes"] == w.T * w.k * 12 and g["ffn"] == base["ffn"]


# (workload, choice-major, token-major, token-major gathered, FP8 choice-major, FP8 token-major)
@pytest.mark.parametrize("w,cm,tm,tm_g,f8,tm_f8", [
    (W.MIXTRAL, 5, 8, 7, 6, 8),        # 4096 ids: one dispatch launch
    (W.TINY_FP32, 6, 9, 8, 7, 9),      # two router launches (float32), 512 ids
    (W.MIXTRAL.replace(name="m16k", T=16384), 6, 8, 7, 7, 8),  # 32768 ids, 256 chunks x 16 columns
    (W.DSV3_SHARED, 9, 10, 9, 10, 10), # 256 x 2048 columns: the column scan; two shared-expert GEMMs
    (W.SWITCH, 7, 8, 7, 8, 8),         # 256 x 128 columns: the column scan
])
def test_launches_per_step(w, cm, tm, tm_g, f8, tm_f8):
    """route (the fused tensor-core router from weights packed beforehand, else logits +
    selection), dispatch (histograms unless the batch holds at most 8192 expert ids, column scans
    unless the histograms hold at most 8192 counts, then slots + row copy), two GEMMs per routed
    and per shared expert block, combine with
    statistics; token-major dispatch takes count, scan, assign and scatter."""
    t = w.replace(priority=W.PRIORITY_TOKEN_MAJOR)
    assert bench.launches_per_step(w) == cm
    assert bench.launches_per_step(w, gather=True) == cm
    assert bench.launches_per_step(t) == tm
    assert bench.launches_per_step(t, gather=True) == tm_g
    assert bench.launches_per_step(w, fp8=True) == f8
    assert bench.launches_per_step(t, fp8=True) == tm_f8


def test_launches_per_step_empty_batch():
    assert bench.launches_per_step(W.MIXTRAL.replace(name="empty", T=0)) == 2


def test_ffn_tiles_rule(monkeypatch):
    monkeypatch.delenv("MOE_FFN_TILES", raising=False)
    assert bench.ffn_tiles(W.MIXTRAL) == "swab"      # 512 rows per expert
    assert bench.ffn_tiles(W.DSV3) == "swab"         # 128 rows per expert
    assert bench.ffn_tiles(W.STRESS) == "pair"       # 6144 rows per expert
    assert bench.ffn_tiles(W.TINY_FP32) == "cuda-core float32"
    monkeypatch.setenv("MOE_FFN_TILES", "single")
    assert bench.ffn_tiles(W.MIXTRAL).startswith("single")


def test_profile_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """A summary counts only while its source hash matches the current GEMM sources."""
    sha = bench.kernel_source_sha(bench.GEMM_SOURCES)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "grouped_gemm_x.md").write_text(f"source_sha256: {sha}\ntraffic_bytes_per_step: 1234\n")
    (prof / "grouped_gemm_y.md").write_text("source_sha256: " + "0" * 64 + "\ntraffic_bytes_per_step: 99\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda files: sha)
    assert bench.profile_traffic("x") == 1234.0
    assert bench.profile_traffic("y") is None
    assert bench.profile_traffic("missing") is None
