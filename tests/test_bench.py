"""The benchmark's accounting on CPU: algorithmic work, launch counts, the
traffic lookup and the peaks (no GPU, no kernel launches).

The per-token flop and byte counts are the scope table's formulas; the
headline figures they give (23.62 GFLOP, 143.65 MB per forward) are the
ones the roofline fraction divides by.
"""
import json
import os

import torch

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def shapes(B, T, Nk, Nv, dk, dv, dtype=torch.bfloat16, g=True, h0=True, N=None):
    """Stand-in inputs with the right shapes and element size (meta tensors)."""
    return dict(q=torch.empty(B, T, Nk, dk, dtype=dtype, device="meta"),
                v=torch.empty(B, T, Nv, dv, dtype=dtype, device="meta"),
                g=torch.empty(B, T, Nv, device="meta") if g else None,
                h0=torch.empty(N or B, Nv, dk, dv, device="meta") if h0 else None,
                N=N or B)


def test_headline_work():
    w = bench.algorithmic(shapes(4, 2048, 16, 16, 128, 128))
    assert w["tokens"] == 8192
    # per token: Nv (6 dk dv + 2C (dk + 2 dv)) + Nk 4 C dk
    assert w["flops"] == 8192 * (16 * (6 * 128 * 128 + 2 * 64 * (128 + 2 * 128)) + 16 * 4 * 64 * 128)
    assert round(w["flops"] / 1e9, 2) == 23.62
    # q, k, v, o in bf16, beta and g in fp32, h0 in and ht out in fp32
    want = 8192 * (2 * 16 * 128 * 2 + 2 * 16 * 128 * 2 + 16 * 4 * 2) + 4 * 16 * 128 * 128 * 4 * 2
    assert w["bytes"] == want and round(w["bytes"] / 1e6, 2) == 143.65


def test_optional_inputs_and_fp32():
    base = bench.algorithmic(shapes(1, 256, 2, 2, 64, 64, dtype=torch.float32, g=False, h0=False))
    # no g: beta only; no h0: ht only; fp32 elements
    assert base["bytes"] == 256 * (2 * 2 * 64 * 4 * 2 + 2 * 4) + 1 * 2 * 64 * 64 * 4
    gated = bench.algorithmic(shapes(1, 256, 2, 2, 64, 64, dtype=torch.float32, g=True, h0=False))
    assert gated["bytes"] - base["bytes"] == 256 * 2 * 4


def test_backward_work_adds_to_the_forward():
    inp = shapes(4, 2048, 16, 16, 128, 128)
    fwd, bwd = bench.algorithmic(inp), bench.algorithmic_bwd(inp)
    assert bwd["flops"] > fwd["flops"] and round(bwd["flops"] / 1e9, 1) == 81.6


def test_launch_counts():
    assert bench.launches_per_call("wy_fwd+tc_fwd") == 2
    assert bench.launches_per_call("fill_zero+wy_fwd+tc_fwd+simt_bwd<bf16,tf32>") == 4
    assert bench.launches_per_call("rec_fwd<bf16>") == 1


def test_traffic_follows_the_sources(tmp_path, monkeypatch):
    """A committed traffic figure is used only while the kernel sources hash
    matches the one it was taken on."""
    rec = {"wl": {"k": {"bytes_per_launch": 123, "sources": bench.sources_hash()}}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.measured_traffic("k", "wl") == 123
    assert bench.measured_traffic("other", "wl") is None
    rec["wl"]["k"]["sources"] = "0" * 16
    path.write_text(json.dumps(rec))
    assert bench.measured_traffic("k", "wl") is None


def test_peaks_and_fp32_alu():
    peaks, src = bench.load_peaks()
    assert src in ("measured", "fallback") and peaks["hbm_gbs"] > 1000 and peaks["bf16_tflops"] > 100
    assert abs(bench.fp32_alu_peak_tflops(2070.0) - 152 * 128 * 2 * 2070e6 / 1e12) < 1e-9


def test_weak_scaling_value():
    assert bench.weak_scaling_value(8192, 1, 1.0) == 8192 / 1e-3
    assert bench.weak_scaling_value(8192, 4, 2.0) == 8192 * 4 / 2e-3
