"""Host-side pieces of bench.py (no GPU): the algorithmic bytes and flops
the roofline divides by, and the rule that a measured traffic figure is
reported only while the kernel's sources are unchanged."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from chunked_prefill_hybrid_gb300 import synth  # noqa: E402

PEAKS = {"hbm_gbs": 6781.8, "bf16_tflops": 1872.1, "source": "test"}


def test_attention_algorithmic_bytes_of_the_13b_batch():
    # chunk 256 at offset 768 (1024 keys) + 18 decodes at ctx 1024 (1025 keys each), 40 KV heads x 128, bf16 K and V,
    # plus q in and o out for the 274 rows
    dims = synth.LLAMA_13B
    ctx_len = [768 + 256] + [1025] * 18
    r = bench.roofline_for("attention", {"attention": (0.1, 1)}, dims, 274, 18, ctx_len, PEAKS)
    want = (1024 + 18 * 1025) * 2 * 40 * 128 * 2 + 2 * 274 * 40 * 128 * 2
    assert r["algorithmic"] == want == 404_439_040
    assert r["bound"] == "hbm"
    assert r["per_launch_us"] == pytest.approx(100.0)
    assert r["frac"] == pytest.approx(want / 100e-6 / 1e9 / 6781.8)


def test_gemm_rooflines_pick_the_larger_bound():
    dims = synth.LLAMA_13B
    prof = {k: (0.05, 1) for k in ("gemm_qkv", "gemm_o", "gemm_gate_up", "gemm_down")}
    gu = bench.roofline_for("gemm_gate_up", prof, dims, 274, 18, [], PEAKS)
    byts = 2 * 13824 * 5120 * 2 + 274 * 5120 * 2 + 274 * 13824 * 2
    # at T = 274 the gate/up product sits just below the measured ridge (about 276 rows)
    assert 2.0 * 274 * 2 * 13824 * 5120 / 1872.1e12 < byts / 6781.8e9
    assert gu["bound"] == "hbm" and gu["algorithmic"] == byts
    big = bench.roofline_for("gemm_gate_up", prof, dims, 512, 18, [], PEAKS)
    assert big["bound"] == "tensor" and big["algorithmic"] == pytest.approx(2.0 * 512 * 2 * 13824 * 5120)
    assert big["unit"] == "TFLOP/s"


def test_measured_traffic_needs_unchanged_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "chunked_prefill_hybrid_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC_PROFILES", {"attention": "p.md"})
    sha = bench.sources_sha256(["k.cu"])
    (tmp_path / "profiles" / "p.md").write_text(
        f"# x\n\ntraffic_bytes_per_launch: 1234\nsources: k.cu\nsources_sha256: {sha}\n")
    assert bench.measured_traffic("attention") == 1234.0
    (csrc / "k.cu").write_text("kernel v2\n")
    assert bench.measured_traffic("attention") is None
    assert bench.measured_traffic("gemm_o") is None


def test_committed_profiles_parse():
    for kind in bench.TRAFFIC_PROFILES:
        v = bench.measured_traffic(kind)
        assert v is None or v > 1e6


def test_gemm_decode_cost_uses_the_linear_ops_only():
    steps, D = 10, 18
    # per-kind (total ms over the steps, launches); attention and norms must not count
    hybrid = {"gemm_qkv": (0.50, 10), "gemm_o": (0.40, 10), "gemm_gate_up": (0.90, 10), "gemm_down": (0.50, 10),
              "attention": (1.0, 10), "rmsnorm": (0.1, 10)}
    chunk = {"gemm_qkv": (0.48, 10), "gemm_o": (0.38, 10), "gemm_gate_up": (0.86, 10), "gemm_down": (0.48, 10),
             "attention": (0.5, 10)}
    dec = {"gemm_qkv": (0.45, 10), "gemm_o": (0.35, 10), "gemm_gate_up": (0.80, 10), "gemm_down": (0.45, 10),
           "attention": (0.6, 10)}
    r = bench.gemm_decode_cost(hybrid, chunk, dec, steps, D)
    assert r["ms_gemm_hybrid"] == pytest.approx(0.23)
    assert r["ms_gemm_chunk_alone"] == pytest.approx(0.22)
    assert r["ms_gemm_decode_only"] == pytest.approx(0.205)
    assert r["per_decode_cost_ratio"] == pytest.approx((0.205 / D) / ((0.23 - 0.22) / D))
    # no marginal cost measured: no ratio
    assert bench.gemm_decode_cost(chunk, chunk, dec, steps, D)["per_decode_cost_ratio"] is None
