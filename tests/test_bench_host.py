"""Host-side arithmetic of bench.py (no GPU): the TF32 denominator, the
per-workload summary and the ncu traffic lookup."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from activation_backward_gb300 import inputs  # noqa: E402


def test_tf32_denominator_is_the_larger_of_the_two_figures():
    peaks = {"bf16_tflops": 1800.0, "hbm_gbs": 6000.0}
    ratio = 1800.0 * 1.1 / 2.25
    v, src = bench.tf32_peak(peaks, "measured", None)
    assert v == ratio and "cuBLAS" not in src
    v, src = bench.tf32_peak(peaks, "measured", ratio + 50.0)
    assert v == ratio + 50.0 and "cuBLAS" in src
    v, _ = bench.tf32_peak(peaks, "measured", ratio - 50.0)
    assert v == ratio


def test_summary_of_a_two_layer_step():
    # the residual block's two layers at batch 2; fake step and phase times
    layers = inputs.make_config(5, batch=2)
    t = {"layers": layers, "step_ms": [1.0, 3.0], "direct_ms": 2.5,
         "paths": ["tc_batch_inner", "tc_rows"], "layout_bytes": [6e6, 2e6],
         "phases": [{"reduce": 0.1, "layout": 0.02, "wgrad": 0.4, "dgrad": 0.3},
                    {"reduce": 0.05, "layout": 0.01, "wgrad": 0.2, "dgrad": 0.1}]}
    d = bench.summarize(t, tf32=1000.0, hbm=5000.0)
    flops = sum(2 * l["geom"].gemm_flops() for l in layers)
    assert d["workload"] == "residual_block"
    assert d["ms_per_step"] == 2.0
    assert abs(d["tflops"] - flops / 2e-3 / 1e12) < 1e-9
    assert abs(d["wgrad_ms"] - 0.6) < 1e-12 and abs(d["dgrad_ms"] - 0.4) < 1e-12
    assert abs(d["gemm_frac_tf32"] - flops / 1e-3 / 1e12 / 1000.0) < 1e-12
    red = sum(inputs.layer_bytes_reduce(l) for l in layers)
    assert abs(d["reduce_frac_hbm"] - red / 0.15e-3 / 1e9 / 5000.0) < 1e-9
    assert abs(d["layout_frac_hbm"] - 8e6 / 0.03e-3 / 1e9 / 5000.0) < 1e-9
    assert abs(d["layers"][1]["layout_frac_hbm"] - 2e6 / 0.01e-3 / 1e9 / 5000.0) < 1e-9
    assert len(d["layers"]) == 2
    g = layers[0]["geom"]
    assert abs(d["layers"][0]["wgrad_frac_tf32"] - g.gemm_flops() / 0.4e-3 / 1e12 / 1000.0) < 1e-9


def test_traffic_lookup_needs_a_matching_source_hash(tmp_path, monkeypatch):
    import hashlib
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    prof = tmp_path / "profiles"
    prof.mkdir()
    sha = hashlib.sha1(b"kernel v1").hexdigest()
    (prof / "x.md").write_text(
        f"traffic: workload=residual_block layer=0 phase=wgrad bytes=123 source=k.cu sha1={sha}\n"
        f"traffic: phase=dgrad bytes=77 source=k.cu sha1={sha}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("wgrad", "residual_block", 0) == 123
    assert bench.profiled_traffic("wgrad", "residual_block", 1) is None
    assert bench.profiled_traffic("dgrad", "darknet_3x3", 0) == 77
    src.write_text("kernel v2")  # the kernel changed since the capture
    assert bench.profiled_traffic("wgrad", "residual_block", 0) is None
