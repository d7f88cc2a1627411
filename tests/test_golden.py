"""Golden fixtures: the page's printed LeNet conv2 geometry, and a stored
oracle result (regression guard, written by tests/golden/make_golden.py)."""
import json
import os

import numpy as np

from activation_backward_gb300 import inputs

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_lenet_conv2_geometry_matches_page():
    g = json.load(open(os.path.join(GOLD, "lenet_conv2_geometry.json")))
    spec = inputs.CONFIGS[1].geom
    assert [spec.N, spec.C, spec.H, spec.W] == g["bottom_NCHW"]
    assert [spec.N, spec.K, spec.P, spec.Q] == g["top_NCHW"]
    assert [spec.K, spec.C * spec.R * spec.S] == g["weight_gemm_view"]
    assert [spec.P * spec.Q, spec.C * spec.R * spec.S] == g["bottom_gemm_view_per_sample"]
    assert [spec.P * spec.Q, spec.K] == g["top_gemm_view_per_sample"]
    assert spec.R == spec.S == g["kernel"]


def test_oracle_tiny_case_unchanged(ref):
    doc = json.load(open(os.path.join(GOLD, "oracle_tiny_case.json")))
    inp = {k: np.asarray(v, np.float32) for k, v in doc["inputs"].items()}
    got = ref.conv_bn_act_backward(inp["x"], inp["output"], inp["z"], inp["delta"], inp["W"],
                                   inp["gamma"], inp["mean"], inp["var"], inp["residual"],
                                   stride=doc["stride"], pad=doc["pad"], act=ref.ACT_LEAKY,
                                   batch_normalize=True, accumulate=0, eps=doc["eps"])
    for k, v in doc["outputs"].items():
        exp = np.asarray(v)
        assert np.allclose(got[k], exp, rtol=1e-12, atol=1e-14), k
