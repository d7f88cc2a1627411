"""Writes tests/golden/oracle_tiny_case.json: the oracle's outputs for one tiny
seeded layer (3x3, stride 2, pad 1, BN + leaky, shortcut residual).  The values
come from the oracle alone; the fixture guards the oracle against unintended
changes.  Run from the repo root:  python tests/golden/make_golden.py"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def tiny_inputs():
    rng = np.random.default_rng(4242)
    N, C, H, W, K = 2, 3, 6, 5, 4
    x = rng.uniform(-1, 1, (N, C, H, W)).astype(np.float32)
    w = rng.uniform(-0.5, 0.5, (K, C, 3, 3)).astype(np.float32)
    P, Q = (H + 2 - 3) // 2 + 1, (W + 2 - 3) // 2 + 1
    z = rng.uniform(-1, 1, (N, K, P, Q)).astype(np.float32)
    mean = z.astype(np.float64).mean(axis=(0, 2, 3)).astype(np.float32)
    var = z.astype(np.float64).var(axis=(0, 2, 3)).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, K).astype(np.float32)
    out = rng.uniform(-1, 1, (N, K, P, Q)).astype(np.float32)  # only its sign is used
    delta = rng.uniform(-1, 1, (N, K, P, Q)).astype(np.float32)
    res = rng.uniform(-1, 1, (N, C, H, W)).astype(np.float32)
    return dict(x=x, W=w, z=z, mean=mean, var=var, gamma=gamma, output=out, delta=delta,
                residual=res)


def run(inp):
    return oracle.conv_bn_act_backward(inp["x"], inp["output"], inp["z"], inp["delta"], inp["W"],
                                       inp["gamma"], inp["mean"], inp["var"], inp["residual"],
                                       stride=2, pad=1, act=oracle.ACT_LEAKY, batch_normalize=True,
                                       accumulate=0, eps=1e-5)


if __name__ == "__main__":
    inp = tiny_inputs()
    got = run(inp)
    doc = {"source": "oracle outputs (tests/golden/make_golden.py); inputs: tiny_inputs()",
           "stride": 2, "pad": 1, "act": "leaky", "bn": True, "eps": 1e-5,
           "inputs": {k: v.astype(np.float64).tolist() for k, v in inp.items()},
           "outputs": {k: v.tolist() for k, v in got.items() if v is not None}}
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny_case.json"),
              "w") as f:
        json.dump(doc, f)
    print("written")
