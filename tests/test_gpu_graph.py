"""CUDA-graph capture of the C-ABI call.

The library call only enqueues stream-ordered work on caller buffers (it
never allocates or synchronises), so it can be captured into a CUDA graph
once and replayed.  A replay must do exactly what a direct call does.  The
results are compared with direct calls on identical inputs, after one replay
(dW, db, dgamma accumulated once onto zeros) and after two (accumulated
twice): bit for bit where the kernels sum in a fixed order, which is every
output but one; the TF32 weight gradient adds its blocks' tiles with L2
reduce-adds, whose order varies from run to run, so there the bar is
rounding-order level (1e-5 of max |value|).
"""
import numpy as np
import pytest
import torch

import activation_backward_gb300 as cba
from activation_backward_gb300 import inputs
from activation_backward_gb300.layer import DeviceLayer, capture_graph

pytestmark = pytest.mark.gpu

KEYS = ("dW", "db", "dgamma", "prev_delta")


def _same(a, b, what, rel=0.0):
    assert (a is None) == (b is None), what
    if a is None:
        return
    if rel == 0.0:
        assert np.array_equal(a, b), f"{what}: max|diff| {np.max(np.abs(a - b)):.3e}"
    else:
        err, scale = float(np.max(np.abs(a - b))), float(np.max(np.abs(b)))
        assert err <= rel * scale, f"{what}: max|diff| {err:.3e} > {rel} * {scale:.3e}"


@pytest.mark.parametrize("math", [cba.CBA_MATH_TF32, cba.CBA_MATH_FFMA], ids=["tf32", "ffma"])
@pytest.mark.parametrize("cid", [2, 3])
def test_graph_replay_matches_direct_calls(cuda_lib, cid, math):
    layer = inputs.make_config(cid, batch=2)[0]
    direct = DeviceLayer(layer, math=math)
    direct.run()
    once = direct.results()
    direct.run()
    twice = direct.results()

    dl = DeviceLayer(layer, math=math)
    graph = capture_graph(dl.run, warmup=1)  # the warm-up call accumulates once
    dl.zero_outputs()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert dl.status() == cba.CBA_OK
    got1 = dl.results()
    graph.replay()
    torch.cuda.synchronize()
    assert dl.status() == cba.CBA_OK
    got2 = dl.results()
    for k in KEYS:
        rel = 1e-5 if (math == cba.CBA_MATH_TF32 and k == "dW") else 0.0
        _same(got1[k], once[k], f"replay 1 {k}", rel)
        _same(got2[k], twice[k], f"replay 2 {k}", rel)
