"""Pins of the oracle's data-movement layers (CPU only): the max-pooling
backward of the LeNet page (第五层 Pooling), the route-layer and YOLO-layer
backward of the YOLOv3 back-propagation page (§6, §2).

Each is checked against a library special case that computes the same
gradient by a different route: torch's max_pool2d with ceil_mode (caffe's
pooled-size rule and window clipping) and its autograd, autograd through
torch.cat, and the gradient of an identity layer.  The generator's mask is
pinned to torch's argmax indices as well.
"""
import numpy as np
import pytest
import torch

import oracle
from activation_backward_gb300 import inputs

POOL_CASES = [
    # N, C, H, W, k, stride, pad
    (4, 20, 24, 24, 2, 2, 0),   # LeNet pool1 geometry (caffe 第五层 Pooling)
    (3, 5, 8, 8, 2, 2, 0),      # LeNet pool2 spatial size
    (2, 3, 13, 13, 3, 2, 1),    # overlapping windows, padding, ceil rule
    (2, 4, 9, 11, 3, 1, 0),     # stride 1: every interior element in 9 windows
    (2, 2, 10, 7, 3, 2, 0),     # ragged: the last window clipped at the bottom edge
]


@pytest.mark.parametrize("n,k,s,pad", [(24, 2, 2, 0), (13, 3, 2, 1), (12, 3, 2, 1),
                                       (7, 3, 2, 0), (10, 3, 3, 1), (5, 2, 1, 1)])
def test_pooled_size_matches_torch_ceil_mode(n, k, s, pad):
    out = torch.nn.functional.max_pool2d(torch.zeros(1, 1, n, n), k, s, pad, ceil_mode=True)
    assert oracle.pooled_size(n, k, s, pad) == out.shape[-1]
    assert inputs.pooled_size(n, k, s, pad) == out.shape[-1]


@pytest.mark.parametrize("case", POOL_CASES, ids=[str(i) for i in range(len(POOL_CASES))])
def test_maxpool_backward_matches_torch_autograd(case):
    N, C, H, W, k, s, pad = case
    c = inputs.make_pool_case(N, C, H, W, k, s, pad, seed=50 + POOL_CASES.index(case))
    x = torch.from_numpy(c["bottom"].astype(np.float64)).requires_grad_(True)
    y, idx = torch.nn.functional.max_pool2d(x, k, s, pad, ceil_mode=True, return_indices=True)
    assert y.shape[-2:] == (c["PH"], c["PW"])
    # the generator's mask is the forward's argmax (values are distinct)
    assert np.array_equal(idx.numpy(), c["mask"])
    (y * torch.from_numpy(c["top_diff"].astype(np.float64))).sum().backward()
    got = oracle.maxpool_backward(c["top_diff"], c["mask"], H, W)
    assert np.max(np.abs(got - x.grad.numpy())) < 1e-12
    # every top gradient lands once: the sums agree per plane
    assert np.allclose(got.sum(axis=(2, 3)), c["top_diff"].astype(np.float64).sum(axis=(2, 3)))


def test_route_backward_matches_autograd_through_concat():
    sizes = [3 * 4 * 4, 5 * 4 * 4, 2 * 4 * 4]
    c = inputs.make_route_case(3, sizes, seed=7)
    xs = [torch.zeros(c["batch"], s, dtype=torch.float64, requires_grad=True) for s in sizes]
    y = torch.cat(xs, dim=1)  # the route layer's forward: inputs side by side per image
    (y * torch.from_numpy(c["route_delta"].astype(np.float64))).sum().backward()
    got = oracle.route_backward(c["route_delta"], sizes, c["input_deltas"])
    for g, x, d0 in zip(got, xs, c["input_deltas"]):
        # the backward adds onto the deltas the input layers already hold
        assert np.max(np.abs(g - (d0.astype(np.float64) + x.grad.numpy()))) < 1e-12


def test_yolo_backward_is_the_identity_gradient():
    rng = np.random.default_rng(3)
    l_delta = rng.standard_normal(1000)
    net0 = rng.standard_normal(1000)
    x = torch.zeros(1000, dtype=torch.float64, requires_grad=True)
    (x * torch.from_numpy(l_delta)).sum().backward()  # the layer passes its input on
    got = oracle.yolo_backward(l_delta, net0)
    assert np.max(np.abs(got - (net0 + x.grad.numpy()))) < 1e-12
