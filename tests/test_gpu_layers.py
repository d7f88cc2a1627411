"""GPU parity of the data-movement layers through the C ABI against the oracle:
max pooling's backward (LeNet page, 第五层 Pooling), the route layer's and the
YOLO layer's backward (YOLOv3 back-propagation page, §6 and §2).

Bars: the YOLO and route layers move and add single values, so their results
are exact (fp32 a + b on both sides); max pooling sums at most a few values
per element in the page's order, 1e-6 relative to the largest magnitude.
"""
import numpy as np
import pytest
import torch

import activation_backward_gb300 as cba
import oracle
from activation_backward_gb300 import inputs

pytestmark = pytest.mark.gpu

POOL_CASES = [
    # N, C, H, W, k, stride, pad
    (64, 20, 24, 24, 2, 2, 0),   # LeNet pool1 (batch 64)
    (64, 50, 8, 8, 2, 2, 0),     # LeNet pool2
    (4, 16, 13, 13, 3, 2, 1),    # overlapping windows, padding, ceil rule
    (2, 8, 17, 23, 3, 1, 0),     # stride 1: up to 9 windows per element
    (3, 5, 10, 7, 3, 2, 0),      # the last window clipped at the edge
    (2, 3, 14, 16, 3, 3, 1),     # stride 3 (not a power of two), 4-wide rows
    (2, 2, 9, 20, 5, 3, 2),      # kernel 5: windows per axis past the unrolled bound
    (1, 1, 1, 1, 1, 1, 0),       # one element
]


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("case", POOL_CASES, ids=[str(i) for i in range(len(POOL_CASES))])
def test_maxpool_backward_parity(cuda_lib, case):
    N, C, H, W, k, s, pad = case
    c = inputs.make_pool_case(N, C, H, W, k, s, pad, seed=80 + POOL_CASES.index(case))
    d = cba.make_pool_desc(N, C, H, W, k, s, pad)
    assert (cba.cba_pooled_size(H, k, s, pad), cba.cba_pooled_size(W, k, s, pad)) == (c["PH"],
                                                                                     c["PW"])
    top, mask = _dev(c["top_diff"]), _dev(c["mask"])
    bottom = torch.full((N, C, H, W), float("nan"), device="cuda")
    cba.cba_maxpool_backward(d, top, mask, bottom)
    torch.cuda.synchronize()
    got = bottom.cpu().numpy().astype(np.float64)
    exp = oracle.maxpool_backward(c["top_diff"], c["mask"], H, W)
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - exp)) <= 1e-6 * max(np.max(np.abs(exp)), 1e-30)
    # deterministic: a second run gives the same bits
    again = torch.full_like(bottom, float("nan"))
    cba.cba_maxpool_backward(d, top, mask, again)
    torch.cuda.synchronize()
    assert torch.equal(bottom, again)


def test_maxpool_backward_ignores_a_mask_outside_its_window(cuda_lib):
    c = inputs.make_pool_case(2, 3, 12, 12, 2, 2, 0, seed=91)
    mask = c["mask"].copy()
    mask[1, 2, 3, 4] = 0  # element (0, 0) is not in window (3, 4)
    d = cba.make_pool_desc(2, 3, 12, 12, 2, 2, 0)
    bottom = torch.empty((2, 3, 12, 12), device="cuda")
    cba.cba_maxpool_backward(d, _dev(c["top_diff"]), _dev(mask), bottom)
    torch.cuda.synchronize()
    td = c["top_diff"].copy()
    td[1, 2, 3, 4] = 0.0  # that top gradient is dropped
    exp = oracle.maxpool_backward(td, c["mask"], 12, 12)
    assert np.max(np.abs(bottom.cpu().numpy() - exp)) <= 1e-6 * np.max(np.abs(exp))


ROUTE_CASES = [
    (16, [128 * 26 * 26, 512 * 26 * 26]),  # a YOLOv3 route at 26x26 (upsampled 128 + 512)
    (3, [4 * 5 * 5, 7 * 3 * 3, 2 * 6 * 6]),  # sizes not multiples of 4: one value per thread
    (2, [8, 12, 4, 16, 20, 24, 28, 32]),   # the most inputs in one call
]


@pytest.mark.parametrize("case", ROUTE_CASES, ids=[str(i) for i in range(len(ROUTE_CASES))])
def test_route_backward_parity(cuda_lib, case):
    batch, sizes = case
    c = inputs.make_route_case(batch, sizes, seed=70 + ROUTE_CASES.index(case))
    route = _dev(c["route_delta"])
    deltas = [_dev(a) for a in c["input_deltas"]]
    cba.cba_route_backward(route, deltas)
    torch.cuda.synchronize()
    exp = oracle.route_backward(c["route_delta"], sizes, c["input_deltas"])
    for g, e in zip(deltas, exp):
        # one fp32 addition per element on the GPU, exact in the fp64 oracle
        assert np.array_equal(g.cpu().numpy(), e.astype(np.float32))


@pytest.mark.parametrize("n,offset", [(16 * 255 * 13 * 13, 0), (1000003, 0), (4097, 1)])
def test_yolo_backward_parity(cuda_lib, n, offset):
    rng = np.random.default_rng(n)
    l_delta = rng.standard_normal(n + offset).astype(np.float32)
    net = rng.standard_normal(n + offset).astype(np.float32)
    # offset 1 makes both views start 4 bytes past a 16-byte boundary
    l_dev, net_dev = _dev(l_delta)[offset:], _dev(net)[offset:]
    cba.cba_yolo_backward(l_dev, net_dev)
    torch.cuda.synchronize()
    exp = oracle.yolo_backward(l_delta[offset:], net[offset:])
    assert np.array_equal(net_dev.cpu().numpy(), exp.astype(np.float32))
