"""Host-side checks of the data-movement layer entry points (no GPU): the
library's pooled-size rule against the oracle's, and argument validation
(every rejected call returns before any CUDA call, so the pointers are never
dereferenced)."""
import ctypes

import pytest

import activation_backward_gb300 as cba
import oracle
from activation_backward_gb300 import _binding as B


@pytest.fixture(scope="module")
def lib():
    from activation_backward_gb300 import build
    build.build()
    return B.load()


def test_pooled_size_agrees_with_the_oracle(lib):
    for n in range(1, 40):
        for k in range(1, 6):
            for s in range(1, 4):
                for pad in range(0, k):
                    if n + 2 * pad < k:
                        continue
                    assert lib.cba_pooled_size(n, k, s, pad) == oracle.pooled_size(n, k, s, pad)
    assert lib.cba_pooled_size(0, 2, 2, 0) == -1
    assert lib.cba_pooled_size(4, 2, 0, 0) == -1


FAKE = 1 << 20  # aligned, never dereferenced


def test_yolo_backward_rejects_bad_arguments(lib):
    assert lib.cba_yolo_backward(FAKE, FAKE, -1, None) == cba.CBA_ERR_ARG
    assert lib.cba_yolo_backward(None, FAKE, 5, None) == cba.CBA_ERR_ARG
    assert lib.cba_yolo_backward(None, None, 0, None) == cba.CBA_OK  # nothing to do


def test_route_backward_rejects_bad_arguments(lib):
    def call(batch, sizes, ptrs, route=FAKE):
        n = len(sizes)
        s = (ctypes.c_longlong * max(n, 1))(*sizes)
        p = (ctypes.c_void_p * max(n, 1))(*ptrs)
        return lib.cba_route_backward(route, batch, n, s, p, None)
    assert call(0, [4], [FAKE]) == cba.CBA_ERR_ARG
    assert call(2, [4, 0], [FAKE, FAKE]) == cba.CBA_ERR_ARG
    assert call(2, [4, 4], [FAKE, None]) == cba.CBA_ERR_ARG
    assert call(2, [4] * (cba.CBA_ROUTE_MAX_INPUTS + 1),
                [FAKE] * (cba.CBA_ROUTE_MAX_INPUTS + 1)) == cba.CBA_ERR_ARG
    assert call(2, [4], [FAKE], route=None) == cba.CBA_ERR_ARG


@pytest.mark.parametrize("bad", [dict(N=0), dict(H=0), dict(kernel_h=0), dict(stride_w=0),
                                 dict(pad_h=-1), dict(pad_w=2), dict(H=1, kernel_h=3)])
def test_maxpool_backward_rejects_bad_descriptors(lib, bad):
    kw = dict(N=2, C=3, H=8, W=8, kernel_h=2, kernel_w=2, stride_h=2, stride_w=2, pad_h=0,
              pad_w=0)
    kw.update(bad)
    d = B.cba_pool_desc_t(**kw)
    assert lib.cba_maxpool_backward(ctypes.byref(d), FAKE, FAKE, FAKE, None) == cba.CBA_ERR_ARG
