"""ctypes wrappers over the oracle's C library (``libcba_ref.so``).

Test infrastructure only (see the package docstring).  All wrappers take numpy
arrays and return float64 numpy arrays; nothing here does arithmetic of the
method itself -- every step runs in ``cba_ref.c``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

# activation codes (the library's cba_act_t)
ACT_LINEAR = 0
ACT_LEAKY = 1
ACT_LOGISTIC = 2
ACT_RELU = 3
ACT_RELIE = 4
ACT_RAMP = 5
ACT_TANH = 6
ACT_PLSE = 7
ACT_ELU = 8
ACT_SELU = 9
ACT_LHTAN = 10
ACT_HARDTAN = 11
ACT_LOGGY = 12
ACT_STAIR = 13

BN_NONE = 0
BN_BATCH = 1     # training mode: batch statistics
BN_FROZEN = 2    # frozen statistics: mean and var are constants of the forward

_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_lp = ctypes.POINTER(ctypes.c_long)
_i = ctypes.c_int
_l = ctypes.c_long
_d = ctypes.c_double


def lib():
    """Load (building first if needed) the oracle library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.cba_ref_activation_gradient.restype = _d
        L.cba_ref_activation_gradient.argtypes = [_i, _d]
        L.cba_ref_out_size.restype = _i
        L.cba_ref_out_size.argtypes = [_i, _i, _i, _i]
        L.cba_ref_get_threads.restype = _i
        L.cba_ref_set_threads.argtypes = [_i]
        L.cba_ref_gradient_array.argtypes = [_dp, _l, _i, _dp]
        L.cba_ref_backward_bias.argtypes = [_dp, _dp, _i, _i, _i]
        L.cba_ref_x_norm.argtypes = [_dp, _dp, _dp, _d, _i, _i, _i, _dp]
        L.cba_ref_backward_scale.argtypes = [_dp, _dp, _i, _i, _i, _dp]
        L.cba_ref_scale_bias.argtypes = [_dp, _dp, _i, _i, _i]
        L.cba_ref_mean_delta.argtypes = [_dp, _dp, _d, _i, _i, _i, _dp]
        L.cba_ref_variance_delta.argtypes = [_dp, _dp, _dp, _dp, _d, _i, _i, _i, _dp]
        L.cba_ref_normalize_delta.argtypes = [_dp, _dp, _dp, _dp, _dp, _d, _i, _i, _i, _dp]
        L.cba_ref_backward_batchnorm.restype = _i
        L.cba_ref_backward_batchnorm.argtypes = [_dp, _dp, _dp, _dp, _dp, _d, _i, _i, _i, _dp,
                                                 _dp, _dp]
        L.cba_ref_bn_backward_caffe.argtypes = [_dp, _dp, _dp, _d, _i, _i, _i, _dp]
        geo = [_i] * 9
        L.cba_ref_conv_wgrad.argtypes = [_dp, _dp] + geo + [_dp]
        L.cba_ref_conv_dgrad.argtypes = [_dp, _dp] + geo + [_dp]
        L.cba_ref_axpy.argtypes = [_l, _d, _dp, _dp]
        L.cba_ref_conv_bn_act_backward_f64.restype = _i
        L.cba_ref_conv_bn_act_backward_f64.argtypes = (
            [_i] * 12 + [_d] + [_dp] * 9 + [_dp] * 5)
        L.cba_ref_conv_bn_act_backward.restype = _i
        L.cba_ref_conv_bn_act_backward.argtypes = (
            [_i] * 12 + [ctypes.c_float] + [_fp] * 9 + [_dp] * 5)
        L.cba_ref_conv_bn_act_backward_grouped_f64.restype = _i
        L.cba_ref_conv_bn_act_backward_grouped_f64.argtypes = (
            [_i] * 13 + [_d] + [_dp] * 9 + [_dp] * 5)
        L.cba_ref_conv_bn_act_backward_grouped.restype = _i
        L.cba_ref_conv_bn_act_backward_grouped.argtypes = (
            [_i] * 13 + [ctypes.c_float] + [_fp] * 9 + [_dp] * 5)
        L.cba_ref_backward_dz.restype = _i
        L.cba_ref_backward_dz.argtypes = ([_i] * 6 + [ctypes.c_float] + [_fp] * 6 +
                                          [_dp] * 3)
        L.cba_ref_wgrad_at.argtypes = [_dp, _fp] + geo + [_lp, _l, _dp]
        L.cba_ref_dgrad_at.argtypes = [_dp, _fp, _fp, _fp, _i] + geo + [_lp, _l, _dp]
        L.cba_ref_yolo_backward.argtypes = [_dp, _l, _dp]
        L.cba_ref_route_backward.argtypes = [_dp, _i, _i, ctypes.POINTER(_i),
                                             ctypes.POINTER(_dp)]
        L.cba_ref_pooled_size.restype = _i
        L.cba_ref_pooled_size.argtypes = [_i, _i, _i, _i]
        L.cba_ref_maxpool_backward.argtypes = [_dp, ctypes.POINTER(_i)] + [_i] * 6 + [_dp]
        _lib = L
    return _lib


def _pd(a):
    """Pointer to a contiguous float64 array (or NULL for None)."""
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_dp)


def _pf(a):
    if a is None:
        return None
    assert a.dtype == np.float32 and a.flags.c_contiguous
    return a.ctypes.data_as(_fp)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def set_threads(n):
    lib().cba_ref_set_threads(int(n))


def get_threads():
    return lib().cba_ref_get_threads()


def out_size(n, k, stride, pad):
    return lib().cba_ref_out_size(n, k, stride, pad)


def activation_gradient(act, y):
    return lib().cba_ref_activation_gradient(int(act), float(y))


def gradient_array(output, act, delta):
    d = _f64(delta).copy()
    lib().cba_ref_gradient_array(_pd(_f64(output)), d.size, int(act), _pd(d))
    return d


def x_norm(z, mean, var, eps):
    z = _f64(z)
    N, K = z.shape[0], z.shape[1]
    sp = z[0, 0].size
    out = np.empty_like(z)
    lib().cba_ref_x_norm(_pd(z), _pd(_f64(mean)), _pd(_f64(var)), float(eps), N, K, sp, _pd(out))
    return out


def backward_batchnorm(z, x_norm_, mean, var, gamma, eps, delta, bias_updates, scale_updates):
    """Darknet order; returns (delta_bn, bias_updates, scale_updates), all new arrays."""
    z = _f64(z)
    N, K = z.shape[0], z.shape[1]
    sp = z[0, 0].size
    d = _f64(delta).copy()
    bu = _f64(bias_updates).copy()
    su = _f64(scale_updates).copy()
    rc = lib().cba_ref_backward_batchnorm(_pd(z), _pd(_f64(x_norm_)), _pd(_f64(mean)),
                                          _pd(_f64(var)), _pd(_f64(gamma)), float(eps), N, K, sp,
                                          _pd(d), _pd(bu), _pd(su))
    assert rc == 0
    return d, bu, su


def bn_backward_caffe(top_diff, x_norm_, var, eps):
    td = _f64(top_diff)
    N, K = td.shape[0], td.shape[1]
    sp = td[0, 0].size
    out = np.empty_like(td)
    lib().cba_ref_bn_backward_caffe(_pd(td), _pd(_f64(x_norm_)), _pd(_f64(var)), float(eps), N, K,
                                    sp, _pd(out))
    return out


def conv_wgrad(delta, x, R, S, stride, pad, dW=None):
    delta, x = _f64(delta), _f64(x)
    N, C, H, W = x.shape
    K = delta.shape[1]
    out = np.zeros((K, C, R, S)) if dW is None else _f64(dW).copy()
    lib().cba_ref_conv_wgrad(_pd(delta), _pd(x), N, C, H, W, K, R, S, stride, pad, _pd(out))
    return out


def conv_dgrad(delta, Wt, H, W, stride, pad, dx=None):
    delta, Wt = _f64(delta), _f64(Wt)
    K, C, R, S = Wt.shape
    N = delta.shape[0]
    out = np.zeros((N, C, H, W)) if dx is None else _f64(dx).copy()
    lib().cba_ref_conv_dgrad(_pd(delta), _pd(Wt), N, C, H, W, K, R, S, stride, pad, _pd(out))
    return out


def conv_bn_act_backward(x, output, z, delta, Wt, gamma, mean, var, residual, *, stride, pad,
                         act, batch_normalize, accumulate, eps, dW=None, db=None, dgamma=None,
                         prev_delta=None, want_prev=True, want_dz=False, f64_inputs=False,
                         groups=1):
    """Run the whole chain.  Inputs are float32 arrays (the GPU's bits) unless
    ``f64_inputs``; returns dict(dW, db, dgamma, prev_delta, dz) of float64
    arrays.  dW/db/dgamma start from the given arrays (zeros if None) and
    accumulate; prev_delta starts from the given array when accumulate=1.
    With ``groups``, Wt is [K, C/groups, R, S]."""
    N, C, H, W = x.shape
    K, Cg, R, S = Wt.shape
    assert Cg * groups == C
    P, Q = out_size(H, R, stride, pad), out_size(W, S, stride, pad)
    o_dW = np.zeros((K, Cg, R, S)) if dW is None else _f64(dW).copy()
    o_db = np.zeros(K) if db is None else _f64(db).copy()
    o_dg = (np.zeros(K) if dgamma is None else _f64(dgamma).copy()) if batch_normalize else None
    o_prev = None
    if want_prev:
        o_prev = np.zeros((N, C, H, W)) if prev_delta is None else _f64(prev_delta).copy()
    o_dz = np.empty((N, K, P, Q)) if want_dz else None
    L = lib()
    if f64_inputs:
        conv = lambda a: _pd(_f64(a))  # noqa: E731
        fn = L.cba_ref_conv_bn_act_backward_grouped_f64
        e = float(eps)
    else:
        conv = lambda a: _pf(None if a is None else np.ascontiguousarray(a, np.float32))  # noqa
        fn = L.cba_ref_conv_bn_act_backward_grouped
        e = ctypes.c_float(eps)
    keep = [x, output, z, delta, Wt, gamma, mean, var, residual]
    ptrs = [conv(a) for a in keep]
    rc = fn(N, C, H, W, K, R, S, stride, pad, int(groups), int(act), int(batch_normalize),
            int(bool(accumulate)), e, *ptrs, _pd(o_dW), _pd(o_db), _pd(o_dg), _pd(o_prev),
            _pd(o_dz))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return dict(dW=o_dW, db=o_db, dgamma=o_dg, prev_delta=o_prev, dz=o_dz)


def backward_dz(output, z, delta, gamma, mean, var, *, act, batch_normalize, eps, db=None,
                dgamma=None):
    """Activation gradient + BN backward (or backward_bias) on the float inputs.
    Returns (dz, db, dgamma) as float64 arrays (db/dgamma accumulate onto the
    given arrays, zeros if None)."""
    delta = np.ascontiguousarray(delta, np.float32)
    N, K, P, Q = delta.shape
    dz = np.empty(delta.shape)
    o_db = np.zeros(K) if db is None else _f64(db).copy()
    o_dg = (np.zeros(K) if dgamma is None else _f64(dgamma).copy()) if batch_normalize else None
    f = lambda a: None if a is None else _pf(np.ascontiguousarray(a, np.float32))  # noqa: E731
    keep = [output, z, delta, gamma, mean, var]
    rc = lib().cba_ref_backward_dz(N, K, P, Q, int(act), int(batch_normalize),
                                   ctypes.c_float(eps), *[f(a) for a in keep], _pd(dz), _pd(o_db),
                                   _pd(o_dg))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return dz, o_db, o_dg


def wgrad_at(dz, x, R, S, stride, pad, idx):
    """Sampled dW elements (flat [K,C,R,S] indices) from the BN-input gradient dz."""
    dz = _f64(dz)
    x = np.ascontiguousarray(x, np.float32)
    N, C, H, W = x.shape
    K = dz.shape[1]
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.empty(idx.size)
    lib().cba_ref_wgrad_at(_pd(dz), _pf(x), N, C, H, W, K, R, S, stride, pad,
                           idx.ctypes.data_as(_lp), idx.size, _pd(out))
    return out


def dgrad_at(dz, Wt, H, W, stride, pad, idx, residual=None, prev_in=None, accumulate=False):
    """Sampled prev_delta elements (flat [N,C,H,W] indices) from dz."""
    dz = _f64(dz)
    Wt = np.ascontiguousarray(Wt, np.float32)
    K, C, R, S = Wt.shape
    N = dz.shape[0]
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.empty(idx.size)
    res = None if residual is None else np.ascontiguousarray(residual, np.float32)
    pin = None if prev_in is None else np.ascontiguousarray(prev_in, np.float32)
    lib().cba_ref_dgrad_at(_pd(dz), _pf(Wt), _pf(res), _pf(pin), int(bool(accumulate)), N, C, H,
                           W, K, R, S, stride, pad, idx.ctypes.data_as(_lp), idx.size, _pd(out))
    return out


# ------------------------------------------------ adjacent data-movement layers

def yolo_backward(l_delta, net_delta):
    """net_delta + l_delta (backward_yolo_layer); returns a new float64 array."""
    out = _f64(net_delta).copy()
    d = _f64(l_delta)
    lib().cba_ref_yolo_backward(_pd(d), d.size, _pd(out))
    return out


def route_backward(route_delta, input_sizes, input_deltas):
    """backward_route_layer: route_delta is [batch, sum(input_sizes)]; returns
    the input deltas (each [batch, input_sizes[i]]) after the additions."""
    rd = _f64(route_delta)
    batch = rd.shape[0]
    outs = [_f64(a).reshape(batch, -1).copy() for a in input_deltas]
    sizes = (ctypes.c_int * len(input_sizes))(*[int(v) for v in input_sizes])
    ptrs = (_dp * len(outs))(*[o.ctypes.data_as(_dp) for o in outs])
    lib().cba_ref_route_backward(_pd(rd), batch, len(outs), sizes, ptrs)
    return outs


def pooled_size(n, k, stride, pad):
    return lib().cba_ref_pooled_size(int(n), int(k), int(stride), int(pad))


def maxpool_backward(top_diff, mask, height, width):
    """PoolingLayer MAX Backward_cpu: top_diff and mask are [N, C, PH, PW] (mask:
    int32 flat index h * width + w in the plane); returns bottom_diff [N, C, H, W]."""
    td = _f64(top_diff)
    mk = np.ascontiguousarray(mask, dtype=np.int32)
    N, C, PH, PW = td.shape
    out = np.empty((N, C, int(height), int(width)))
    lib().cba_ref_maxpool_backward(_pd(td), mk.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                   N, C, int(height), int(width), PH, PW, _pd(out))
    return out
