"""Thin ctypes binding of libcba's C ABI (``include/cba.h``).

Argument marshalling only: every step of the backward runs in the CUDA
library.  Tensors are passed as device pointers (``torch.Tensor.data_ptr()``
or plain integers); streams as ``cudaStream_t`` handles (default: torch's
current stream).  There is no CPU path: if ``libcba.so`` is missing the
binding raises instead of computing anything.
"""
import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcba.so")

CBA_OK = 0
CBA_ERR_ARG = -1
CBA_ERR_UNSUPPORTED = -2
CBA_ERR_ALIGN = -3
CBA_ERR_WORKSPACE = -4
CBA_ERR_CUDA = -5
CBA_ERR_DEVICE_TIMEOUT = -6
CBA_ERR_SCRATCH_LIMIT = -7
CBA_NOALLOC_MAX_K = 16384

CBA_ACT_LINEAR = 0
CBA_ACT_LEAKY = 1
CBA_ACT_LOGISTIC = 2
CBA_ACT_RELU = 3
CBA_ACT_RELIE = 4
CBA_ACT_RAMP = 5
CBA_ACT_TANH = 6
CBA_ACT_PLSE = 7
CBA_ACT_ELU = 8
CBA_ACT_SELU = 9
CBA_ACT_LHTAN = 10
CBA_ACT_HARDTAN = 11
CBA_ACT_LOGGY = 12
CBA_ACT_STAIR = 13
ACT_NAMES = {CBA_ACT_LINEAR: "linear", CBA_ACT_LEAKY: "leaky", CBA_ACT_LOGISTIC: "logistic",
             CBA_ACT_RELU: "relu", CBA_ACT_RELIE: "relie", CBA_ACT_RAMP: "ramp",
             CBA_ACT_TANH: "tanh", CBA_ACT_PLSE: "plse", CBA_ACT_ELU: "elu",
             CBA_ACT_SELU: "selu", CBA_ACT_LHTAN: "lhtan", CBA_ACT_HARDTAN: "hardtan",
             CBA_ACT_LOGGY: "loggy", CBA_ACT_STAIR: "stair"}
CBA_MATH_TF32 = 0
CBA_MATH_FFMA = 1

# every symbol include/cba.h declares
EXPORTS = ("cba_workspace_bytes", "cba_workspace_bytes_ex", "cba_workspace_bytes_grouped",
           "cba_conv_bn_act_backward_grouped", "cba_conv_bn_act_backward_grouped_traced",
           "cba_conv_bn_act_backward", "cba_conv_bn_act_backward_traced",
           "cba_get_status", "cba_bn_act_backward_noalloc",
           "cba_selftest_bounded_wait", "cba_yolo_backward", "cba_route_backward",
           "cba_pooled_size", "cba_maxpool_backward", "cba_error_string", "cba_last_cuda_error",
           "cba_version", "cba_plan_info")
CBA_ROUTE_MAX_INPUTS = 8
CBA_WS_RECOMPUTE_Z = 1
CBA_PHASE_EVENTS = 5
CBA_PATH_FFMA = 0
CBA_PATH_TC_ROWS = 1
CBA_PATH_TC_BATCH_INNER = 2
CBA_PATH_TC_GEMM_1X1 = 3


class cba_desc_t(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("C", ctypes.c_int), ("H", ctypes.c_int),
                ("W", ctypes.c_int), ("K", ctypes.c_int), ("R", ctypes.c_int),
                ("S", ctypes.c_int), ("stride", ctypes.c_int), ("pad", ctypes.c_int),
                ("act", ctypes.c_int), ("batch_normalize", ctypes.c_int),
                ("accumulate", ctypes.c_int), ("eps", ctypes.c_float), ("math", ctypes.c_int)]


class cba_plan_info_t(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("layout_bytes_read", ctypes.c_longlong),
                ("layout_bytes_written", ctypes.c_longlong)]


class cba_pool_desc_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("N", "C", "H", "W", "kernel_h", "kernel_w",
                                              "stride_h", "stride_w", "pad_h", "pad_w")]


class CbaError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {cba_error_string(code)} (code {code})")
        self.code = code


_lib = None


def load(path=LIB_PATH):
    """Load libcba.so.  Raises if it has not been built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libcba.so not built ({path}); run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    L.cba_workspace_bytes.restype = sz
    L.cba_workspace_bytes.argtypes = [ctypes.POINTER(cba_desc_t)]
    L.cba_workspace_bytes_grouped.restype = sz
    L.cba_workspace_bytes_grouped.argtypes = [ctypes.POINTER(cba_desc_t), ctypes.c_int,
                                              ctypes.c_uint]
    L.cba_conv_bn_act_backward_grouped.restype = ctypes.c_int
    L.cba_conv_bn_act_backward_grouped.argtypes = ([ctypes.POINTER(cba_desc_t), ctypes.c_int] +
                                                   [vp] * 15 + [sz, vp])
    L.cba_conv_bn_act_backward_grouped_traced.restype = ctypes.c_int
    L.cba_conv_bn_act_backward_grouped_traced.argtypes = (
        [ctypes.POINTER(cba_desc_t), ctypes.c_int] + [vp] * 15 +
        [sz, vp, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int)])
    L.cba_workspace_bytes_ex.restype = sz
    L.cba_workspace_bytes_ex.argtypes = [ctypes.POINTER(cba_desc_t), ctypes.c_uint]
    L.cba_conv_bn_act_backward.restype = ctypes.c_int
    L.cba_conv_bn_act_backward.argtypes = [ctypes.POINTER(cba_desc_t)] + [vp] * 15 + [sz, vp]
    L.cba_conv_bn_act_backward_traced.restype = ctypes.c_int
    L.cba_conv_bn_act_backward_traced.argtypes = (
        [ctypes.POINTER(cba_desc_t)] + [vp] * 15 + [sz, vp, ctypes.POINTER(ctypes.c_void_p),
                                                    ctypes.POINTER(ctypes.c_int)])
    L.cba_bn_act_backward_noalloc.restype = ctypes.c_int
    L.cba_bn_act_backward_noalloc.argtypes = [ctypes.POINTER(cba_desc_t)] + [vp] * 10
    L.cba_get_status.restype = ctypes.c_int
    L.cba_get_status.argtypes = [vp, sz, vp]
    L.cba_selftest_bounded_wait.restype = ctypes.c_int
    L.cba_selftest_bounded_wait.argtypes = [vp, sz, ctypes.c_uint, vp]
    L.cba_yolo_backward.restype = ctypes.c_int
    L.cba_yolo_backward.argtypes = [vp, vp, ctypes.c_longlong, vp]
    L.cba_route_backward.restype = ctypes.c_int
    L.cba_route_backward.argtypes = [vp, ctypes.c_int, ctypes.c_int,
                                     ctypes.POINTER(ctypes.c_longlong),
                                     ctypes.POINTER(ctypes.c_void_p), vp]
    L.cba_pooled_size.restype = ctypes.c_int
    L.cba_pooled_size.argtypes = [ctypes.c_int] * 4
    L.cba_maxpool_backward.restype = ctypes.c_int
    L.cba_maxpool_backward.argtypes = [ctypes.POINTER(cba_pool_desc_t), vp, vp, vp, vp]
    L.cba_error_string.restype = ctypes.c_char_p
    L.cba_error_string.argtypes = [ctypes.c_int]
    L.cba_last_cuda_error.restype = ctypes.c_int
    L.cba_version.restype = ctypes.c_int
    L.cba_plan_info.restype = ctypes.c_int
    L.cba_plan_info.argtypes = [ctypes.POINTER(cba_desc_t), ctypes.c_int, ctypes.c_int,
                                ctypes.POINTER(cba_plan_info_t)]
    _lib = L
    return L


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _bytes(t):
    if isinstance(t, int):
        raise TypeError("pass the workspace as a tensor, or (pointer, nbytes)")
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_desc(N, C, H, W, K, R, S, stride=1, pad=0, act=CBA_ACT_LEAKY, batch_normalize=1,
              accumulate=0, eps=1e-5, math=CBA_MATH_TF32):
    return cba_desc_t(N, C, H, W, K, R, S, stride, pad, act, int(batch_normalize),
                      int(accumulate), eps, math)


def cba_workspace_bytes(desc):
    return load().cba_workspace_bytes(ctypes.byref(desc))


def cba_workspace_bytes_ex(desc, flags):
    return load().cba_workspace_bytes_ex(ctypes.byref(desc), int(flags))


def cba_workspace_bytes_grouped(desc, groups, flags=0):
    return load().cba_workspace_bytes_grouped(ctypes.byref(desc), int(groups), int(flags))


def cba_conv_bn_act_backward_grouped(desc, groups, x, output, z, delta, W, gamma, mean, var,
                                     residual, dW, db, dgamma, prev_delta, dz_out, workspace,
                                     workspace_bytes=None, stream=None, check=True):
    """Grouped-convolution layer backward (W, dW [K, C/groups, R, S])."""
    wsb = _bytes(workspace) if workspace_bytes is None else int(workspace_bytes)
    rc = load().cba_conv_bn_act_backward_grouped(
        ctypes.byref(desc), int(groups), _ptr(x), _ptr(output), _ptr(z), _ptr(delta), _ptr(W),
        _ptr(gamma), _ptr(mean), _ptr(var), _ptr(residual), _ptr(dW), _ptr(db), _ptr(dgamma),
        _ptr(prev_delta), _ptr(dz_out), _ptr(workspace), wsb, _stream(stream))
    if check and rc != CBA_OK:
        raise CbaError(rc, "cba_conv_bn_act_backward_grouped")
    return rc


def _events(events):
    """None, or a C array of the CUDA events of CBA_PHASE_EVENTS torch.cuda.Event."""
    if events is None:
        return None
    assert len(events) == CBA_PHASE_EVENTS
    for e in events:
        if e.cuda_event == 0:  # torch creates the CUDA event on its first record
            e.record()
    return (ctypes.c_void_p * CBA_PHASE_EVENTS)(*[e.cuda_event for e in events])


def cba_conv_bn_act_backward_grouped_traced(desc, groups, x, output, z, delta, W, gamma, mean,
                                            var, residual, dW, db, dgamma, prev_delta, dz_out,
                                            workspace, workspace_bytes=None, stream=None,
                                            events=None, check=True):
    """As cba_conv_bn_act_backward_grouped, with ``events`` as for
    cba_conv_bn_act_backward_traced; returns (rc, kernels enqueued)."""
    wsb = _bytes(workspace) if workspace_bytes is None else int(workspace_bytes)
    n = ctypes.c_int(0)
    rc = load().cba_conv_bn_act_backward_grouped_traced(
        ctypes.byref(desc), int(groups), _ptr(x), _ptr(output), _ptr(z), _ptr(delta), _ptr(W),
        _ptr(gamma), _ptr(mean), _ptr(var), _ptr(residual), _ptr(dW), _ptr(db), _ptr(dgamma),
        _ptr(prev_delta), _ptr(dz_out), _ptr(workspace), wsb, _stream(stream), _events(events),
        ctypes.byref(n))
    if check and rc != CBA_OK:
        raise CbaError(rc, "cba_conv_bn_act_backward_grouped_traced")
    return rc, n.value


def cba_conv_bn_act_backward(desc, x, output, z, delta, W, gamma, mean, var, residual, dW, db,
                             dgamma, prev_delta, dz_out, workspace, workspace_bytes=None,
                             stream=None, check=True):
    """Enqueue one layer backward.  Returns the C return code; raises CbaError
    on a non-zero code when ``check``."""
    wsb = _bytes(workspace) if workspace_bytes is None else int(workspace_bytes)
    rc = load().cba_conv_bn_act_backward(
        ctypes.byref(desc), _ptr(x), _ptr(output), _ptr(z), _ptr(delta), _ptr(W), _ptr(gamma),
        _ptr(mean), _ptr(var), _ptr(residual), _ptr(dW), _ptr(db), _ptr(dgamma),
        _ptr(prev_delta), _ptr(dz_out), _ptr(workspace), wsb, _stream(stream))
    if check and rc != CBA_OK:
        raise CbaError(rc, "cba_conv_bn_act_backward")
    return rc


def cba_conv_bn_act_backward_traced(desc, x, output, z, delta, W, gamma, mean, var, residual,
                                    dW, db, dgamma, prev_delta, dz_out, workspace,
                                    workspace_bytes=None, stream=None, events=None, check=True):
    """As cba_conv_bn_act_backward; ``events`` is None or 5 torch.cuda.Event
    (created with enable_timing=True) recorded between the phases.  Returns
    (code, number of kernels enqueued)."""
    wsb = _bytes(workspace) if workspace_bytes is None else int(workspace_bytes)
    ev = _events(events)
    n = ctypes.c_int(0)
    rc = load().cba_conv_bn_act_backward_traced(
        ctypes.byref(desc), _ptr(x), _ptr(output), _ptr(z), _ptr(delta), _ptr(W), _ptr(gamma),
        _ptr(mean), _ptr(var), _ptr(residual), _ptr(dW), _ptr(db), _ptr(dgamma),
        _ptr(prev_delta), _ptr(dz_out), _ptr(workspace), wsb, _stream(stream), ev,
        ctypes.byref(n))
    if check and rc != CBA_OK:
        raise CbaError(rc, "cba_conv_bn_act_backward_traced")
    return rc, n.value


def cba_bn_act_backward_noalloc(desc, output, z, delta, gamma, mean, var, db, dgamma, dz_out,
                                stream=None, check=True):
    """Enqueue the activation-gradient + BN-backward pass (db, dgamma, dz)
    without a workspace; the library uses its own static device scratch.
    Returns the C return code; raises CbaError on a non-zero code when
    ``check``."""
    rc = load().cba_bn_act_backward_noalloc(
        ctypes.byref(desc), _ptr(output), _ptr(z), _ptr(delta), _ptr(gamma), _ptr(mean),
        _ptr(var), _ptr(db), _ptr(dgamma), _ptr(dz_out), _stream(stream))
    if check and rc != CBA_OK:
        raise CbaError(rc, "cba_bn_act_backward_noalloc")
    return rc


def cba_plan_info(desc, groups=1, with_prev=True):
    """(path, layout bytes read, layout bytes written) of a call with this
    descriptor; raises CbaError for a descriptor the call would refuse."""
    info = cba_plan_info_t()
    rc = load().cba_plan_info(ctypes.byref(desc), int(groups), int(bool(with_prev)),
                              ctypes.byref(info))
    if rc != CBA_OK:
        raise CbaError(rc, "cba_plan_info")
    return info.path, info.layout_bytes_read, info.layout_bytes_written


def cba_get_status(workspace, workspace_bytes=None, stream=None):
    wsb = _bytes(workspace) if workspace_bytes is None else int(workspace_bytes)
    return load().cba_get_status(_ptr(workspace), wsb, _stream(stream))


def cba_selftest_bounded_wait(workspace, timeout_us, workspace_bytes=None, stream=None):
    wsb = _bytes(workspace) if workspace_bytes is None else int(workspace_bytes)
    return load().cba_selftest_bounded_wait(_ptr(workspace), wsb, int(timeout_us),
                                            _stream(stream))


def cba_error_string(code):
    return load().cba_error_string(int(code)).decode()


def cba_last_cuda_error():
    return load().cba_last_cuda_error()


def cba_version():
    return load().cba_version()


# ------------------------------------------------ data-movement layers

def _checked(rc, what, check):
    if check and rc != CBA_OK:
        raise CbaError(rc, what)
    return rc


def cba_yolo_backward(l_delta, net_delta, n=None, stream=None, check=True):
    """net_delta += l_delta over n elements (default: all of l_delta)."""
    n = l_delta.numel() if n is None else int(n)
    rc = load().cba_yolo_backward(_ptr(l_delta), _ptr(net_delta), n, _stream(stream))
    return _checked(rc, "cba_yolo_backward", check)


def cba_route_backward(route_delta, input_deltas, batch=None, stream=None, check=True):
    """Split route_delta [batch, outputs] back onto the input deltas (tensors of
    batch * size_i elements each), adding."""
    batch = route_delta.shape[0] if batch is None else int(batch)
    n = len(input_deltas)
    sizes = (ctypes.c_longlong * n)(*[t.numel() // batch for t in input_deltas])
    ptrs = (ctypes.c_void_p * n)(*[_ptr(t) for t in input_deltas])
    rc = load().cba_route_backward(_ptr(route_delta), batch, n, sizes, ptrs, _stream(stream))
    return _checked(rc, "cba_route_backward", check)


def cba_pooled_size(n, kernel, stride, pad):
    return load().cba_pooled_size(int(n), int(kernel), int(stride), int(pad))


def make_pool_desc(N, C, H, W, kernel, stride, pad=0):
    return cba_pool_desc_t(N, C, H, W, kernel, kernel, stride, stride, pad, pad)


def cba_maxpool_backward(desc, top_diff, mask, bottom_diff, stream=None, check=True):
    """bottom_diff = scatter of top_diff to the mask's indices (gather form)."""
    rc = load().cba_maxpool_backward(ctypes.byref(desc), _ptr(top_diff), _ptr(mask),
                                     _ptr(bottom_diff), _stream(stream))
    return _checked(rc, "cba_maxpool_backward", check)
