"""Device-side convenience around the C ABI: uploads one layer's inputs to
the GPU, owns its output and workspace tensors, and enqueues the backward.

PyTorch is used only for device memory and streams; every arithmetic step
runs in libcba's kernels.
"""
import torch

from . import _binding as B


def _dev(a, device):
    if a is None:
        return None
    return torch.from_numpy(a).to(device=device, dtype=torch.float32).contiguous()


class DeviceLayer:
    """One layer call's device buffers.

    ``layer`` is an input dict from ``inputs.make_layer`` / ``make_config``
    (numpy fp32 arrays).  ``math`` is CBA_MATH_TF32 or CBA_MATH_FFMA.
    Outputs dW, db, dgamma start at zero (they accumulate); prev_delta starts
    at zero, or at ``prev_init`` when given."""

    def __init__(self, layer, math=B.CBA_MATH_TF32, device="cuda", accumulate=None,
                 with_prev=True, with_residual=True, prev_init=None, want_dz=False,
                 z_free=False):
        g = layer["geom"]
        self.geom = g
        self.layer = layer
        acc = layer["accumulate"] if accumulate is None else int(accumulate)
        self.desc = B.make_desc(g.N, g.C, g.H, g.W, g.K, g.R, g.S, g.stride, g.pad,
                                act=layer["act"], batch_normalize=int(layer["bn"]),
                                accumulate=acc, eps=layer["eps"], math=math)
        self.x = _dev(layer["x"], device)
        self.W = _dev(layer["W"], device)
        self.output = _dev(layer["output"], device) if layer["act"] != B.CBA_ACT_LINEAR else None
        # z_free: the library recomputes z = conv(x, W) in the workspace
        self.z = _dev(layer["z"], device) if layer["bn"] and not z_free else None
        self.delta = _dev(layer["delta"], device)
        self.gamma = _dev(layer["gamma"], device) if layer["bn"] else None
        self.mean = _dev(layer["mean"], device) if layer["bn"] else None
        self.var = _dev(layer["var"], device) if layer["bn"] else None
        res = layer.get("residual") if with_residual else None
        self.residual = _dev(res, device)
        f = dict(device=device, dtype=torch.float32)
        self.groups = int(layer.get("groups", 1))
        self.dW = torch.zeros((g.K, g.C // self.groups, g.R, g.S), **f)
        self.db = torch.zeros(g.K, **f)
        self.dgamma = torch.zeros(g.K, **f) if layer["bn"] else None
        self.prev = None
        if with_prev:
            self.prev = (torch.zeros((g.N, g.C, g.H, g.W), **f) if prev_init is None
                         else _dev(prev_init, device))
        self.dz = torch.empty((g.N, g.K, g.P, g.Q), **f) if want_dz else None
        flags = B.CBA_WS_RECOMPUTE_Z if z_free else 0
        nbytes = B.cba_workspace_bytes_grouped(self.desc, self.groups, flags)
        if nbytes == 0:
            raise B.CbaError(B.CBA_ERR_ARG, "cba_workspace_bytes")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def zero_outputs(self):
        self.dW.zero_()
        self.db.zero_()
        if self.dgamma is not None:
            self.dgamma.zero_()
        if self.prev is not None:
            self.prev.zero_()

    def run(self, stream=None, check=True):
        if self.groups > 1:
            return B.cba_conv_bn_act_backward_grouped(
                self.desc, self.groups, self.x, self.output, self.z, self.delta, self.W,
                self.gamma, self.mean, self.var, self.residual, self.dW, self.db, self.dgamma,
                self.prev, self.dz, self.workspace, stream=stream, check=check)
        return B.cba_conv_bn_act_backward(self.desc, self.x, self.output, self.z, self.delta,
                                          self.W, self.gamma, self.mean, self.var, self.residual,
                                          self.dW, self.db, self.dgamma, self.prev, self.dz,
                                          self.workspace, stream=stream, check=check)

    def run_traced(self, events=None, stream=None):
        """Enqueue with 5 phase events (see cba_conv_bn_act_backward_traced);
        returns the number of kernels enqueued."""
        if self.groups > 1:
            _, n = B.cba_conv_bn_act_backward_grouped_traced(
                self.desc, self.groups, self.x, self.output, self.z, self.delta, self.W,
                self.gamma, self.mean, self.var, self.residual, self.dW, self.db, self.dgamma,
                self.prev, self.dz, self.workspace, stream=stream, events=events)
            return n
        _, n = B.cba_conv_bn_act_backward_traced(
            self.desc, self.x, self.output, self.z, self.delta, self.W, self.gamma, self.mean,
            self.var, self.residual, self.dW, self.db, self.dgamma, self.prev, self.dz,
            self.workspace, stream=stream, events=events)
        return n

    def status(self, stream=None):
        return B.cba_get_status(self.workspace, stream=stream)

    def results(self):
        """Host float64 copies of the outputs."""
        out = dict(dW=self.dW, db=self.db, dgamma=self.dgamma, prev_delta=self.prev, dz=self.dz)
        return {k: (None if v is None else v.double().cpu().numpy()) for k, v in out.items()}


def capture_graph(fn, warmup=2):
    """Capture `fn()` -- a sequence of library calls on the current stream,
    e.g. ``layer.run`` -- into a CUDA graph and return it (replay it with
    ``graph.replay()``).  The library calls only enqueue stream-ordered work
    on caller-provided buffers, so a replay repeats them on the same buffers
    without any host-side launch cost.  `fn` runs `warmup` times first,
    outside the capture (the first call on a device sets up per-kernel
    attributes)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warmup):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph
