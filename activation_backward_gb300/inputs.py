"""Seeded synthetic inputs for the conv + BN + activation backward.

This module only *generates inputs*: it draws the seeded tensors and runs the
layer's FORWARD pass (convolution, batch statistics, scale, activation) to
produce the cached tensors a backward call consumes (``z``, ``mean``, ``var``,
``output``).  It contains none of the backward arithmetic.  Both the CUDA path
and the oracle take their inputs from here, so both see identical fp32 bits.

Workloads (shapes from the pages):

* ``lenet_conv2``  -- caffe LeNet conv2 ("LeNet反向过程", 第四层 Convolution):
  bottom (64,20,12,12) -> top (64,50,8,8), 5x5 kernels, no BN, linear.
* ``darknet_3x3``  -- darknet 3x3 conv + BN + leaky, 16 x 64->128 at 52x52.
* ``yolov3_down``  -- YOLOv3 downsampling conv, 3x3 stride 2, 256->512, 52->26.
* ``yolo_head_1x1`` -- YOLO head 1x1 conv, 1024->255 at 13x13, no BN, linear,
  with a 90%-zero delta (the sparse detection-loss gradient pattern).
* ``residual_block`` -- darknet residual block at 26x26: 1x1 512->256 BN+leaky,
  then 3x3 256->512 BN+leaky, plus the shortcut (two layer calls).

Random numbers come from numpy's PCG64 (``default_rng(seed)``), which gives
the same stream on every platform; the draws happen in a fixed order
(x, W, gamma, delta, mask, residual).  "N(0, v)" means variance v.  The forward
convolution runs in float64 (torch CPU ``conv2d``, a library call) and is then
rounded to fp32; the batch statistics are the biased (1/m) mean and variance
of that fp32 ``z``; the BN shift beta is 0.
"""
from dataclasses import dataclass, replace

import numpy as np

ACT_LINEAR = 0
ACT_LEAKY = 1
EPS = 1e-5


@dataclass(frozen=True)
class Geometry:
    N: int
    C: int
    H: int
    W: int
    K: int
    R: int
    S: int
    stride: int = 1
    pad: int = 0

    @property
    def P(self):
        return (self.H + 2 * self.pad - self.R) // self.stride + 1

    @property
    def Q(self):
        return (self.W + 2 * self.pad - self.S) // self.stride + 1

    def gemm_flops(self):
        """Algorithmic FLOPs of ONE of the two GEMMs (wgrad or dgrad):
        2 * N * K * C * R * S * P * Q (multiply-adds counted as 2)."""
        return 2 * self.N * self.K * self.C * self.R * self.S * self.P * self.Q


@dataclass(frozen=True)
class LayerSpec:
    name: str
    geom: Geometry
    act: int
    bn: bool
    accumulate: int = 0
    dist: str = "normal"  # "uniform" for LeNet
    sparse_delta: float = 0.0  # fraction of zero delta entries


CONFIGS = {
    1: LayerSpec("lenet_conv2", Geometry(64, 20, 12, 12, 50, 5, 5, 1, 0), ACT_LINEAR, False,
                 dist="uniform"),
    2: LayerSpec("darknet_3x3", Geometry(16, 64, 52, 52, 128, 3, 3, 1, 1), ACT_LEAKY, True),
    3: LayerSpec("yolov3_down", Geometry(16, 256, 52, 52, 512, 3, 3, 2, 1), ACT_LEAKY, True),
    4: LayerSpec("yolo_head_1x1", Geometry(64, 1024, 13, 13, 255, 1, 1, 1, 0), ACT_LINEAR, False,
                 sparse_delta=0.9),
    # config 5 is a block of two layers; these are its two convolutions
    5: LayerSpec("residual_block", Geometry(32, 512, 26, 26, 256, 1, 1, 1, 0), ACT_LEAKY, True),
}
BLOCK_CONV2 = Geometry(32, 256, 26, 26, 512, 3, 3, 1, 1)


def seed_of(config_id):
    return 1000 + int(config_id)


def _forward_conv64(x, w, stride, pad, groups=1):
    import torch
    with torch.no_grad():
        z = torch.nn.functional.conv2d(torch.from_numpy(x.astype(np.float64)),
                                       torch.from_numpy(w.astype(np.float64)), stride=stride,
                                       padding=pad, groups=groups)
    return z.numpy()


def _leaky(v):
    return np.where(v > 0, v, 0.1 * v)


def _bn_forward(z32, gamma, act, eps=EPS):
    """Forward batch-norm (training mode) + activation.  Returns mean, var
    (biased) and the post-activation output, all fp32."""
    z = z32.astype(np.float64)
    mean = z.mean(axis=(0, 2, 3))
    var = ((z - mean[None, :, None, None]) ** 2).mean(axis=(0, 2, 3))
    mean32, var32 = mean.astype(np.float32), var.astype(np.float32)
    xh = (z - mean32.astype(np.float64)[None, :, None, None]) / np.sqrt(
        var32.astype(np.float64)[None, :, None, None] + np.float64(np.float32(eps)))
    y = gamma.astype(np.float64)[None, :, None, None] * xh  # beta = 0
    out = _leaky(y) if act == ACT_LEAKY else y
    return mean32, var32, out.astype(np.float32)


def _draw(rng, dist, shape, var=1.0):
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, size=shape).astype(np.float32)
    return (rng.standard_normal(size=shape) * np.sqrt(var)).astype(np.float32)


def make_layer(spec, seed, *, batch=None, residual=False, x=None, delta_var=0.01, groups=1):
    """Inputs of one layer call.  Returns a dict with the geometry and flags
    and fp32 arrays x, W, gamma, z, mean, var, output, delta, residual.

    ``batch`` overrides N (a smaller case with the same channel and spatial
    geometry); ``x`` supplies the layer input (for the block's second layer)."""
    g = spec.geom if batch is None else replace(spec.geom, N=int(batch))
    rng = np.random.default_rng(seed)
    if x is None:
        x = _draw(rng, spec.dist, (g.N, g.C, g.H, g.W))
    Cg = g.C // groups  # input channels a filter sees (grouped convolution)
    fan_in = Cg * g.R * g.S
    if spec.dist == "uniform":
        W = _draw(rng, "uniform", (g.K, Cg, g.R, g.S))
    else:
        W = _draw(rng, "normal", (g.K, Cg, g.R, g.S), var=2.0 / fan_in)  # He init
    gamma = rng.uniform(0.5, 1.5, size=g.K).astype(np.float32) if spec.bn else None
    if spec.dist == "uniform":
        delta = _draw(rng, "uniform", (g.N, g.K, g.P, g.Q))
    else:
        delta = _draw(rng, "normal", (g.N, g.K, g.P, g.Q), var=delta_var)
    if spec.sparse_delta > 0:
        keep = rng.uniform(size=delta.shape) >= spec.sparse_delta
        delta = (delta * keep).astype(np.float32)
    res = _draw(rng, "normal", (g.N, g.C, g.H, g.W), var=0.01) if residual else None

    z = _forward_conv64(x, W, g.stride, g.pad, groups).astype(np.float32)
    if spec.bn:
        mean, var, output = _bn_forward(z, gamma, spec.act)
    else:
        mean = var = None
        output = (_leaky(z.astype(np.float64)) if spec.act == ACT_LEAKY else z).astype(np.float32)
        z = None  # the backward needs the pre-BN output only with BN
    return dict(name=spec.name, geom=g, act=spec.act, bn=spec.bn, accumulate=spec.accumulate,
                eps=EPS, x=x, W=W, gamma=gamma, z=z, mean=mean, var=var, output=output,
                delta=delta, residual=res, groups=int(groups))


def make_grouped_config(config_id, groups, *, batch=None):
    """A one-call workload (configs 1-4) as a grouped convolution: the same
    geometry with W [K, C/groups, R, S]."""
    spec = CONFIGS[int(config_id)]
    layer = make_layer(spec, seed_of(config_id) + 31 * int(groups), batch=batch, groups=groups)
    return dict(layer, name=f"{spec.name} (groups {int(groups)})")


def _act_forward(act, v):
    """The forward activations (the *_activate functions of the YOLOv3
    back-propagation page, §7), float64, by activation code."""
    if act == 0:
        return v
    if act == 1:
        return _leaky(v)
    if act == 2:
        return 1.0 / (1.0 + np.exp(-v))
    if act == 3:
        return v * (v > 0)
    if act == 4:
        return np.where(v > 0, v, 0.01 * v)
    if act == 5:
        return v * (v > 0) + 0.1 * v
    if act == 6:
        return np.tanh(v)
    if act == 7:
        return np.where(v < -4, 0.01 * (v + 4), np.where(v > 4, 0.01 * (v - 4) + 1, 0.125 * v + 0.5))
    if act == 8:
        return np.where(v >= 0, v, np.expm1(np.minimum(v, 0)))
    if act == 9:
        return np.where(v >= 0, 1.0507 * v, 1.0507 * 1.6732 * np.expm1(np.minimum(v, 0)))
    if act == 10:
        return np.where(v < 0, 0.001 * v, np.where(v > 1, 0.001 * (v - 1) + 1, v))
    if act == 11:
        return np.clip(v, -1.0, 1.0)
    if act == 12:
        return 2.0 / (1.0 + np.exp(-v)) - 1
    if act == 13:
        n = np.floor(v)
        return np.where(n % 2 == 0, np.floor(v / 2.0), (v - n) + np.floor(v / 2.0))
    raise ValueError(f"unknown activation {act}")


def with_activation(layer, act):
    """The same layer call with another activation: ``output`` is recomputed as
    act(pre-activation).  The pre-activation is gamma * (z - mean) / sqrt(var +
    eps) for BN layers (beta = 0, as in make_layer), and is recovered from the
    linear or leaky output of a layer without BN."""
    if layer["bn"]:
        z = layer["z"].astype(np.float64)
        m = layer["mean"].astype(np.float64)[None, :, None, None]
        v = layer["var"].astype(np.float64)[None, :, None, None]
        pre = layer["gamma"].astype(np.float64)[None, :, None, None] * (z - m) / np.sqrt(
            v + np.float64(np.float32(layer["eps"])))
    else:
        y = layer["output"].astype(np.float64)
        pre = np.where(y > 0, y, y / 0.1) if layer["act"] == ACT_LEAKY else y
    out = _act_forward(int(act), pre).astype(np.float32)
    return dict(layer, act=int(act), output=out, name=f"{layer['name']} (act {int(act)})")


def with_frozen_stats(layer, seed):
    """The same layer call with frozen BN statistics (batch_normalize = 2): the
    mean is moved by up to half a standard deviation and the variance scaled
    by 0.5-2, per channel, so that they are not the batch's own.  Random draws
    only; the other tensors are shared with ``layer``."""
    if not layer["bn"]:
        raise ValueError("frozen statistics need a BN layer")
    rng = np.random.default_rng(seed)
    K = layer["geom"].K
    mean = layer["mean"] + rng.uniform(-0.5, 0.5, K) * np.sqrt(layer["var"])
    var = layer["var"] * rng.uniform(0.5, 2.0, K)
    return dict(layer, bn=2, mean=mean.astype(np.float32), var=var.astype(np.float32),
                name=layer["name"] + " (frozen stats)")


def make_config(config_id, *, batch=None):
    """The layer call(s) of one workload: a list of input dicts.

    Configs 1-4 are one call.  Config 5 (residual block) is two calls in
    backward order: the 3x3 conv (its delta is the block delta D, its input
    is the 1x1 conv's output), then the 1x1 conv (its prev_delta gets the
    shortcut residual D).  The 1x1 conv's incoming delta is, in the real block,
    the 3x3 conv's prev_delta; here it is its own seeded N(0, 0.01) draw so
    that each call can be checked on its own -- the chained block is built by
    ``chain_block``."""
    config_id = int(config_id)
    seed = seed_of(config_id)
    if config_id in (1, 2, 3, 4):
        return [make_layer(CONFIGS[config_id], seed, batch=batch)]
    if config_id != 5:
        raise ValueError(f"unknown config {config_id}")
    spec1 = CONFIGS[5]
    l1 = make_layer(spec1, seed, batch=batch)  # X, W1, gamma1, z1, y1 (its output)
    spec2 = LayerSpec("residual_block.conv2", BLOCK_CONV2, ACT_LEAKY, True)
    l2 = make_layer(spec2, seed + 100, batch=batch, x=l1["output"])
    # block delta D: the gradient at the block output (after the shortcut add)
    D = l2["delta"]
    l2 = dict(l2, name="residual_block.conv2")
    l1 = dict(l1, name="residual_block.conv1", residual=D)
    return [l2, l1]


def layer_bytes_reduce(layer):
    """Algorithmic bytes of the per-channel reduction pass: 4 B per element of
    delta, plus output (leaky) and z (BN)."""
    g = layer["geom"]
    m = g.N * g.K * g.P * g.Q
    n = 1 + (1 if layer["act"] == ACT_LEAKY else 0) + (1 if layer["bn"] else 0)
    return 4 * m * n


# ------------------------------------------------ adjacent data-movement layers

def pooled_size(n, k, stride, pad):
    """caffe PoolingLayer output size: ceil((n + 2 pad - k) / stride) + 1, one
    less when the last window would start in the bottom padding."""
    out = -(-(n + 2 * pad - k) // stride) + 1
    if pad > 0 and (out - 1) * stride >= n + pad:
        out -= 1
    return out


def make_pool_case(N, C, H, W, k, stride, pad, seed):
    """Inputs of a max-pooling backward: the forward's mask (flat index h * W + w
    of each window's first maximum in scan order, as caffe's forward records it)
    from a seeded bottom of distinct values, and a seeded top gradient."""
    rng = np.random.default_rng(seed)
    bottom = rng.permutation(N * C * H * W).reshape(N, C, H, W).astype(np.float64)
    bottom = (bottom / bottom.size - 0.5).astype(np.float32)
    PH, PW = pooled_size(H, k, stride, pad), pooled_size(W, k, stride, pad)
    mask = np.empty((N, C, PH, PW), np.int32)
    for ph in range(PH):
        h0, h1 = max(ph * stride - pad, 0), min(ph * stride - pad + k, H)
        for pw in range(PW):
            w0, w1 = max(pw * stride - pad, 0), min(pw * stride - pad + k, W)
            win = bottom[:, :, h0:h1, w0:w1].reshape(N, C, -1)
            a = np.argmax(win, axis=2)  # first maximum in scan order
            mask[:, :, ph, pw] = (h0 + a // (w1 - w0)) * W + (w0 + a % (w1 - w0))
    top_diff = (rng.standard_normal((N, C, PH, PW)) * 0.1).astype(np.float32)
    return dict(N=N, C=C, H=H, W=W, k=k, stride=stride, pad=pad, PH=PH, PW=PW,
                bottom=bottom, mask=mask, top_diff=top_diff)


def make_route_case(batch, input_sizes, seed):
    """Inputs of a route-layer backward: the route delta [batch, sum(sizes)] and
    the input layers' deltas [batch, size_i] the backward adds onto."""
    rng = np.random.default_rng(seed)
    outputs = int(sum(input_sizes))
    route_delta = (rng.standard_normal((batch, outputs)) * 0.1).astype(np.float32)
    deltas = [(rng.standard_normal((batch, int(s))) * 0.1).astype(np.float32)
              for s in input_sizes]
    return dict(batch=batch, input_sizes=[int(s) for s in input_sizes],
                route_delta=route_delta, input_deltas=deltas)
