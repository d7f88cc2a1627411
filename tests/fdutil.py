"""Test helpers: a float64 forward of one conv(+BN)+activation layer written
with library primitives (torch CPU conv2d, numpy reductions), and a central
finite-difference gradient.  These pin the oracle from outside: the oracle's
backward is compared with the numerical derivative of this forward."""
import numpy as np
import torch


def conv64(x, w, stride, pad, groups=1):
    with torch.no_grad():
        return torch.nn.functional.conv2d(torch.from_numpy(np.asarray(x, np.float64)),
                                          torch.from_numpy(np.asarray(w, np.float64)),
                                          stride=stride, padding=pad, groups=groups).numpy()


def _stair(v):
    n = np.floor(v)
    return np.where(n % 2 == 0, np.floor(v / 2.0), (v - n) + np.floor(v / 2.0))


# the forward activations (the *_activate functions of the YOLOv3 back-propagation
# page, §7), by activation code
_ACT_FWD = {
    0: lambda v: v,                                                   # linear
    1: lambda v: np.where(v > 0, v, 0.1 * v),                         # leaky
    2: lambda v: 1.0 / (1.0 + np.exp(-v)),                            # logistic
    3: lambda v: v * (v > 0),                                         # relu
    4: lambda v: np.where(v > 0, v, 0.01 * v),                        # relie
    5: lambda v: v * (v > 0) + 0.1 * v,                               # ramp
    6: lambda v: (np.exp(2 * v) - 1) / (np.exp(2 * v) + 1),           # tanh
    7: lambda v: np.where(v < -4, 0.01 * (v + 4),
                          np.where(v > 4, 0.01 * (v - 4) + 1, 0.125 * v + 0.5)),   # plse
    8: lambda v: (v >= 0) * v + (v < 0) * (np.exp(v) - 1),            # elu
    9: lambda v: (v >= 0) * 1.0507 * v + (v < 0) * 1.0507 * 1.6732 * (np.exp(v) - 1),  # selu
    10: lambda v: np.where(v < 0, 0.001 * v, np.where(v > 1, 0.001 * (v - 1) + 1, v)),  # lhtan
    11: lambda v: np.clip(v, -1.0, 1.0),                              # hardtan
    12: lambda v: 2.0 / (1.0 + np.exp(-v)) - 1,                       # loggy
    13: _stair,                                                       # stair
}

# where each forward is not differentiable
ACT_KINKS = {1: [0.0], 3: [0.0], 4: [0.0], 5: [0.0], 7: [-4.0, 4.0], 8: [0.0], 9: [0.0],
             10: [0.0, 1.0], 11: [-1.0, 1.0], 13: "integers"}


def act_fwd(act, v):
    return _ACT_FWD[act](np.asarray(v, np.float64))


def min_kink_distance(act, v):
    """Distance of each pre-activation value from the activation's kinks."""
    v = np.asarray(v, np.float64)
    k = ACT_KINKS.get(act)
    if k is None:
        return np.full(v.shape, np.inf)
    if k == "integers":
        return np.abs(v - np.round(v))
    return np.min(np.abs(v[..., None] - np.asarray(k)), axis=-1)


def layer_forward(x, w, gamma, beta, *, stride, pad, act, bn, eps, stats=None, groups=1):
    """Forward of the layer: z = conv(x, w); BN with the batch statistics
    (biased variance) if bn, or with the fixed (mean, var) of ``stats`` (frozen
    statistics: constants of the forward); then scale, shift and activation.
    Without BN, beta is the conv bias.  Returns (z, mean, var, pre_activation,
    output)."""
    z = conv64(x, w, stride, pad, groups)
    if bn and stats is not None:
        mean, var = (np.asarray(a, np.float64) for a in stats)
        xh = (z - mean[None, :, None, None]) / np.sqrt(var[None, :, None, None] + eps)
        pre = gamma[None, :, None, None] * xh + beta[None, :, None, None]
    elif bn:
        mean = z.mean(axis=(0, 2, 3))
        var = ((z - mean[None, :, None, None]) ** 2).mean(axis=(0, 2, 3))
        xh = (z - mean[None, :, None, None]) / np.sqrt(var[None, :, None, None] + eps)
        pre = gamma[None, :, None, None] * xh + beta[None, :, None, None]
    else:
        mean = var = None
        pre = z + beta[None, :, None, None]
    return z, mean, var, pre, act_fwd(act, pre)


def central_diff(f, x, h_rel=1e-6, h_abs=1e-7):
    """Central finite differences of the scalar function f at every element of x."""
    x = np.array(x, dtype=np.float64, copy=True)
    g = np.empty_like(x)
    flat = x.reshape(-1)
    gf = g.reshape(-1)
    for i in range(flat.size):
        v = flat[i]
        h = max(abs(v) * h_rel, h_abs) * 100.0
        flat[i] = v + h
        fp = f(x)
        flat[i] = v - h
        fm = f(x)
        flat[i] = v
        gf[i] = (fp - fm) / (2 * h)
    return g
