"""Test helpers: a float64 forward of one conv(+BN)+activation layer written
with library primitives (torch CPU conv2d, numpy reductions), and a central
finite-difference gradient.  These pin the oracle from outside: the oracle's
backward is compared with the numerical derivative of this forward."""
import numpy as np
import torch


def conv64(x, w, stride, pad):
    with torch.no_grad():
        return torch.nn.functional.conv2d(torch.from_numpy(np.asarray(x, np.float64)),
                                          torch.from_numpy(np.asarray(w, np.float64)),
                                          stride=stride, padding=pad).numpy()


def act_fwd(act, v):
    if act == 0:
        return v
    if act == 1:
        return np.where(v > 0, v, 0.1 * v)
    if act == 2:
        return 1.0 / (1.0 + np.exp(-v))
    raise ValueError(act)


def layer_forward(x, w, gamma, beta, *, stride, pad, act, bn, eps, stats=None):
    """Forward of the layer: z = conv(x, w); BN with the batch statistics
    (biased variance) if bn, or with the fixed (mean, var) of ``stats`` (frozen
    statistics: constants of the forward); then scale, shift and activation.
    Without BN, beta is the conv bias.  Returns (z, mean, var, pre_activation,
    output)."""
    z = conv64(x, w, stride, pad)
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
