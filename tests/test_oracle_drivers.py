"""Pins of the oracle entry points the GPU parity tests call as checkers.

The GPU tests compare against two oracle drivers that the finite-difference
pins of test_oracle_pins.py do not reach directly:

- ``backward_dz`` (activation gradient + BN backward alone, fp32 inputs), the
  checker of db, dgamma and dz at full sizes and the source of the dz that the
  sampled weight / input gradients consume;
- the fp32-input chain driver (``conv_bn_act_backward`` without
  ``f64_inputs``), which every GPU parity test calls.

Each is pinned here against something other than itself: dz against central
differences of the layer's forward with respect to the BN input z (the BN
statistics recomputed from z inside the loss, as in training, or held fixed),
and each driver against the finite-difference-pinned fp64 chain on the same
values, bit for bit.  Sources: backward_convolutional_layer (§3.1) and
backward_batchnorm_layer with mean_delta_cpu / variance_delta_cpu /
normalize_delta_cpu (§4) of "YOLOv3反向传播原理 之 全流程源码分析"."""
import numpy as np
import pytest

from tests.fdutil import act_fwd, central_diff, layer_forward

# eps as the float the fp32 drivers widen, so both drivers see the same value
EPS = float(np.float32(1e-5))


def _rng(seed):
    return np.random.default_rng(seed)


def _bn_layer(seed, act, N=2, K=3, P=4, Q=5, frozen=False):
    """fp32 z, the forward's (mean, var) in fp32, gamma, beta, the fp32 output
    y = act(gamma * xhat + beta) and an fp32 incoming delta; redrawn until no
    pre-activation sits within 5e-3 of the activation's kink at 0."""
    for attempt in range(100):
        rng = _rng(seed + attempt)
        z = rng.standard_normal((N, K, P, Q)).astype(np.float32)
        z64 = z.astype(np.float64)
        if frozen:  # statistics that are not the batch's own
            mean = (z64.mean(axis=(0, 2, 3)) + rng.uniform(-0.5, 0.5, K)).astype(np.float32)
            var = (z64.var(axis=(0, 2, 3)) * rng.uniform(0.5, 2.0, K)).astype(np.float32)
        else:
            mean = z64.mean(axis=(0, 2, 3)).astype(np.float32)
            var = z64.var(axis=(0, 2, 3)).astype(np.float32)
        gamma = rng.uniform(0.5, 1.5, K).astype(np.float32)
        beta = rng.uniform(-0.3, 0.3, K).astype(np.float32)
        xh = (z64 - mean[None, :, None, None]) / np.sqrt(var[None, :, None, None] + EPS)
        pre = gamma[None, :, None, None] * xh + beta[None, :, None, None]
        if act != 0 and np.min(np.abs(pre)) < 5e-3:
            continue
        y = act_fwd(act, pre).astype(np.float32)
        delta = rng.standard_normal(z.shape).astype(np.float32)
        return z, mean, var, gamma, beta, y, delta
    raise RuntimeError("no draw clear of the kink")


@pytest.mark.parametrize("act", [0, 1, 8], ids=["linear", "leaky", "elu"])
@pytest.mark.parametrize("bn", [1, 2], ids=["batch", "frozen"])
def test_backward_dz_is_the_gradient_wrt_the_bn_input(ref, act, bn):
    """dz = dL/dz for L(z) = sum D * act(gamma * BN(z) + beta): with bn = 1 the
    batch mean and (biased) variance are recomputed from z inside L, so the
    mean_delta / variance_delta paths are exercised; with bn = 2 they are the
    fixed statistics.  db = sum delta' and dgamma = sum delta' * xhat are the
    gradients of L with respect to beta and gamma."""
    z, mean, var, gamma, beta, y, D = _bn_layer(40 + 3 * act + bn, act, frozen=(bn == 2))
    m64, v64 = mean.astype(np.float64), var.astype(np.float64)
    g64, b64 = gamma.astype(np.float64), beta.astype(np.float64)

    def forward(zv, g=g64, b=b64):
        if bn == 1:
            mu = zv.mean(axis=(0, 2, 3))
            va = ((zv - mu[None, :, None, None]) ** 2).mean(axis=(0, 2, 3))
        else:
            mu, va = m64, v64
        xh = (zv - mu[None, :, None, None]) / np.sqrt(va[None, :, None, None] + EPS)
        return float(np.sum(D * act_fwd(act, g[None, :, None, None] * xh + b[None, :, None, None])))

    z64 = z.astype(np.float64)
    dz, db, dg = ref.backward_dz(y, z, D, gamma, mean, var, act=act, batch_normalize=bn, eps=EPS)
    fd_z = central_diff(forward, z64)
    fd_b = central_diff(lambda v: forward(z64, b=v), b64)
    fd_g = central_diff(lambda v: forward(z64, g=v), g64)

    def close(a, b, tol):
        scale = max(np.max(np.abs(b)), 1e-12)
        assert np.max(np.abs(a - b)) <= tol * scale, (np.max(np.abs(a - b)), scale)

    # the fp32 statistics differ from the exact batch ones by ~1e-7 relative
    close(dz, fd_z, 2e-5)
    close(db, fd_b, 2e-6)
    close(dg, fd_g, 2e-6)


@pytest.mark.parametrize("act", [0, 1, 3], ids=["linear", "leaky", "relu"])
def test_backward_dz_without_bn_is_delta_times_the_activation_gradient(ref, act):
    """Without BN (backward_bias path): dz = dL/d(pre) for L = sum D * act(pre)
    and db = sum over (n, p, q) of it."""
    rng = _rng(70 + act)
    N, K, P, Q = 3, 4, 3, 5
    for _ in range(100):
        pre = rng.standard_normal((N, K, P, Q))
        if np.min(np.abs(pre)) > 5e-3:
            break
    y = act_fwd(act, pre).astype(np.float32)
    D = rng.standard_normal(pre.shape).astype(np.float32)
    dz, db, dg = ref.backward_dz(y, None, D, None, None, None, act=act, batch_normalize=0,
                                 eps=EPS)
    assert dg is None
    fd = central_diff(lambda v: float(np.sum(D * act_fwd(act, v))), pre)
    assert np.max(np.abs(dz - fd)) <= 1e-6 * np.max(np.abs(fd))
    assert np.allclose(db, fd.sum(axis=(0, 2, 3)), rtol=1e-6, atol=0)


@pytest.mark.parametrize("act", [0, 1, 8], ids=["linear", "leaky", "elu"])
@pytest.mark.parametrize("bn", [0, 1, 2], ids=["none", "batch", "frozen"])
def test_backward_dz_equals_the_chain_dz(ref, act, bn):
    """backward_dz and the full chain (dz_out) give identical dz, db and dgamma
    on the same fp32 inputs, and both accumulate db / dgamma onto given values."""
    z, mean, var, gamma, beta, y, D = _bn_layer(90 + 3 * act + bn, act, N=2, K=4, P=5, Q=5,
                                                frozen=(bn == 2))
    rng = _rng(500 + act + 10 * bn)
    N, K, P, Q = z.shape
    C = 3
    x = rng.standard_normal((N, C, P + 2, Q + 2)).astype(np.float32)
    w = (rng.standard_normal((K, C, 3, 3)) * 0.3).astype(np.float32)
    db0 = rng.standard_normal(K)
    dg0 = rng.standard_normal(K) if bn else None
    bnargs = (z, gamma, mean, var) if bn else (None, None, None, None)
    chain = ref.conv_bn_act_backward(x, y, bnargs[0], D, w, bnargs[1], bnargs[2], bnargs[3], None,
                                     stride=1, pad=0, act=act, batch_normalize=bn, accumulate=0,
                                     eps=EPS, db=db0, dgamma=dg0, want_prev=False, want_dz=True)
    dz, db, dg = ref.backward_dz(y, bnargs[0], D, bnargs[1], bnargs[2], bnargs[3], act=act,
                                 batch_normalize=bn, eps=EPS, db=db0, dgamma=dg0)
    assert np.array_equal(dz, chain["dz"])
    assert np.array_equal(db, chain["db"])
    if bn:
        assert np.array_equal(dg, chain["dgamma"])
    else:
        assert dg is None and chain["dgamma"] is None


DRIVER_CASES = [
    # N, C, H, W, K, R, S, stride, pad, groups, act, bn, residual, accumulate
    (2, 4, 7, 6, 6, 3, 3, 2, 1, 2, 1, 1, True, 1),
    (3, 3, 5, 5, 4, 3, 3, 1, 1, 1, 0, 0, True, 0),
    (2, 4, 6, 6, 4, 1, 1, 1, 0, 2, 8, 2, False, 1),
    (2, 2, 7, 7, 3, 5, 5, 1, 2, 1, 1, 1, True, 0),
]


@pytest.mark.parametrize("case", DRIVER_CASES, ids=[str(i) for i in range(len(DRIVER_CASES))])
def test_fp32_driver_equals_the_f64_driver(ref, case):
    """The fp32-input driver widens its inputs exactly and runs the fp64 chain:
    every output equals the fp64 driver's on the same values, bit for bit
    (a swapped or misrouted pointer in the wrapper fails this)."""
    N, C, H, W, K, R, S, st, pad, G, act, bn, res, acc = case
    rng = _rng(700 + DRIVER_CASES.index(case))
    f32 = lambda a: np.asarray(a, np.float32)  # noqa: E731
    x = f32(rng.standard_normal((N, C, H, W)))
    w = f32(rng.standard_normal((K, C // G, R, S)) * 0.4)
    P = (H + 2 * pad - R) // st + 1
    Q = (W + 2 * pad - S) // st + 1
    z = f32(rng.standard_normal((N, K, P, Q)))
    y = f32(rng.standard_normal((N, K, P, Q)))
    D = f32(rng.standard_normal((N, K, P, Q)))
    gamma = f32(rng.uniform(0.5, 1.5, K))
    mean = f32(rng.uniform(-0.2, 0.2, K))
    var = f32(rng.uniform(0.5, 1.5, K))
    residual = f32(rng.standard_normal(x.shape)) if res else None
    init = dict(dW=rng.standard_normal(w.shape), db=rng.standard_normal(K),
                dgamma=rng.standard_normal(K) if bn else None,
                prev_delta=rng.standard_normal(x.shape))
    args = (x, y, z if bn else None, D, w, gamma if bn else None, mean if bn else None,
            var if bn else None, residual)
    kw = dict(stride=st, pad=pad, act=act, batch_normalize=bn, accumulate=acc, eps=EPS, groups=G,
              want_dz=True, **init)
    a = ref.conv_bn_act_backward(*args, **kw)
    b = ref.conv_bn_act_backward(*[None if v is None else v.astype(np.float64) for v in args],
                                 f64_inputs=True, **kw)
    for key in ("dW", "db", "dgamma", "prev_delta", "dz"):
        if a[key] is None:
            assert b[key] is None, key
        else:
            assert np.array_equal(a[key], b[key]), key
    # and the values moved: the call did something with every output
    assert not np.array_equal(a["dW"], init["dW"])
    assert not np.array_equal(a["prev_delta"], init["prev_delta"])
