"""Pins of the oracle against things other than itself (CPU only).

* central finite differences of an independent float64 forward (the whole
  chain: activation, BN backward, bias/scale updates, dW, dx, shortcut add);
* the finite-difference harness itself against closed forms the pages print
  (sigmoid' = s(1-s); softmax-with-loss gradient = (p - onehot)/N);
* an im2col + matmul restatement and torch's float64 conv gradients (library
  special case) for the two convolution gradients;
* the 1x1 / stride 1 / pad 0 case = the inner-product (textbook GEMM) form;
* BN identities, and caffe's formulation of the BN backward;
* accumulation semantics (beta = 1 for dW, db, dgamma; = / += for prev_delta).
"""
import numpy as np
import pytest
import torch

from tests.fdutil import act_fwd, central_diff, layer_forward, min_kink_distance

EPS = 1e-5


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------- harness

def test_fd_harness_sigmoid_closed_form(ref):
    """caffe's sigmoid is 0.5*tanh(0.5x)+0.5 and its derivative s(1-s)
    (caffe source study page, SigmoidLayer Backward_cpu); darknet's
    logistic_gradient is (1-y)*y on the output y (YOLOv3 backprop page, §7)."""
    x = np.linspace(-4, 4, 17)
    for xi in x:
        f = lambda v: float(0.5 * np.tanh(0.5 * v[0]) + 0.5)  # noqa: E731
        g = central_diff(f, np.array([xi]))[0]
        s = 0.5 * np.tanh(0.5 * xi) + 0.5
        assert abs(g - s * (1 - s)) < 1e-9
        # the oracle's logistic gradient, evaluated on the output
        assert abs(ref.activation_gradient(ref.ACT_LOGISTIC, s) - g) < 1e-9


def test_fd_harness_softmax_loss_closed_form():
    """SoftmaxWithLoss backward subtracts 1 at the label and scales by
    loss_weight / outer_num (caffe LeNet backward page, 第九层
    SoftmaxWithLossLayer): grad = (p - onehot) / N."""
    rng = _rng(7)
    N, D = 4, 5
    logits = rng.standard_normal((N, D))
    labels = rng.integers(0, D, size=N)

    def loss(v):
        v = v.reshape(N, D)
        m = v.max(axis=1, keepdims=True)
        lse = np.log(np.exp(v - m).sum(axis=1)) + m[:, 0]
        return float(np.mean(lse - v[np.arange(N), labels]))

    g = central_diff(loss, logits).reshape(N, D)
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    onehot = np.zeros((N, D))
    onehot[np.arange(N), labels] = 1
    assert np.max(np.abs(g - (p - onehot) / N)) < 1e-8


# ------------------------------------------------ whole chain vs finite diff

FD_CASES = [
    # N, C, H, W, K, R, S, stride, pad, act, bn, residual
    (2, 3, 5, 5, 4, 3, 3, 1, 1, 1, True, False),
    (2, 3, 6, 5, 4, 3, 3, 2, 1, 1, True, True),
    (2, 3, 5, 6, 4, 3, 3, 1, 0, 0, False, False),
    (3, 4, 4, 4, 3, 1, 1, 1, 0, 1, True, True),
    (2, 2, 7, 7, 3, 5, 5, 1, 0, 0, False, True),
    (2, 3, 5, 5, 2, 3, 3, 2, 0, 1, False, False),
]


def _draw_case(case, seed):
    N, C, H, W, K, R, S, st, pad, act, bn, res = case
    for attempt in range(50):
        rng = _rng(seed + attempt)
        x = rng.standard_normal((N, C, H, W))
        w = rng.standard_normal((K, C, R, S)) * 0.5
        gamma = rng.uniform(0.5, 1.5, K)
        beta = rng.uniform(-0.3, 0.3, K)
        _, _, _, pre, _ = layer_forward(x, w, gamma, beta, stride=st, pad=pad, act=act, bn=bn,
                                        eps=EPS)
        if act == 1 and np.min(np.abs(pre)) < 5e-3:
            continue  # keep clear of the leaky kink
        D = rng.standard_normal(pre.shape)
        Dres = rng.standard_normal(x.shape) if res else None
        return x, w, gamma, beta, D, Dres
    raise RuntimeError("no draw clear of the kink")


@pytest.mark.parametrize("case", FD_CASES, ids=[str(i) for i in range(len(FD_CASES))])
def test_chain_matches_finite_differences(ref, case):
    N, C, H, W, K, R, S, st, pad, act, bn, res = case
    x, w, gamma, beta, D, Dres = _draw_case(case, 100 + FD_CASES.index(case))
    kw = dict(stride=st, pad=pad, act=act, bn=bn, eps=EPS)

    def loss_x(v):
        L = float(np.sum(D * layer_forward(v, w, gamma, beta, **kw)[4]))
        if Dres is not None:
            L += float(np.sum(Dres * v))  # the shortcut: block input feeds the sum directly
        return L

    def loss_w(v):
        return float(np.sum(D * layer_forward(x, v, gamma, beta, **kw)[4]))

    def loss_g(v):
        return float(np.sum(D * layer_forward(x, w, v, beta, **kw)[4]))

    def loss_b(v):
        return float(np.sum(D * layer_forward(x, w, gamma, v, **kw)[4]))

    z, mean, var, pre, out = layer_forward(x, w, gamma, beta, **kw)
    got = ref.conv_bn_act_backward(x, out, z if bn else None, D, w, gamma if bn else None,
                                   mean, var, Dres, stride=st, pad=pad, act=act,
                                   batch_normalize=bn, accumulate=0, eps=EPS, f64_inputs=True)

    def close(a, b, tol=2e-6):
        scale = max(np.max(np.abs(b)), 1e-12)
        assert np.max(np.abs(a - b)) <= tol * scale, (np.max(np.abs(a - b)), scale)

    close(got["prev_delta"], central_diff(loss_x, x))
    close(got["dW"], central_diff(loss_w, w))
    close(got["db"], central_diff(loss_b, beta))
    if bn:
        close(got["dgamma"], central_diff(loss_g, gamma))


FROZEN_CASES = [
    # N, C, H, W, K, R, S, stride, pad, act, residual
    (2, 3, 5, 5, 4, 3, 3, 1, 1, 1, False),
    (2, 3, 6, 5, 4, 3, 3, 2, 1, 0, True),
    (3, 4, 4, 4, 3, 1, 1, 1, 0, 1, True),
]


@pytest.mark.parametrize("case", FROZEN_CASES, ids=[str(i) for i in range(len(FROZEN_CASES))])
def test_frozen_stats_chain_matches_finite_differences(ref, case):
    """batch_normalize = 2: the mean and variance are constants of the forward
    (caffe use_global_stats), so the finite differences of the forward with
    those fixed statistics are the exact gradients of every output."""
    N, C, H, W, K, R, S, st, pad, act, res = case
    for attempt in range(50):
        seed = 300 + 100 * FROZEN_CASES.index(case) + attempt
        x, w, gamma, beta, D, Dres = _draw_case((N, C, H, W, K, R, S, st, pad, act, True, res),
                                                seed)
        rng = _rng(seed + 5000)
        z0 = layer_forward(x, w, gamma, beta, stride=st, pad=pad, act=0, bn=False, eps=EPS)[0]
        # statistics that are not the batch's own: shifted mean, scaled variance
        mean = z0.mean(axis=(0, 2, 3)) + rng.uniform(-0.5, 0.5, K)
        var = z0.var(axis=(0, 2, 3)) * rng.uniform(0.5, 2.0, K)
        kw = dict(stride=st, pad=pad, act=act, bn=True, eps=EPS, stats=(mean, var))
        z, _, _, pre, out = layer_forward(x, w, gamma, beta, **kw)
        if act != 1 or np.min(np.abs(pre)) >= 5e-3:
            break  # clear of the leaky kink
    else:
        raise RuntimeError("no draw clear of the kink")

    def loss_x(v):
        L = float(np.sum(D * layer_forward(v, w, gamma, beta, **kw)[4]))
        if Dres is not None:
            L += float(np.sum(Dres * v))
        return L

    got = ref.conv_bn_act_backward(x, out, z, D, w, gamma, mean, var, Dres, stride=st, pad=pad,
                                   act=act, batch_normalize=2, accumulate=0, eps=EPS,
                                   f64_inputs=True)

    def close(a, b, tol=2e-6):
        scale = max(np.max(np.abs(b)), 1e-12)
        assert np.max(np.abs(a - b)) <= tol * scale, (np.max(np.abs(a - b)), scale)

    close(got["prev_delta"], central_diff(loss_x, x))
    close(got["dW"], central_diff(
        lambda v: float(np.sum(D * layer_forward(x, v, gamma, beta, **kw)[4])), w))
    close(got["dgamma"], central_diff(
        lambda v: float(np.sum(D * layer_forward(x, w, v, beta, **kw)[4])), gamma))
    close(got["db"], central_diff(
        lambda v: float(np.sum(D * layer_forward(x, w, gamma, v, **kw)[4])), beta))
    # and it differs from the training-mode backward on the same inputs
    trn = ref.conv_bn_act_backward(x, out, z, D, w, gamma, mean, var, Dres, stride=st, pad=pad,
                                   act=act, batch_normalize=1, accumulate=0, eps=EPS,
                                   f64_inputs=True)
    assert np.max(np.abs(trn["dW"] - got["dW"])) > 1e-3 * np.max(np.abs(got["dW"]))


@pytest.mark.parametrize("act", range(14))
def test_activation_gradient_matches_fd_of_the_forward(ref, act):
    """Each activation's gradient, a function of the output y, against the
    central difference of the printed forward at the same pre-activation."""
    x = np.linspace(-6.0, 6.0, 1201) + 0.0037
    x = x[min_kink_distance(act, x) > 1e-3]
    h = 1e-6
    fd = (act_fwd(act, x + h) - act_fwd(act, x - h)) / (2 * h)
    y = act_fwd(act, x)
    got = np.array([ref.activation_gradient(act, v) for v in y])
    assert np.max(np.abs(got - fd)) < 2e-6, np.max(np.abs(got - fd))


ACT_CHAIN_CASES = [
    # N, C, H, W, K, R, S, stride, pad, act, bn, residual
    (2, 3, 5, 5, 4, 3, 3, 1, 1, 2, True, False),   # logistic
    (2, 3, 6, 5, 4, 3, 3, 2, 1, 6, False, True),   # tanh
    (2, 3, 5, 5, 3, 3, 3, 1, 1, 8, True, True),    # elu
    (3, 4, 4, 4, 3, 1, 1, 1, 0, 9, False, False),  # selu
    (2, 3, 5, 5, 4, 3, 3, 1, 1, 7, True, False),   # plse
]


@pytest.mark.parametrize("case", ACT_CHAIN_CASES, ids=[str(c[9]) for c in ACT_CHAIN_CASES])
def test_chain_with_other_activations_matches_finite_differences(ref, case):
    N, C, H, W, K, R, S, st, pad, act, bn, res = case
    for attempt in range(50):
        x, w, gamma, beta, D, Dres = _draw_case(case[:9] + (0, bn, res),
                                                600 + 100 * ACT_CHAIN_CASES.index(case) + attempt)
        kw = dict(stride=st, pad=pad, act=act, bn=bn, eps=EPS)
        z, mean, var, pre, out = layer_forward(x, w, gamma, beta, **kw)
        if np.min(min_kink_distance(act, pre)) > 5e-3:
            break
    else:
        raise RuntimeError("no draw clear of the kinks")

    def loss(xv=x, wv=w, gv=gamma, bv=beta):
        L = float(np.sum(D * layer_forward(xv, wv, gv, bv, **kw)[4]))
        if Dres is not None:
            L += float(np.sum(Dres * xv))
        return L

    got = ref.conv_bn_act_backward(x, out, z if bn else None, D, w, gamma if bn else None,
                                   mean, var, Dres, stride=st, pad=pad, act=act,
                                   batch_normalize=int(bn), accumulate=0, eps=EPS,
                                   f64_inputs=True)

    def close(a, b, tol=2e-6):
        scale = max(np.max(np.abs(b)), 1e-12)
        assert np.max(np.abs(a - b)) <= tol * scale, (np.max(np.abs(a - b)), scale)

    close(got["prev_delta"], central_diff(lambda v: loss(xv=v), x))
    close(got["dW"], central_diff(lambda v: loss(wv=v), w))
    close(got["db"], central_diff(lambda v: loss(bv=v), beta))
    if bn:
        close(got["dgamma"], central_diff(lambda v: loss(gv=v), gamma))


GROUP_CASES = [
    # N, C, H, W, K, R, S, stride, pad, act, bn, residual, groups
    (2, 4, 5, 5, 6, 3, 3, 1, 1, 1, True, False, 2),
    (2, 6, 6, 5, 3, 3, 3, 2, 1, 0, False, True, 3),
    (3, 4, 4, 4, 4, 1, 1, 1, 0, 1, True, True, 4),    # depthwise 1x1
    (2, 4, 5, 5, 4, 3, 3, 1, 1, 1, True, False, 4),   # depthwise 3x3
]


@pytest.mark.parametrize("case", GROUP_CASES, ids=[str(i) for i in range(len(GROUP_CASES))])
def test_grouped_chain_matches_finite_differences(ref, case):
    """l.groups ([YOLO] §3.1): the whole chain of a grouped convolution against
    finite differences of torch's grouped conv2d forward."""
    N, C, H, W, K, R, S, st, pad, act, bn, res, G = case
    rng = _rng(800 + GROUP_CASES.index(case))
    for attempt in range(50):
        x = rng.standard_normal((N, C, H, W))
        w = rng.standard_normal((K, C // G, R, S)) * 0.5
        gamma = rng.uniform(0.5, 1.5, K)
        beta = rng.uniform(-0.3, 0.3, K)
        kw = dict(stride=st, pad=pad, act=act, bn=bn, eps=EPS, groups=G)
        z, mean, var, pre, out = layer_forward(x, w, gamma, beta, **kw)
        if act != 1 or np.min(np.abs(pre)) >= 5e-3:
            break
    else:
        raise RuntimeError("no draw clear of the kink")
    D = rng.standard_normal(pre.shape)
    Dres = rng.standard_normal(x.shape) if res else None

    def loss(xv=x, wv=w, gv=gamma, bv=beta):
        L = float(np.sum(D * layer_forward(xv, wv, gv, bv, **kw)[4]))
        if Dres is not None:
            L += float(np.sum(Dres * xv))
        return L

    got = ref.conv_bn_act_backward(x, out, z if bn else None, D, w, gamma if bn else None,
                                   mean, var, Dres, stride=st, pad=pad, act=act,
                                   batch_normalize=int(bn), accumulate=0, eps=EPS,
                                   f64_inputs=True, groups=G)

    def close(a, b, tol=2e-6):
        scale = max(np.max(np.abs(b)), 1e-12)
        assert np.max(np.abs(a - b)) <= tol * scale, (np.max(np.abs(a - b)), scale)

    close(got["prev_delta"], central_diff(lambda v: loss(xv=v), x))
    close(got["dW"], central_diff(lambda v: loss(wv=v), w))
    close(got["db"], central_diff(lambda v: loss(bv=v), beta))
    if bn:
        close(got["dgamma"], central_diff(lambda v: loss(gv=v), gamma))


@pytest.mark.parametrize("G", [2, 4, 8])
def test_grouped_conv_gradients_vs_torch(ref, G):
    """Linear, no BN: dW and dx of a grouped convolution against torch's float64
    grouped conv2d_weight / conv2d_input (a library special case)."""
    rng = _rng(900 + G)
    N, C, H, W, K, R, S, st, pad = 2, 8, 7, 6, 16, 3, 3, 2, 1
    x = rng.standard_normal((N, C, H, W))
    w = rng.standard_normal((K, C // G, R, S))
    P, Q = (H + 2 * pad - R) // st + 1, (W + 2 * pad - S) // st + 1
    D = rng.standard_normal((N, K, P, Q))
    got = ref.conv_bn_act_backward(x, None, None, D, w, None, None, None, None, stride=st,
                                   pad=pad, act=0, batch_normalize=0, accumulate=0, eps=EPS,
                                   f64_inputs=True, groups=G)
    tx, tw, tD = (torch.from_numpy(a) for a in (x, w, D))
    gw = torch.nn.grad.conv2d_weight(tx, tw.shape, tD, stride=st, padding=pad, groups=G)
    gx = torch.nn.grad.conv2d_input(tx.shape, tw, tD, stride=st, padding=pad, groups=G)
    assert np.max(np.abs(got["dW"] - gw.numpy())) < 1e-10
    assert np.max(np.abs(got["prev_delta"] - gx.numpy())) < 1e-10


# ------------------------------------- convolution gradients, other forms

def _im2col(img, R, S, stride, pad):
    """im2col of one image [C,H,W] -> [C*R*S, P*Q]; row c*R*S + r*S + s,
    column p*Q + q, zero outside the image (YOLOv3 backprop page, §3.2,
    im2col_cpu / im2col_get_pixel)."""
    C, H, W = img.shape
    P = (H + 2 * pad - R) // stride + 1
    Q = (W + 2 * pad - S) // stride + 1
    padded = np.zeros((C, H + 2 * pad, W + 2 * pad))
    padded[:, pad:pad + H, pad:pad + W] = img
    col = np.empty((C * R * S, P * Q))
    for c in range(C):
        for r in range(R):
            for s in range(S):
                win = padded[c, r:r + stride * (P - 1) + 1:stride, s:s + stride * (Q - 1) + 1:stride]
                col[(c * R + r) * S + s] = win.reshape(-1)
    return col


def _col2im(col, C, H, W, R, S, stride, pad):
    """The adding inverse of _im2col (col2im_cpu / col2im_add_pixel)."""
    P = (H + 2 * pad - R) // stride + 1
    Q = (W + 2 * pad - S) // stride + 1
    padded = np.zeros((C, H + 2 * pad, W + 2 * pad))
    for c in range(C):
        for r in range(R):
            for s in range(S):
                padded[c, r:r + stride * (P - 1) + 1:stride, s:s + stride * (Q - 1) + 1:stride] += \
                    col[(c * R + r) * S + s].reshape(P, Q)
    return padded[:, pad:pad + H, pad:pad + W]


CONV_CASES = [(2, 3, 7, 6, 5, 3, 3, 1, 1), (2, 4, 9, 8, 3, 3, 3, 2, 1), (3, 2, 6, 6, 4, 1, 1, 1, 0),
              (2, 3, 8, 7, 2, 5, 5, 1, 2), (1, 2, 9, 9, 3, 3, 3, 2, 0), (2, 2, 5, 5, 2, 2, 3, 1, 1)]


@pytest.mark.parametrize("case", CONV_CASES)
def test_conv_gradients_vs_im2col_gemm(ref, case):
    """The per-image GEMMs of backward_convolutional_layer (YOLOv3 backprop
    page §3.1): dW += delta_i . col_i^T and dx_i = col2im(W^T . delta_i)."""
    N, C, H, W, K, R, S, st, pad = case
    rng = _rng(sum(case))
    x = rng.standard_normal((N, C, H, W))
    w = rng.standard_normal((K, C, R, S))
    P, Q = (H + 2 * pad - R) // st + 1, (W + 2 * pad - S) // st + 1
    d = rng.standard_normal((N, K, P, Q))
    dW = np.zeros((K, C * R * S))
    dx = np.zeros((N, C, H, W))
    for n in range(N):
        col = _im2col(x[n], R, S, st, pad)
        dW += d[n].reshape(K, P * Q) @ col.T
        dx[n] = _col2im(w.reshape(K, -1).T @ d[n].reshape(K, P * Q), C, H, W, R, S, st, pad)
    got_w = ref.conv_wgrad(d, x, R, S, st, pad)
    got_x = ref.conv_dgrad(d, w, H, W, st, pad)
    assert np.max(np.abs(got_w.reshape(K, -1) - dW)) <= 1e-12 * np.max(np.abs(dW))
    assert np.max(np.abs(got_x - dx)) <= 1e-12 * np.max(np.abs(dx))
    # library special case: torch's float64 convolution gradients
    tw = torch.nn.grad.conv2d_weight(torch.from_numpy(x), w.shape, torch.from_numpy(d), stride=st,
                                     padding=pad).numpy()
    tx = torch.nn.grad.conv2d_input(x.shape, torch.from_numpy(w), torch.from_numpy(d), stride=st,
                                    padding=pad).numpy()
    assert np.max(np.abs(got_w - tw)) <= 1e-12 * np.max(np.abs(tw))
    assert np.max(np.abs(got_x - tx)) <= 1e-12 * np.max(np.abs(tx))
    # the gather forms agree with the loops on every element
    got_w_at = ref.wgrad_at(d, x.astype(np.float32), R, S, st, pad, np.arange(got_w.size))
    xf = x.astype(np.float32).astype(np.float64)
    ref_w32 = ref.conv_wgrad(d, xf, R, S, st, pad)
    assert np.max(np.abs(got_w_at - ref_w32.reshape(-1))) <= 1e-12 * np.max(np.abs(ref_w32))
    wf = w.astype(np.float32)
    got_x_at = ref.dgrad_at(d, wf, H, W, st, pad, np.arange(dx.size))
    ref_x32 = ref.conv_dgrad(d, wf.astype(np.float64), H, W, st, pad)
    assert np.max(np.abs(got_x_at - ref_x32.reshape(-1))) <= 1e-12 * np.max(np.abs(ref_x32))


def test_one_by_one_is_inner_product(ref):
    """A 1x1, stride 1, pad 0 conv is an inner-product layer per pixel
    (caffe LeNet backward page, 第八层 InnerProduct: dW += top_diff^T . bottom,
    bottom_diff = top_diff . W): dW = sum_n delta_n . X_n^T, dx_n = W^T . delta_n."""
    rng = _rng(11)
    N, C, H, W, K = 3, 6, 4, 5, 7
    x = rng.standard_normal((N, C, H, W))
    w = rng.standard_normal((K, C, 1, 1))
    d = rng.standard_normal((N, K, H, W))
    X = x.reshape(N, C, H * W)
    Dm = d.reshape(N, K, H * W)
    dW = sum(Dm[n] @ X[n].T for n in range(N))
    dx = np.stack([w[:, :, 0, 0].T @ Dm[n] for n in range(N)]).reshape(N, C, H, W)
    assert np.allclose(ref.conv_wgrad(d, x, 1, 1, 1, 0)[:, :, 0, 0], dW, rtol=0, atol=1e-12)
    assert np.allclose(ref.conv_dgrad(d, w, H, W, 1, 0), dx, rtol=0, atol=1e-12)


# ----------------------------------------------------------- BN backward

def _bn_inputs(seed, N=4, K=3, P=5, Q=6):
    rng = _rng(seed)
    z = rng.standard_normal((N, K, P, Q)) * 2 + 0.7
    mean = z.mean(axis=(0, 2, 3))
    var = ((z - mean[None, :, None, None]) ** 2).mean(axis=(0, 2, 3))
    gamma = rng.uniform(0.5, 1.5, K)
    d = rng.standard_normal((N, K, P, Q))
    return z, mean, var, gamma, d


def test_bn_identities(ref):
    """With the batch statistics: sum over (n,p,q) of the BN-input gradient is 0,
    and sum(grad * x_norm) = (gamma/sigma) * sum(delta * x_norm) * eps/(var+eps)."""
    z, mean, var, gamma, d = _bn_inputs(3)
    K = z.shape[1]
    xn = ref.x_norm(z, mean, var, EPS)
    dbn, db, dg = ref.backward_batchnorm(z, xn, mean, var, gamma, EPS, d, np.zeros(K), np.zeros(K))
    s0 = dbn.sum(axis=(0, 2, 3))
    assert np.max(np.abs(s0)) < 1e-12 * np.abs(dbn).sum()
    s1 = (dbn * xn).sum(axis=(0, 2, 3))
    S2 = (d * xn).sum(axis=(0, 2, 3))
    expect = gamma / np.sqrt(var + EPS) * S2 * EPS / (var + EPS)
    assert np.allclose(s1, expect, rtol=1e-9, atol=1e-13)
    # the parameter updates are the two plain sums
    assert np.allclose(db, d.sum(axis=(0, 2, 3)), rtol=1e-13, atol=0)
    assert np.allclose(dg, S2, rtol=1e-13, atol=0)


def test_bn_darknet_equals_caffe(ref):
    """Darknet's three-step BN backward (YOLOv3 backprop page §4) equals caffe's
    (dY - mean(dY) - mean(dY.Y).Y)/sqrt(var+eps) (BatchNorm 理解 page,
    Backward_cpu) with dY = gamma*delta (the Scale layer in front of it)."""
    z, mean, var, gamma, d = _bn_inputs(5)
    K = z.shape[1]
    xn = ref.x_norm(z, mean, var, EPS)
    dbn, _, _ = ref.backward_batchnorm(z, xn, mean, var, gamma, EPS, d, np.zeros(K), np.zeros(K))
    caffe = ref.bn_backward_caffe(gamma[None, :, None, None] * d, xn, var, EPS)
    assert np.max(np.abs(dbn - caffe)) <= 1e-12 * np.max(np.abs(caffe))


def test_mean_delta_is_the_printed_truncated_form(ref):
    """mean_delta_cpu (YOLOv3 backprop page, §4) is the derivative through the
    mean's direct use only: it leaves out vd * sum(-2(z - mean))/m, the part
    that reaches the mean through the variance.  Take G = dL/dxhat fixed and
    f(mu) = sum G * (z - mu) / sqrt(v(mu) + eps) with v(mu) = mean((z - mu)^2),
    a mean that is NOT the batch mean.  The central difference of f is then
    mean_delta + variance_delta * sum(-2(z - mu))/m, and mean_delta alone
    misses it by that term; at the batch mean the term is rounding-level."""
    z, _, _, _, G = _bn_inputs(9)
    N, K, P, Q = z.shape
    m = N * P * Q
    rng = _rng(19)
    mu = z.mean(axis=(0, 2, 3)) + rng.uniform(0.3, 0.6, K) * rng.choice([-1, 1], K)

    def v_of(mv):
        return ((z - mv[None, :, None, None]) ** 2).mean(axis=(0, 2, 3))

    def f(mv):
        return float(np.sum(G * (z - mv[None, :, None, None]) /
                            np.sqrt(v_of(mv)[None, :, None, None] + EPS)))

    def oracle_parts(mv):
        var = v_of(mv)
        md, vd = np.empty(K), np.empty(K)
        L = ref.lib()
        L.cba_ref_mean_delta(ref.ref._pd(G), ref.ref._pd(var), EPS, N, K, P * Q, ref.ref._pd(md))
        L.cba_ref_variance_delta(ref.ref._pd(z), ref.ref._pd(G), ref.ref._pd(mv),
                                 ref.ref._pd(var), EPS, N, K, P * Q, ref.ref._pd(vd))
        return md, vd

    # per channel, f's derivative in mu_k is the k-th component of the gradient
    fd = central_diff(f, mu)
    md, vd = oracle_parts(mu)
    omitted = vd * (-2.0 * (z - mu[None, :, None, None])).sum(axis=(0, 2, 3)) / m
    assert np.max(np.abs(md + omitted - fd)) <= 1e-6 * np.max(np.abs(fd))
    assert np.min(np.abs(omitted)) > 1e-2 * np.max(np.abs(fd))  # the omission shows
    assert np.max(np.abs(md - fd)) > 1e-2 * np.max(np.abs(fd))
    # at the batch mean the omitted term vanishes up to rounding
    mb = z.mean(axis=(0, 2, 3))
    md_b, vd_b = oracle_parts(mb)
    om_b = vd_b * (-2.0 * (z - mb[None, :, None, None])).sum(axis=(0, 2, 3)) / m
    assert np.max(np.abs(om_b)) <= 1e-12 * np.max(np.abs(md_b))
    assert np.max(np.abs(md_b - central_diff(f, mb))) <= 1e-6 * np.max(np.abs(md_b))


def test_leaky_gradient_tie_at_zero(ref):
    """leaky_gradient is (y>0) ? 1 : .1 (YOLOv3 backprop page §7); caffe's ReLU
    backward (x>0) + slope*(x<=0) (LeNet page, 第七层 ReLU) agrees, also at 0."""
    for y, g in [(1.0, 1.0), (1e-30, 1.0), (0.0, 0.1), (-0.0, 0.1), (-2.0, 0.1)]:
        assert ref.activation_gradient(ref.ACT_LEAKY, y) == g
        assert float((y > 0) + 0.1 * (y <= 0)) == g
    assert ref.activation_gradient(ref.ACT_LINEAR, -3.0) == 1.0


# ------------------------------------------------------------ accumulation

def test_accumulation_semantics(ref):
    """dW, db, dgamma accumulate (gemm beta = 1, scale_updates +=); prev_delta
    is written (accumulate = 0) or added to (accumulate = 1)."""
    rng = _rng(21)
    N, C, H, W, K = 2, 3, 6, 6, 4
    x = rng.standard_normal((N, C, H, W)).astype(np.float32)
    w = (rng.standard_normal((K, C, 3, 3)) * 0.3).astype(np.float32)
    from tests.fdutil import layer_forward as lf
    z, mean, var, pre, out = lf(x, w, np.ones(K), np.zeros(K), stride=1, pad=1, act=1, bn=True,
                                eps=EPS)
    d = rng.standard_normal(out.shape).astype(np.float32)
    args = (x, out.astype(np.float32), z.astype(np.float32), d, w, np.ones(K, np.float32),
            mean.astype(np.float32), var.astype(np.float32), None)
    kw = dict(stride=1, pad=1, act=1, batch_normalize=True, eps=EPS)
    one = ref.conv_bn_act_backward(*args, accumulate=0, **kw)
    two = ref.conv_bn_act_backward(*args, accumulate=1, dW=one["dW"], db=one["db"],
                                   dgamma=one["dgamma"], prev_delta=one["prev_delta"], **kw)
    for key in ("dW", "db", "dgamma", "prev_delta"):
        assert np.allclose(two[key], 2 * one[key], rtol=1e-12, atol=1e-15), key
    again = ref.conv_bn_act_backward(*args, accumulate=0, prev_delta=two["prev_delta"], **kw)
    assert np.allclose(again["prev_delta"], one["prev_delta"], rtol=0, atol=0)
    skip = ref.conv_bn_act_backward(*args, accumulate=0, want_prev=False, **kw)
    assert skip["prev_delta"] is None and np.allclose(skip["dW"], one["dW"], rtol=0, atol=0)
