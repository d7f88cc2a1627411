"""GPU parity: the CUDA path through the C ABI against the oracle.

Element by element on reduced-batch versions of the five workloads (same
channel and spatial geometry, so the tiles and ragged tails are the same),
on sampled outputs at full size, and on edge shapes.  Bars (max |err| per
tensor, relative to max |ref| of that tensor): 2e-3 for the TF32
tensor-core mode, 1e-5 for the FFMA mode.
"""
import functools
import os

import numpy as np
import pytest
import torch

import activation_backward_gb300 as cba
from activation_backward_gb300 import inputs
from activation_backward_gb300.layer import DeviceLayer

pytestmark = pytest.mark.gpu

TF32, FFMA = cba.CBA_MATH_TF32, cba.CBA_MATH_FFMA
TOL = {TF32: 2e-3, FFMA: 1e-5}
MATHS = [pytest.param(TF32, id="tf32"), pytest.param(FFMA, id="ffma")]
KEYS = ("dW", "db", "dgamma", "prev_delta")


@functools.lru_cache(maxsize=None)
def config_layers(cid, batch=None):
    return inputs.make_config(cid, batch=batch)


def oracle_chain(ref, layer, **kw):
    g = layer["geom"]
    return ref.conv_bn_act_backward(layer["x"], layer["output"], layer["z"], layer["delta"],
                                    layer["W"], layer["gamma"], layer["mean"], layer["var"],
                                    layer["residual"], stride=g.stride, pad=g.pad,
                                    act=layer["act"], batch_normalize=layer["bn"],
                                    accumulate=kw.pop("accumulate", layer["accumulate"]),
                                    eps=layer["eps"], groups=layer.get("groups", 1), **kw)


def assert_close(got, exp, tol, what, atol=1e-30):
    assert got.shape == exp.shape, (what, got.shape, exp.shape)
    assert np.all(np.isfinite(got)), what
    err = float(np.max(np.abs(got - exp))) if exp.size else 0.0
    scale = float(np.max(np.abs(exp))) if exp.size else 0.0
    assert err <= tol * scale + atol, f"{what}: max|err| {err:.3e} > {tol} * {scale:.3e} + {atol}"


def run_gpu(layer, math, **kw):
    dl = DeviceLayer(layer, math=math, **kw)
    dl.run()
    assert dl.status() == cba.CBA_OK
    torch.cuda.synchronize()
    return dl, dl.results()


def test_the_in_tree_library_is_loaded(cuda_lib):
    maps = open("/proc/self/maps").read()
    here = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "activation_backward_gb300", "libcba.so")
    assert os.path.realpath(here) in maps or here in maps


SMALL = [(1, 4), (2, 2), (3, 2), (4, 4), (5, 2)]


OTHER_ACTS = list(range(2, 14))


@pytest.mark.parametrize("act", OTHER_ACTS, ids=[cba.ACT_NAMES[a] for a in OTHER_ACTS])
def test_parity_other_activations(ref, cuda_lib, act):
    # activations other than linear and leaky (a gradient_array pass, then the
    # main kernels in linear mode): a BN layer in TF32, a layer without BN in FFMA
    for cid, batch, math in ((2, 1, TF32), (1, 4, FFMA)):
        layer = inputs.with_activation(config_layers(cid, batch)[0], act)
        _, got = run_gpu(layer, math, want_dz=True)
        exp = oracle_chain(ref, layer, want_dz=True)
        for k in KEYS + ("dz",):
            if exp.get(k) is not None:
                assert_close(got[k], exp[k], TOL[math], f"{layer['name']} {k}")


GROUPED = [(2, 2, 2), (2, 2, 4), (2, 1, 64), (3, 2, 8)]


@pytest.mark.parametrize("math", MATHS)
@pytest.mark.parametrize("cid,batch,groups", GROUPED,
                         ids=[f"cfg{c}_n{b}_g{g}" for c, b, g in GROUPED])
def test_parity_grouped(ref, cuda_lib, cid, batch, groups, math):
    # l.groups: output channel k meets only the input channels of its group
    layer = inputs.make_grouped_config(cid, groups, batch=batch)
    _, got = run_gpu(layer, math, want_dz=True)
    exp = oracle_chain(ref, layer, want_dz=True)
    for k in KEYS + ("dz",):
        if exp.get(k) is not None:
            assert_close(got[k], exp[k], TOL[math], f"{layer['name']} {k}")


GROUPED_EDGE = [
    # N, C, H, W, K, R, S, stride, pad, act, bn, groups
    # stride 2, groups of 8 input / 12 output channels (batch-innermost wgrad)
    (2, 24, 9, 10, 36, 3, 3, 2, 1, 1, True, 3),
    # 1x1 layer with 16-byte rows (TMA-fed wgrad): groups of 6 / 5
    (2, 48, 8, 8, 40, 1, 1, 1, 0, 0, False, 8),
    # depthwise: one input and one output channel per group
    (2, 32, 7, 7, 32, 3, 3, 1, 1, 1, True, 32),
    # groups of 130 channels straddle the 128-channel tiles
    (1, 260, 6, 6, 260, 3, 3, 1, 1, 1, True, 2),
]


@pytest.mark.parametrize("math", MATHS)
@pytest.mark.parametrize("case", GROUPED_EDGE, ids=[str(i) for i in range(len(GROUPED_EDGE))])
def test_parity_grouped_edge_shapes(ref, cuda_lib, case, math):
    N, C, H, W, K, R, S, st, pad, act, bn, groups = case
    spec = inputs.LayerSpec("grouped edge", inputs.Geometry(N, C, H, W, K, R, S, st, pad), act, bn)
    layer = inputs.make_layer(spec, 700 + GROUPED_EDGE.index(case), residual=True, groups=groups)
    _, got = run_gpu(layer, math, want_dz=True)
    exp = oracle_chain(ref, layer, want_dz=True)
    for k in KEYS + ("dz",):
        if exp.get(k) is not None:
            assert_close(got[k], exp[k], TOL[math], f"grouped edge {case} {k}")


def test_parity_grouped_z_free_accumulate(ref, cuda_lib):
    # grouped, z recomputed per group, prev_delta added onto its contents
    layer = inputs.make_grouped_config(2, 4, batch=2)
    prev0 = (np.random.default_rng(5).standard_normal(layer["x"].shape) * 0.01).astype(np.float32)
    _, got = run_gpu(layer, TF32, z_free=True, accumulate=1, prev_init=prev0)
    exp = oracle_chain(ref, layer, accumulate=1, prev_delta=prev0)
    for k in KEYS:
        if exp.get(k) is not None:
            assert_close(got[k], exp[k], TOL[TF32], f"{layer['name']} z-free {k}")


ZFREE = [(2, 2), (3, 2), (5, 2)]


@pytest.mark.parametrize("math", MATHS)
@pytest.mark.parametrize("cid,batch", ZFREE, ids=[f"cfg{c}_n{b}" for c, b in ZFREE])
def test_parity_z_free(ref, cuda_lib, cid, batch, math):
    # BN without z: the library recomputes z = conv(x, W) (fp32) in its workspace;
    # the oracle gets the generator's z (an fp64 convolution rounded to fp32)
    for layer in config_layers(cid, batch):
        _, got = run_gpu(layer, math, want_dz=True, z_free=True)
        exp = oracle_chain(ref, layer, want_dz=True)
        for k in KEYS + ("dz",):
            if exp.get(k) is not None:
                assert_close(got[k], exp[k], TOL[math], f"{layer['name']} z-free {k}")


FROZEN = [(2, 2), (3, 2), (5, 2)]


@pytest.mark.parametrize("math", MATHS)
@pytest.mark.parametrize("cid,batch", FROZEN, ids=[f"cfg{c}_n{b}" for c, b in FROZEN])
def test_parity_frozen_bn_statistics(ref, cuda_lib, cid, batch, math):
    # batch_normalize = 2: mean/var are constants of the forward; the BN-input
    # gradient dz is compared as well (dz_out)
    for i, layer in enumerate(config_layers(cid, batch)):
        layer = inputs.with_frozen_stats(layer, 900 + 10 * cid + i)
        _, got = run_gpu(layer, math, want_dz=True)
        exp = oracle_chain(ref, layer, want_dz=True)
        for k in KEYS + ("dz",):
            if exp.get(k) is not None:
                assert_close(got[k], exp[k], TOL[math], f"{layer['name']} {k}")


@pytest.mark.parametrize("math", MATHS)
@pytest.mark.parametrize("cid,batch", SMALL, ids=[f"cfg{c}_n{b}" for c, b in SMALL])
def test_parity_elementwise_reduced_batch(ref, cuda_lib, cid, batch, math):
    for layer in config_layers(cid, batch):
        _, got = run_gpu(layer, math)
        exp = oracle_chain(ref, layer)
        for k in KEYS:
            if exp[k] is not None:
                assert_close(got[k], exp[k], TOL[math], f"{layer['name']} {k}")


@pytest.mark.parametrize("math", MATHS)
@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_parity_full_size_sampled(ref, cuda_lib, cid, math):
    """Full workload sizes, the launch configuration the bench times.  db and
    dgamma are checked in full; dW and prev_delta on 3000 sampled elements
    each (plus the corners), computed one by one by the oracle."""
    for li, layer in enumerate(config_layers(cid)):
        g = layer["geom"]
        _, got = run_gpu(layer, math)
        dz, db, dg = ref.backward_dz(layer["output"], layer["z"], layer["delta"], layer["gamma"],
                                     layer["mean"], layer["var"], act=layer["act"],
                                     batch_normalize=layer["bn"], eps=layer["eps"])
        tol = TOL[math]
        assert_close(got["db"], db, tol, "db")
        if layer["bn"]:
            assert_close(got["dgamma"], dg, tol, "dgamma")
        rng = np.random.default_rng(7 * cid + li)
        nw = got["dW"].size
        iw = np.unique(np.concatenate([rng.choice(nw, min(nw, 3000), replace=False),
                                       [0, nw - 1]]))
        ew = ref.wgrad_at(dz, layer["x"], g.R, g.S, g.stride, g.pad, iw)
        assert_close(got["dW"].reshape(-1)[iw], ew, tol, "dW sampled")
        npv = got["prev_delta"].size
        ip = np.unique(np.concatenate([rng.choice(npv, 3000, replace=False), [0, npv - 1]]))
        ep = ref.dgrad_at(dz, layer["W"], g.H, g.W, g.stride, g.pad, ip,
                          residual=layer["residual"])
        assert_close(got["prev_delta"].reshape(-1)[ip], ep, tol, "prev_delta sampled")


def _desc(g, act, bn, math=TF32):
    return cba.make_desc(g.N, g.C, g.H, g.W, g.K, g.R, g.S, g.stride, g.pad, act=act,
                         batch_normalize=int(bn), math=math)


def test_plan_paths(cuda_lib):
    """The kernels each workload's calls run: every layer on the tensor cores,
    the stride-1 3x3 and 1x1 layers whose input rows are 16-byte strided
    (config 2's 52-wide rows, the residual block's 1x1 layer viewing each
    26 x 26 plane as one row) with the TMA-row weight gradient, the others
    (5x5, stride 2, 13 x 13 planes, 26-wide rows) with the batch-innermost
    one; FFMA mode on the CUDA cores; the parity shapes below reach both
    tensor-core paths."""
    C = inputs.CONFIGS
    bi, rows = cba.CBA_PATH_TC_BATCH_INNER, cba.CBA_PATH_TC_ROWS
    g1 = cba.CBA_PATH_TC_GEMM_1X1
    for cid, path in ((1, bi), (2, rows), (3, bi), (4, bi)):
        assert cba.cba_plan_info(_desc(C[cid].geom, C[cid].act, C[cid].bn))[0] == path, cid
    assert cba.cba_plan_info(_desc(inputs.BLOCK_CONV2, 1, True))[0] == bi
    assert cba.cba_plan_info(_desc(C[5].geom, 1, True))[0] == g1
    assert cba.cba_plan_info(_desc(C[5].geom, 1, True), groups=2)[0] == rows
    assert cba.cba_plan_info(_desc(C[2].geom, 1, True, FFMA))[0] == cba.CBA_PATH_FFMA
    seen = {cba.cba_plan_info(_desc(inputs.Geometry(*c[:9]), c[9], c[10]))[0] for c in EDGE}
    assert seen == {bi, rows, g1}


EDGE = [
    # N, C, H, W, K, R, S, stride, pad, act, bn
    (2, 3, 7, 9, 5, 3, 3, 1, 1, 1, True),
    (3, 17, 13, 11, 33, 3, 3, 2, 1, 1, True),
    (2, 32, 13, 13, 255, 1, 1, 1, 0, 0, False),
    (2, 20, 12, 12, 50, 5, 5, 1, 0, 0, False),
    (1, 8, 6, 6, 7, 3, 3, 1, 0, 1, False),
    (2, 5, 10, 9, 6, 2, 3, 2, 0, 1, True),
    (1, 4, 5, 5, 3, 5, 5, 1, 2, 0, True),
    (1, 3, 1, 1, 2, 1, 1, 1, 0, 1, True),
    (2, 64, 9, 9, 130, 3, 3, 1, 1, 1, True),
    (1, 129, 8, 8, 64, 3, 3, 2, 1, 1, True),
    (4, 16, 16, 16, 16, 1, 1, 2, 0, 1, False),
    (2, 24, 15, 14, 40, 3, 3, 3, 2, 0, True),
    # weight gradient fed by TMA (input width a multiple of 4): a ragged last
    # column chunk; a 1x1 layer viewed as one row per plane; two 128-channel
    # tiles of k with an odd number of 32-channel chunks
    (2, 24, 12, 36, 40, 3, 3, 1, 1, 1, True),
    (2, 48, 8, 8, 24, 1, 1, 1, 0, 0, False),
    (2, 16, 8, 12, 160, 3, 3, 1, 1, 1, True),
    # input gradient with two k-chunks per stage and an odd chunk count (the
    # last stage's second chunk lies past K and is zero-filled)
    (2, 16, 10, 10, 96, 3, 3, 1, 1, 1, True),
    # 1x1 layers as plain GEMMs: partial channel, position and k tiles; tiny
    # planes, channels and k (boxes mostly out of bounds)
    (3, 36, 6, 10, 70, 1, 1, 1, 0, 1, True),
    (2, 260, 16, 20, 300, 1, 1, 1, 0, 1, True),
    (1, 4, 2, 2, 3, 1, 1, 1, 0, 1, True),
    (3, 8, 3, 4, 40, 1, 1, 1, 0, 0, False),
]


@pytest.mark.parametrize("math", MATHS)
@pytest.mark.parametrize("case", EDGE, ids=[str(i) for i in range(len(EDGE))])
def test_parity_edge_shapes(ref, cuda_lib, case, math):
    N, C, H, W, K, R, S, st, pad, act, bn = case
    spec = inputs.LayerSpec("edge", inputs.Geometry(N, C, H, W, K, R, S, st, pad), act, bn)
    layer = inputs.make_layer(spec, 500 + EDGE.index(case), residual=True)
    _, got = run_gpu(layer, math)
    exp = oracle_chain(ref, layer)
    # With one element per channel (N*P*Q = 1) and batch statistics, the
    # BN-input gradient dz = a*delta' - a*delta' is zero in exact arithmetic,
    # so dW and prev_delta (both linear in dz) are zero too; fp32 leaves
    # rounding noise of the size of the inputs times 2^-24, which an absolute
    # floor admits for those two tensors only.  db = delta' is not zero and
    # keeps the relative bar; dgamma = delta' * xhat with xhat = 0 exactly.
    one = bn and N * ((H + 2 * pad - R) // st + 1) * ((W + 2 * pad - S) // st + 1) == 1
    for k in KEYS:
        if exp[k] is not None:
            atol = 1e-6 if one and k in ("dW", "prev_delta") else 1e-30
            assert_close(got[k], exp[k], TOL[math], k, atol=atol)


@pytest.mark.parametrize("math", MATHS)
def test_two_calls_accumulate(ref, cuda_lib, math):
    layer = config_layers(2, 2)[0]
    for acc in (0, 1):
        dl = DeviceLayer(layer, math=math, accumulate=acc)
        dl.run()
        first = dl.results()
        dl.run()
        assert dl.status() == cba.CBA_OK
        second = dl.results()
        for k in ("dW", "db", "dgamma"):
            assert_close(second[k], 2 * first[k], TOL[math], k)
        exp_prev = 2 * first["prev_delta"] if acc else first["prev_delta"]
        assert_close(second["prev_delta"], exp_prev, TOL[math], f"prev acc={acc}")


def test_accumulate_onto_existing_prev(ref, cuda_lib):
    layer = config_layers(3, 2)[0]
    rng = np.random.default_rng(3)
    seed = rng.standard_normal(layer["x"].shape).astype(np.float32)
    _, got = run_gpu(layer, FFMA, accumulate=1, prev_init=seed)
    exp = oracle_chain(ref, layer, accumulate=1, prev_delta=seed)
    assert_close(got["prev_delta"], exp["prev_delta"], TOL[FFMA], "prev_delta")


def test_accumulate_onto_existing_prev_1x1(ref, cuda_lib):
    # the plain-GEMM 1x1 path adds at the L2 onto prev (with the shortcut
    # pre-pass putting residual + old prev there first)
    spec = inputs.LayerSpec("1x1 acc", inputs.Geometry(2, 40, 8, 12, 56, 1, 1, 1, 0), 1, True)
    layer = inputs.make_layer(spec, 811, residual=True)
    seed = np.random.default_rng(4).standard_normal(layer["x"].shape).astype(np.float32)
    for math in MATHS:
        _, got = run_gpu(layer, math.values[0], accumulate=1, prev_init=seed)
        exp = oracle_chain(ref, layer, accumulate=1, prev_delta=seed)
        for k in KEYS:
            if exp.get(k) is not None:
                assert_close(got[k], exp[k], TOL[math.values[0]], f"1x1 acc {k}")


def test_strided_1x1_without_residual_stores_zero_classes(ref, cuda_lib):
    # 1x1 stride 2: three of the four stride phase classes have no kernel tap,
    # so the input gradient must store zeros there (no shortcut to add onto);
    # the classes run side by side in one launch
    spec = inputs.LayerSpec("1x1 s2", inputs.Geometry(3, 24, 14, 18, 40, 1, 1, 2, 0), 1, True)
    layer = inputs.make_layer(spec, 907, residual=False)
    for math in MATHS:
        _, got = run_gpu(layer, math.values[0])
        exp = oracle_chain(ref, layer)
        for k in KEYS:
            if exp.get(k) is not None:
                assert_close(got[k], exp[k], TOL[math.values[0]], f"1x1 s2 {k}")


def test_prev_delta_null_skips_dgrad(ref, cuda_lib):
    layer = config_layers(2, 2)[0]
    _, got = run_gpu(layer, TF32, with_prev=False)
    assert got["prev_delta"] is None
    exp = oracle_chain(ref, layer, want_prev=False)
    assert_close(got["dW"], exp["dW"], TOL[TF32], "dW")


@pytest.mark.parametrize("cid", [2, 4])
def test_dz_out_and_bn_identities(ref, cuda_lib, cid):
    layer = config_layers(cid, 2)[0]
    _, got = run_gpu(layer, FFMA, want_dz=True)
    exp = oracle_chain(ref, layer, want_dz=True)
    assert_close(got["dz"], exp["dz"], 1e-5, "dz")
    if layer["bn"]:
        s = got["dz"].sum(axis=(0, 2, 3))
        assert np.max(np.abs(s)) <= 1e-4 * np.max(np.abs(got["dz"])) * got["dz"][:, 0].size ** 0.5


@pytest.mark.parametrize("math", MATHS)
def test_residual_block_chained(ref, cuda_lib, math):
    """Config 5 as a chain: the 3x3 conv's prev_delta is the 1x1 conv's delta."""
    conv2, conv1 = config_layers(5, 2)
    dl2, got2 = run_gpu(conv2, math)
    exp2 = oracle_chain(ref, conv2)
    chained = dict(conv1, delta=exp2["prev_delta"].astype(np.float32))
    dl1 = DeviceLayer(chained, math=math)
    dl1.delta.copy_(dl2.prev)  # the GPU's own delta for the GPU chain
    dl1.run()
    assert dl1.status() == cba.CBA_OK
    got1 = dl1.results()
    exp1 = oracle_chain(ref, chained)
    tol = 2 * TOL[math]  # two layers of rounding
    for k in KEYS:
        assert_close(got1[k], exp1[k], tol, f"conv1 {k}")


def test_bounded_wait_reports_timeout(cuda_lib):
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    ws.zero_()
    assert cba.cba_selftest_bounded_wait(ws, 2000) == cba.CBA_OK
    assert cba.cba_get_status(ws) == cba.CBA_ERR_DEVICE_TIMEOUT
    assert cba.cba_get_status(ws) == cba.CBA_OK  # cleared
    # the context is still usable
    layer = config_layers(1, 2)[0]
    run_gpu(layer, TF32)


COMBOS = [(act, bn, zf, g, m) for act in (8, 6) for bn in (1, 2) for zf in (False, True)
          for g in (1, 2) for m in (TF32, FFMA)]


@pytest.mark.parametrize("act,bn,z_free,groups,math", COMBOS,
                         ids=[f"a{a}_bn{b}_z{int(z)}_g{g}_{'tf32' if m == TF32 else 'ffma'}"
                              for a, b, z, g, m in COMBOS])
def test_parity_feature_combinations(ref, cuda_lib, act, bn, z_free, groups, math):
    # the features that share workspace regions, together: another activation
    # (delta' pass), frozen statistics, z recomputed, groups; a small 3x3 layer
    base = (inputs.make_grouped_config(2, groups, batch=1) if groups > 1
            else config_layers(2, 1)[0])
    layer = inputs.with_activation(base, act)
    if bn == 2:
        layer = inputs.with_frozen_stats(layer, 40 + act)
    _, got = run_gpu(layer, math, want_dz=True, z_free=z_free)
    exp = oracle_chain(ref, layer, want_dz=True)
    for k in KEYS + ("dz",):
        if exp.get(k) is not None:
            assert_close(got[k], exp[k], TOL[math], f"{layer['name']} {k}")
