"""cba_bn_act_backward_noalloc (static device scratch, no workspace) against
the workspace entry point cba_conv_bn_act_backward, both through the C ABI.

The no-allocation pass must give the same db, dgamma and dz as the full call
(the same kernels; its reduction may use fewer blocks per channel, so the
bar is a tight relative tolerance rather than bit equality).  Several calls in
a row with different channel counts check that the scratch left behind by one
call does not leak into the next.  This file is collected last, so it also
runs after every other test has used the device.
"""
import ctypes

import numpy as np
import pytest
import torch

import activation_backward_gb300 as cba
from activation_backward_gb300 import _binding as B
from activation_backward_gb300 import inputs
from activation_backward_gb300.layer import DeviceLayer

TOL = 1e-6  # max |err| / max |ref| per tensor


def _close(got, exp, what):
    got = got.detach().cpu().numpy().astype(np.float64)
    exp = exp.detach().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), what
    err = float(np.max(np.abs(got - exp)))
    scale = float(np.max(np.abs(exp)))
    assert err <= TOL * scale + 1e-30, f"{what}: max|err| {err:.3e} vs max|ref| {scale:.3e}"


def _check_one(layer, seed):
    """One no-allocation call against the full call on the same inputs; db and
    dgamma start from the same non-zero values (both calls add)."""
    dl = DeviceLayer(layer, with_prev=False, want_dz=True)
    g = dl.geom
    gen = torch.Generator().manual_seed(seed)
    db0 = torch.randn(g.K, generator=gen).cuda()
    dg0 = torch.randn(g.K, generator=gen).cuda() if dl.dgamma is not None else None
    dl.db.copy_(db0)
    if dg0 is not None:
        dl.dgamma.copy_(dg0)
    dl.run()
    assert dl.status() == cba.CBA_OK

    db = db0.clone()
    dgamma = dg0.clone() if dg0 is not None else None
    dz = torch.full_like(dl.dz, float("nan"))
    rc = cba.cba_bn_act_backward_noalloc(dl.desc, dl.output, dl.z, dl.delta, dl.gamma, dl.mean,
                                         dl.var, db, dgamma, dz)
    assert rc == cba.CBA_OK
    torch.cuda.synchronize()
    name = layer["name"]
    _close(db, dl.db, f"{name} db")
    if dgamma is not None:
        _close(dgamma, dl.dgamma, f"{name} dgamma")
    _close(dz, dl.dz, f"{name} dz")


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_on_calls_in_a_row(cuda_lib):
    # K = 128 (BN, leaky), then K = 512 (BN, leaky, stride 2), then K = 50
    # (no BN, linear), then K = 128 again: each call reuses the scratch the
    # previous one left behind.
    cases = [(2, 2, 11), (3, 1, 12), (1, 4, 13), (2, 3, 14)]
    for cid, batch, seed in cases:
        layer = inputs.make_config(cid, batch=batch)[0]
        _check_one(layer, seed)
    # and with frozen BN statistics (batch_normalize = 2)
    _check_one(inputs.with_frozen_stats(inputs.make_config(2, batch=2)[0], 15), 16)
    # and with an activation the gradient_array pass handles (delta' goes
    # through dz, which is then transformed in place)
    _check_one(inputs.with_activation(inputs.make_config(2, batch=2)[0], cba.CBA_ACT_ELU), 17)


def _oracle_close(got, exp, what, tol=1e-5):
    got = got.detach().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), what
    err = float(np.max(np.abs(got - exp)))
    scale = float(np.max(np.abs(exp)))
    assert err <= tol * scale + 1e-30, f"{what}: max|err| {err:.3e} vs max|ref| {scale:.3e}"


def _noalloc_vs_oracle(ref, layer, stream=None):
    """One no-allocation call (db, dgamma starting from zero) against the
    oracle's activation-gradient + BN backward on the same fp32 inputs, at the
    fp32 bar of the FFMA mode (the pass does no TF32 rounding)."""
    dl = DeviceLayer(layer, with_prev=False, want_dz=True)
    db = torch.zeros_like(dl.db)
    dgamma = torch.zeros_like(dl.dgamma) if dl.dgamma is not None else None
    dz = torch.full_like(dl.dz, float("nan"))
    torch.cuda.synchronize()  # the uploads are done before another stream reads them
    rc = cba.cba_bn_act_backward_noalloc(dl.desc, dl.output, dl.z, dl.delta, dl.gamma, dl.mean,
                                         dl.var, db, dgamma, dz, stream=stream)
    assert rc == cba.CBA_OK
    torch.cuda.synchronize()
    e_dz, e_db, e_dg = ref.backward_dz(layer["output"], layer["z"], layer["delta"],
                                       layer["gamma"], layer["mean"], layer["var"],
                                       act=layer["act"], batch_normalize=layer["bn"],
                                       eps=layer["eps"])
    name = layer["name"]
    _oracle_close(db, e_db, f"{name} db")
    if dgamma is not None:
        _oracle_close(dgamma, e_dg, f"{name} dgamma")
    _oracle_close(dz, e_dz, f"{name} dz")


@pytest.mark.gpu
def test_noalloc_matches_the_oracle_including_the_largest_k_and_a_side_stream(ref, cuda_lib):
    # config 2 (BN, leaky) and config 4 (no BN, 90% zero delta) on torch's
    # current stream, against the oracle directly
    _noalloc_vs_oracle(ref, inputs.make_config(2, batch=2)[0])
    _noalloc_vs_oracle(ref, inputs.make_config(4, batch=2)[0])
    # K at the limit with one spatial position and N = 8: the 1 MiB scratch then
    # holds the counters (64 KiB), the coefficients (256 KiB) and only five
    # partials per channel
    spec = inputs.LayerSpec("noalloc_max_k", inputs.Geometry(8, 4, 1, 1, cba.CBA_NOALLOC_MAX_K,
                                                             1, 1), cba.CBA_ACT_LEAKY, True)
    _noalloc_vs_oracle(ref, inputs.make_layer(spec, 77))
    # on a stream other than torch's current one: the call still runs on the
    # device that holds delta, ordered on that stream
    side = torch.cuda.Stream()
    _noalloc_vs_oracle(ref, inputs.make_config(3, batch=1)[0], stream=side)


@pytest.mark.gpu
def test_noalloc_on_a_side_stream_matches_the_workspace_entry_point(cuda_lib):
    layer = inputs.make_config(5, batch=2)[0]
    dl = DeviceLayer(layer, with_prev=False, want_dz=True)
    dl.run()
    assert dl.status() == cba.CBA_OK
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    db = torch.zeros_like(dl.db)
    dgamma = torch.zeros_like(dl.dgamma)
    dz = torch.full_like(dl.dz, float("nan"))
    # the workspace call added onto dl's zero-initialised db / dgamma
    for _ in range(2):  # two calls in a row on the side stream
        db.zero_()
        dgamma.zero_()
        side.wait_stream(torch.cuda.current_stream())
        rc = cba.cba_bn_act_backward_noalloc(dl.desc, dl.output, dl.z, dl.delta, dl.gamma,
                                             dl.mean, dl.var, db, dgamma, dz, stream=side)
        assert rc == cba.CBA_OK
        side.synchronize()
        _close(db, dl.db, "side stream db")
        _close(dgamma, dl.dgamma, "side stream dgamma")
        _close(dz, dl.dz, "side stream dz")


def test_noalloc_rejects_k_beyond_the_scratch_limit():
    """K > CBA_NOALLOC_MAX_K returns CBA_ERR_SCRATCH_LIMIT before any CUDA
    call: the pointers are never dereferenced (host-side check, no GPU)."""
    from activation_backward_gb300 import build
    build.build()
    L = B.load()
    k = cba.CBA_NOALLOC_MAX_K + 1
    d = cba.make_desc(1, 1, 1, 1, k, 1, 1, act=cba.CBA_ACT_LEAKY, batch_normalize=1)
    fake = 1 << 20  # aligned, never dereferenced
    rc = L.cba_bn_act_backward_noalloc(ctypes.byref(d), *([fake] * 9), None)
    assert rc == cba.CBA_ERR_SCRATCH_LIMIT
    assert "CBA_NOALLOC_MAX_K" in cba.cba_error_string(rc)
    d_ok = cba.make_desc(1, 1, 1, 1, cba.CBA_NOALLOC_MAX_K, 1, 1)
    # at the limit the size check passes; a NULL delta is then the error
    rc = L.cba_bn_act_backward_noalloc(ctypes.byref(d_ok), *([fake] * 2), None, *([fake] * 6),
                                        None)
    assert rc == cba.CBA_ERR_ARG


def test_noalloc_needs_dz_for_other_activations():
    """Activations other than linear and leaky keep delta' in dz_out: without
    it the call returns CBA_ERR_UNSUPPORTED before any CUDA call."""
    from activation_backward_gb300 import build
    build.build()
    L = B.load()
    d = cba.make_desc(1, 2, 4, 4, 8, 1, 1, act=cba.CBA_ACT_TANH, batch_normalize=1)
    fake = 1 << 20  # aligned, never dereferenced
    rc = L.cba_bn_act_backward_noalloc(ctypes.byref(d), *([fake] * 8), None, None)
    assert rc == cba.CBA_ERR_UNSUPPORTED
