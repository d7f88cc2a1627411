"""Host-side checks of the C ABI (no GPU needed, no compute calls).

The library must load and export every symbol include/cba.h declares;
descriptor validation, the workspace query and the argument checks all run on
the host and return their error codes before any CUDA call is made.  Every
call below fails validation, so no pointer is ever dereferenced.
"""
import ctypes
import os
import re

import pytest

import activation_backward_gb300 as cba
from activation_backward_gb300 import _binding as B
from activation_backward_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from activation_backward_gb300 import build
    build.build()
    return B.load()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "cba.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cba_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert "cba_conv_bn_act_backward" in names and "cba_workspace_bytes" in names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(B.EXPORTS) == names


def test_version_and_error_strings(lib):
    assert cba.cba_version() >= 100
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = cba.cba_error_string(code)
        assert s and "unknown" not in s
    assert "unknown" in cba.cba_error_string(-99)


@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_workspace_query_for_the_workloads(lib, cid):
    for layer_geom in ([inputs.CONFIGS[cid].geom] + ([inputs.BLOCK_CONV2] if cid == 5 else [])):
        g = layer_geom
        for math in (cba.CBA_MATH_TF32, cba.CBA_MATH_FFMA):
            d = cba.make_desc(g.N, g.C, g.H, g.W, g.K, g.R, g.S, g.stride, g.pad, math=math)
            n = cba.cba_workspace_bytes(d)
            assert n > 0 and n % 256 == 0
            assert n < 1 << 30  # bounded scratch


BAD = [dict(N=0), dict(C=-1), dict(K=0), dict(R=0), dict(stride=0), dict(pad=-1), dict(act=14),
       dict(math=3), dict(batch_normalize=3), dict(batch_normalize=-1), dict(accumulate=5), dict(H=2, R=5, pad=0),
       dict(eps=float("nan"))]


@pytest.mark.parametrize("bad", BAD, ids=[str(b) for b in BAD])
def test_invalid_descriptor_is_rejected(lib, bad):
    kw = dict(N=2, C=3, H=5, W=5, K=4, R=3, S=3, stride=1, pad=1, act=1, batch_normalize=1,
              accumulate=0, eps=1e-5, math=0)
    kw.update(bad)
    d = B.cba_desc_t(**kw)
    assert lib.cba_workspace_bytes(ctypes.byref(d)) == 0
    fake = 0x10000
    rc = lib.cba_conv_bn_act_backward(ctypes.byref(d), *([fake] * 15), 1 << 20, None)
    assert rc == cba.CBA_ERR_ARG


def test_too_large_is_unsupported(lib):
    d = cba.make_desc(1 << 12, 1 << 10, 1 << 5, 1 << 5, 4, 1, 1)  # 2^32 input elements
    assert lib.cba_workspace_bytes(ctypes.byref(d)) == 0
    rc = lib.cba_conv_bn_act_backward(ctypes.byref(d), *([0x10000] * 15), 1 << 20, None)
    assert rc == B.CBA_ERR_UNSUPPORTED


def _call(lib, d, **ptrs):
    names = ["x", "output", "z", "delta", "W", "gamma", "mean", "var", "residual", "dW", "db",
             "dgamma", "prev", "dz", "ws"]
    base = {n: 0x100000 + 0x1000 * i for i, n in enumerate(names)}
    base["dz"] = None
    base["residual"] = None
    base.update(ptrs)
    wsb = ptrs.get("wsb", 1 << 30)
    args = [base[n] for n in names]
    return lib.cba_conv_bn_act_backward(ctypes.byref(d), *args, wsb, None)


def test_required_pointers(lib):
    d = cba.make_desc(2, 3, 5, 5, 4, 3, 3, 1, 1, act=cba.CBA_ACT_LEAKY, batch_normalize=1)
    for name in ("x", "delta", "W", "dW", "db", "output", "gamma", "mean", "var", "dgamma"):
        assert _call(lib, d, **{name: None}) == cba.CBA_ERR_ARG, name
    # with BN, z may be NULL (recomputed), but only with the larger workspace:
    # the plain size stops at the workspace check, before any launch
    plain = lib.cba_workspace_bytes(ctypes.byref(d))
    assert _call(lib, d, z=None, wsb=plain) == cba.CBA_ERR_WORKSPACE
    # linear without BN: output, z, gamma, mean, var, dgamma may be NULL; the
    # call then stops at the (too small) workspace check, still before any launch
    d2 = cba.make_desc(2, 3, 5, 5, 4, 3, 3, 1, 1, act=cba.CBA_ACT_LINEAR, batch_normalize=0)
    rc = _call(lib, d2, output=None, z=None, gamma=None, mean=None, var=None, dgamma=None,
               wsb=16)
    assert rc == cba.CBA_ERR_WORKSPACE


def test_alignment_and_workspace_checks(lib):
    d = cba.make_desc(2, 3, 5, 5, 4, 3, 3, 1, 1)
    assert _call(lib, d, x=0x100004) == cba.CBA_ERR_ALIGN
    assert _call(lib, d, prev=0x100008) == cba.CBA_ERR_ALIGN
    assert _call(lib, d, ws=None) == cba.CBA_ERR_WORKSPACE
    need = lib.cba_workspace_bytes(ctypes.byref(d))
    assert _call(lib, d, wsb=need - 1) == cba.CBA_ERR_WORKSPACE
    assert _call(lib, d, ws=0x100010) == cba.CBA_ERR_ALIGN  # workspace needs 256 B


def test_status_and_selftest_argument_checks(lib):
    assert lib.cba_get_status(None, 1024, None) == cba.CBA_ERR_WORKSPACE
    assert lib.cba_selftest_bounded_wait(None, 1024, 100, None) == cba.CBA_ERR_WORKSPACE
    assert lib.cba_selftest_bounded_wait(0x100000, 1024, 0, None) == cba.CBA_ERR_ARG
    assert lib.cba_selftest_bounded_wait(0x100000, 1024, 3000000, None) == cba.CBA_ERR_ARG


def test_binding_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(RuntimeError):
        B._lib_saved = B._lib
        try:
            B._lib = None
            B.load(str(tmp_path / "missing.so"))
        finally:
            B._lib = B._lib_saved


def test_workspace_query_for_z_free_calls(lib):
    d = cba.make_desc(2, 3, 5, 5, 4, 3, 3, 1, 1, act=cba.CBA_ACT_LEAKY, batch_normalize=1)
    base = lib.cba_workspace_bytes(ctypes.byref(d))
    zfree = lib.cba_workspace_bytes_ex(ctypes.byref(d), cba.CBA_WS_RECOMPUTE_Z)
    assert lib.cba_workspace_bytes_ex(ctypes.byref(d), 0) == base
    assert zfree >= base + 2 * 4 * 5 * 5 * 4  # room for z [N, K, P, Q] fp32
    assert lib.cba_workspace_bytes_ex(ctypes.byref(d), 2) == 0  # unknown flag
    d0 = cba.make_desc(2, 3, 5, 5, 4, 3, 3, 1, 1, act=cba.CBA_ACT_LINEAR, batch_normalize=0)
    assert lib.cba_workspace_bytes_ex(ctypes.byref(d0), cba.CBA_WS_RECOMPUTE_Z) == \
        lib.cba_workspace_bytes(ctypes.byref(d0))  # no BN, no z


def test_workspace_query_for_grouped_calls(lib):
    d = cba.make_desc(2, 8, 5, 5, 12, 3, 3, 1, 1, act=cba.CBA_ACT_LEAKY, batch_normalize=1)
    assert lib.cba_workspace_bytes_grouped(ctypes.byref(d), 1, 0) == \
        lib.cba_workspace_bytes(ctypes.byref(d))
    g4 = lib.cba_workspace_bytes_grouped(ctypes.byref(d), 4, 0)
    assert g4 > 0
    assert lib.cba_workspace_bytes_grouped(ctypes.byref(d), 4, cba.CBA_WS_RECOMPUTE_Z) > g4
    assert lib.cba_workspace_bytes_grouped(ctypes.byref(d), 3, 0) == 0  # 3 does not divide 8
    assert lib.cba_workspace_bytes_grouped(ctypes.byref(d), 0, 0) == 0
    assert lib.cba_workspace_bytes_grouped(ctypes.byref(d), 4, 2) == 0  # unknown flag


def test_plan_info_query(lib):
    d = cba.make_desc(2, 8, 5, 5, 12, 3, 3, 1, 1, act=cba.CBA_ACT_LEAKY, batch_normalize=1)
    path, rd, wr = cba.cba_plan_info(d)
    assert path in (cba.CBA_PATH_FFMA, cba.CBA_PATH_TC_ROWS, cba.CBA_PATH_TC_BATCH_INNER,
                    cba.CBA_PATH_TC_GEMM_1X1)
    if path == cba.CBA_PATH_FFMA:  # no operand layout pass
        assert rd == 0 and wr == 0
    else:
        assert rd >= 3 * 4 * 2 * 12 * 5 * 5 and wr > 0  # delta, output, z read
    f = cba.make_desc(2, 8, 5, 5, 12, 3, 3, 1, 1, act=cba.CBA_ACT_LEAKY, batch_normalize=1,
                      math=cba.CBA_MATH_FFMA)
    assert cba.cba_plan_info(f) == (cba.CBA_PATH_FFMA, 0, 0)
    with pytest.raises(cba.CbaError):
        cba.cba_plan_info(d, groups=3)  # 3 does not divide 8
    bad = cba.make_desc(0, 8, 5, 5, 12, 3, 3, 1, 1)
    with pytest.raises(cba.CbaError):
        cba.cba_plan_info(bad)
    info = B.cba_plan_info_t()
    assert lib.cba_plan_info(ctypes.byref(d), 1, 1, None) == cba.CBA_ERR_ARG
    assert lib.cba_plan_info(None, 1, 1, ctypes.byref(info)) == cba.CBA_ERR_ARG
