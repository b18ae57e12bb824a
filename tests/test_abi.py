"""The C-ABI library builds, loads without a GPU and exports every function
that include/*.h declares; host-side argument checks of sf_create run without
touching the device."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\*?\s+\*?(sf\w*)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from sparse_reuse_gb300 import build
    build.build()
    import sparse_reuse_gb300 as sf
    return sf


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"sf_create", "sf_verify", "sf_destroy", "sf_status_str"} <= names
    raw = ctypes.CDLL(lib.LIB_PATH)
    for n in sorted(names):
        assert hasattr(raw, n), f"{n} declared in include/ but not exported"
    assert set(lib.EXPORTS) >= {n for n in names if n.startswith("sf_")}


def test_status_strings(lib):
    for st in range(8):
        assert lib.lib.sf_status_str(st)
    assert lib.lib.sf_status_str(99) == b"unknown status"


def _shapes(lib, **kw):
    base = dict(n_layers=1, d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=64, d_ffn=688,
                dtype=lib.SF_F32, rms_eps=1e-6, rope_theta=1e4, block_len=32, max_requests=1,
                max_branches=3, max_prefix=64)
    base.update(kw)
    return lib.SfShapes(*[base[f] for f, _ in lib.SfShapes._fields_])


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), 4), (dict(d_model=200), 4), (dict(n_q_heads=5), 4), (dict(block_len=65), 4),
    (dict(max_requests=64, max_branches=64), 4), (dict(n_layers=0), 1), (dict(dtype=7), 1),
    (dict(rms_eps=-1.0), 1),
])
def test_create_rejects_bad_shapes_before_any_device_work(lib, kw, status):
    ctx = ctypes.c_void_p()
    w = (lib.SfLayerWeights * 1)(lib.SfLayerWeights(*([1] * 9)))
    st = lib.lib.sf_create(ctypes.byref(_shapes(lib, **kw)), w, ctypes.byref(ctx))
    assert st == status and not ctx.value


def test_create_rejects_null_weights(lib):
    ctx = ctypes.c_void_p()
    w = (lib.SfLayerWeights * 1)(lib.SfLayerWeights(*([1] * 8 + [0])))
    assert lib.lib.sf_create(ctypes.byref(_shapes(lib)), w, ctypes.byref(ctx)) == lib.SF_ERR_INVALID_ARG
    assert lib.lib.sf_create(None, w, ctypes.byref(ctx)) == lib.SF_ERR_INVALID_ARG


def _gate_noalloc(lib, hidden, dtype, parent, h_out, rc, delta=0.1, R=1, B=2):
    par = (ctypes.c_int32 * parent.size)(*parent.ravel().tolist())
    # device addresses are never dereferenced: every case is refused on the host
    return lib.lib.sfk_gate_noalloc(None, hidden, dtype, par, R, B, 32, 256, delta, h_out, 16, rc, 16, 16, 16)


def test_noalloc_gate_host_checks_before_any_device_work(lib):
    import numpy as np
    good, bad_tree = np.array([[-1, 0, 1]], np.int32), np.array([[0, 0, 1]], np.int32)
    assert _gate_noalloc(lib, 16, lib.SF_F32, bad_tree, 16, 16) == lib.SF_ERR_TREE
    assert _gate_noalloc(lib, 16, lib.SF_F32, good, 16, 16, delta=float("nan")) == lib.SF_ERR_INVALID_ARG
    assert _gate_noalloc(lib, 16, lib.SF_F32, np.tile(good, (100, 1)), 16, 16, R=100) == lib.SF_ERR_SHAPE
    # misaligned buffers are refused before the tree is looked at: fp32 rows
    # need 16 bytes, bf16 rows 8, H_out 16, the int32 outputs 4
    for dtype, hidden, h_out, rc in ((lib.SF_F32, 24, 16, 16), (lib.SF_BF16, 20, 16, 16),
                                     (lib.SF_F32, 16, 24, 16), (lib.SF_F32, 16, 16, 18)):
        assert _gate_noalloc(lib, hidden, dtype, bad_tree, h_out, rc) == lib.SF_ERR_INVALID_ARG
    # bf16 rows 8-byte aligned pass the alignment check (and stop at the tree)
    assert _gate_noalloc(lib, 24, lib.SF_BF16, bad_tree, 16, 16) == lib.SF_ERR_TREE


def test_gemm_host_checks_before_any_device_work(lib):
    f = lib.lib.sfk_gemm_bf16
    # M not a multiple of 128, K not a multiple of 64, a cluster larger than 8,
    # a misaligned operand: all refused without a launch
    assert f(None, 16, 64, 16, 100, 64, None, 1, 16, 100, 1, None) == lib.SF_ERR_INVALID_ARG
    assert f(None, 16, 64, 16, 128, 96, None, 1, 16, 128, 1, None) == lib.SF_ERR_INVALID_ARG
    assert f(None, 16, 64, 16, 128, 1024, None, 1, 16, 128, 9, None) == lib.SF_ERR_INVALID_ARG
    assert f(None, 24, 64, 16, 128, 1024, None, 1, 16, 128, 1, None) == lib.SF_ERR_INVALID_ARG
    assert f(None, 16, 64, 24, 128, 1024, None, 1, 16, 128, 1, None) == lib.SF_ERR_INVALID_ARG
