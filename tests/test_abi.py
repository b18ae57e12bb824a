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
