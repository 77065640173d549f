"""The C-ABI library builds for sm_103a, loads without a GPU and exports every
function include/dflash.h declares; host-side argument checks answer without
touching the device."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def lib():
    from block_speculative_drafting_gb300.csrc.build import build
    path = build()
    return C.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_\w+)\s*\(", text)) - {"DFLASH_MAT_LAYER"})


def test_header_declares_the_path():
    names = declared_functions()
    for must in ("dflash_init", "dflash_ctx_append", "dflash_block", "dflash_seq_new", "dflash_free"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_python_binding_signatures(lib):
    from block_speculative_drafting_gb300 import _abi
    assert set(_abi._SIGS) == set(declared_functions())
    _abi.load()


def test_geometry_rejected_before_any_device_work():
    import block_speculative_drafting_gb300 as dfl
    import workloads as W
    bad = [dict(head_dim=96), dict(hidden=200), dict(heads=6, kv_heads=4), dict(window=-1), dict(windows=(4, -2)),
           dict(block=1), dict(conv_kernel=-1), dict(conv_kernel=2, conv_group=6), dict(conv_kernel=2, conv_group=96),
           dict(selector_rank=4, selector_top=0), dict(selector_rank=4, selector_top=33)]
    base = W.WORKLOADS["tiny_f32"].geom
    import dataclasses
    w = W.make_weights(base)
    for change in bad:
        g = dataclasses.replace(base, **change)
        with pytest.raises(dfl.DFlashError) as e:
            dfl.Model(g, w)
        assert e.value.code == dfl._abi.DFLASH_EGEOM


def test_null_arguments(lib):
    import block_speculative_drafting_gb300 as dfl
    L = dfl.lib()
    out = C.c_void_p()
    assert L.dflash_init(None, None, 0, None, C.byref(out)) == dfl._abi.DFLASH_EINVAL
    assert b"NULL" in L.dflash_last_error(None)
    assert L.dflash_block(None, None, 0, None, None, 2, None, None, 0, None) == dfl._abi.DFLASH_EINVAL
    assert L.dflash_truncate(None, 0) == dfl._abi.DFLASH_EINVAL
