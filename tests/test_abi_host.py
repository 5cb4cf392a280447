"""CPU-side checks of the C ABI: the library builds, loads without a GPU and
exports every function that include/tp3d.h declares; no compute is called."""
import ctypes
import os
import re

import pytest

import tensor_transformer_layer_cube_gb300 as t

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(tp3d_\w+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    t.build()
    return t.lib()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert {"tp3d_linear", "tp3d_mlp", "tp3d_layer_fwd", "tp3d_layer_bwd", "tp3d_reshard"} <= declared
    h = ctypes.CDLL(t.LIB_PATH)
    for name in sorted(declared):
        assert hasattr(h, name), name


def test_status_strings(lib):
    for code in range(9):
        assert t.tp3d_status_string(code)
    assert "wait" in t.tp3d_status_string(6)


def test_binding_wraps_every_declared_function():
    for name in _declared():
        assert hasattr(t, name), name


def test_struct_sizes_match_the_header(lib):
    assert ctypes.sizeof(t.tp3d_layout) == 16
    assert ctypes.sizeof(t.tp3d_layer_cfg) == 32
    assert ctypes.sizeof(t.tp3d_layer_params) == 12 * ctypes.sizeof(ctypes.c_void_p)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # no fallback path: without the built library, loading and every compute
    # entry point raise instead of computing anything on the host
    monkeypatch.setattr(t, "_lib", None)
    monkeypatch.setattr(t, "LIB_PATH", str(tmp_path / "absent" / "libtp3d.so"))
    with pytest.raises(RuntimeError, match="missing"):
        t.lib()
    with pytest.raises(RuntimeError, match="missing"):
        t.tp3d_linear(None, 2, 0, 64, 64, 64, 1, None, None, None, 0, None)
    with pytest.raises(RuntimeError, match="missing"):
        t.tp3d_reshard(None, 8, 8, 2, t.tp3d_layout(), None, t.tp3d_layout(), None)
