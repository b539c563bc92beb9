"""The C ABI without a GPU: symbols, host-only logic, argument rejection.

Nothing here launches a kernel; every rejected call must return before it
would touch the device.
"""
import ctypes as C
import re
from pathlib import Path

import numpy as np
import pytest

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def pi():
    import __graft_entry__
    __graft_entry__._builder().build()
    import activation_sparse_rank_gb300 as pi
    return pi


def _declared():
    text = (ROOT / "include" / "pi.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pi_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["pi_layer_create", "pi_layer_destroy", "pi_predict", "pi_compact_active",
              "pi_sparse_ffn", "pi_ffn_dense_ref", "pi_workspace_bytes", "pi_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(pi):
    lib = C.CDLL(str(pi.lib_path))
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_hot_first_perm_matches_oracle(pi):
    from oracle import ffn as O
    rng = np.random.default_rng(3)
    for n in (1, 7, 1000, 4096):
        counts = rng.integers(0, 20, n).astype(np.int32)
        np.testing.assert_array_equal(pi.hot_first_perm(counts), O.hot_first_order(counts))


def test_status_strings(pi):
    assert pi.lib.pi_status_string(0) == b"PI_OK"
    assert pi.lib.pi_status_string(5) == b"PI_ERR_DEVICE_CHECK"


def test_rejections_before_any_launch(pi):
    lib = pi.lib
    h = C.c_void_p()
    assert lib.pi_layer_create(None, None, None, None) == 1
    assert lib.pi_layer_create(C.byref(h), None, None, None) == 1
    assert b"desc" in lib.pi_last_error()
    bad = pi.binding.pi_layer_desc(1004, 64, 16, 0, None, None, None, None, None, None, None)
    assert lib.pi_layer_create(C.byref(h), C.byref(bad), None, None) == 2   # d % 8 != 0
    bad = pi.binding.pi_layer_desc(64, 64, 12, 0, None, None, None, None, None, None, None)
    assert lib.pi_layer_create(C.byref(h), C.byref(bad), None, None) == 2   # rank % 8 != 0
    bad = pi.binding.pi_layer_desc(64, 64, 16, 7, None, None, None, None, None, None, None)
    assert lib.pi_layer_create(C.byref(h), C.byref(bad), None, None) == 1   # act
    ok_shape = pi.binding.pi_layer_desc(64, 64, 16, 0, None, None, None, None, None, None, None)
    assert lib.pi_layer_create(C.byref(h), C.byref(ok_shape), None, None) == 1  # NULL weights
    assert not h.value
    assert lib.pi_predict(None, None, 1, None, None, None, 0, None) == 1
    assert lib.pi_sparse_ffn(None, None, 1, None, None, None, None, 0, None) == 1
    assert lib.pi_compact_active(None, None, 1, None, None, None) == 1
    assert lib.pi_ffn_dense_ref(None, None, 1, None, None, 0, None) == 1
    assert lib.pi_layer_forward(None, None, 1, None, None, None, None, 0, None) == 1
    assert lib.pi_workspace_bytes(None, 1) == 0
    assert lib.pi_hot_first_perm(None, 4, None) == 1
    assert lib.pi_layer_destroy(None) == 0


def test_binding_constants_match_the_header(pi):
    text = (ROOT / "include" / "pi.h").read_text()
    defs = dict(re.findall(r"#define\s+(PI_[A-Z_]+)\s+\(?([0-9]+)", text))
    assert int(defs["PI_MAX_BATCH"]) == pi.binding.PI_MAX_BATCH
    assert int(defs["PI_STACK_LAYERS_PER_LAUNCH"]) == pi.binding.PI_STACK_LAYERS_PER_LAUNCH
    enums = dict(re.findall(r"\b(PI_(?:ACT|ROWS)_[A-Z0-9_]+)\s*=\s*([0-9]+)", text))
    for name, value in enums.items():
        assert getattr(pi.binding, name) == int(value), name


def test_binding_checks_arguments_before_the_library(pi):
    # argument marshalling refuses host tensors, wrong dtypes and unknown
    # activations before any pointer reaches the C ABI
    import torch
    W = torch.zeros(8, 8, dtype=torch.float16)
    b = torch.zeros(8)
    with pytest.raises(ValueError):
        pi.binding.make_desc(W, None, b, W, W, W, None, "gelu")
    with pytest.raises(TypeError):
        pi.binding.make_desc(W, None, b, W, W, W, None, "relu")       # host memory
    with pytest.raises(TypeError):
        pi.Layer.from_dict(dict(W_up=W, W_gate=None, b=b, W_down=W, W_p1=W, W_p2=W,
                                c_p=None, act="relu"))

