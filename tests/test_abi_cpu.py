"""Host-side checks of the C-ABI library that need no GPU.

* the library builds for sm_103a and exports every function the header
  declares;
* argument validation happens on the host and returns the documented status
  codes before anything touches a device.
"""
import ctypes

import pytest

import nvfp4_weight_only_w4a16_gb300 as P
from nvfp4_weight_only_w4a16_gb300.binding import Config


@pytest.fixture(scope="module")
def lib():
    P.build()
    return P.load_library()


def test_exports_every_header_symbol(lib):
    names = P.header_functions()
    assert "nvfp4_moe_create" in names and "nvfp4_moe_forward" in names and "nvfp4_moe_pack" in names
    assert "nvfp4_linear_create" in names and "nvfp4_linear_forward" in names and "nvfp4_linear_pack" in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(10):
        s = lib.nvfp4_moe_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.nvfp4_moe_status_string(99).decode() == "unknown status"


def _create(lib, **kw):
    base = dict(num_experts=8, hidden=256, inter=512, max_tokens=16, max_top_k=2,
                decode_max_tokens=16, logits_dtype=0, device=0, out_dtype=0, num_shared_experts=0)
    base.update(kw)
    cfg = Config(**base)
    h = ctypes.c_void_p()
    return lib.nvfp4_moe_create(ctypes.byref(cfg), ctypes.byref(h)), h


@pytest.mark.parametrize("kw", [
    dict(num_experts=0), dict(num_experts=257), dict(hidden=100), dict(hidden=192),
    dict(inter=64), dict(max_tokens=0), dict(max_top_k=0), dict(max_top_k=17),
    dict(num_experts=4, max_top_k=5), dict(decode_max_tokens=17),
    dict(num_shared_experts=2), dict(num_shared_experts=-1),
    dict(num_experts=256, num_shared_experts=1), dict(num_experts=32, max_top_k=16, num_shared_experts=1),
])
def test_create_rejects_bad_shapes(lib, kw):
    st, h = _create(lib, **kw)
    assert st == P.STATUS_CODE["NVFP4_MOE_ERR_UNSUPPORTED_SHAPE"]
    assert not h.value


def test_create_rejects_bad_dtype_and_nulls(lib):
    st, h = _create(lib, logits_dtype=7)
    assert st == P.STATUS_CODE["NVFP4_MOE_ERR_INVALID_ARG"]
    st, h = _create(lib, out_dtype=2)
    assert st == P.STATUS_CODE["NVFP4_MOE_ERR_INVALID_ARG"]
    assert lib.nvfp4_moe_create(None, None) == P.STATUS_CODE["NVFP4_MOE_ERR_INVALID_ARG"]


def test_null_handle_calls(lib):
    inv = P.STATUS_CODE["NVFP4_MOE_ERR_INVALID_ARG"]
    assert lib.nvfp4_moe_forward(None, None, 1, 1, None, None, None) == inv
    assert lib.nvfp4_moe_pack(None, None, None, None, None, None, None) == inv
    assert lib.nvfp4_moe_set_path(None, 0) == inv
    assert lib.nvfp4_moe_debug_dequant(None, 0, 0, None, None) == inv
    assert lib.nvfp4_moe_debug_set_fault(None, 0) == inv
    assert lib.nvfp4_moe_debug_packed_blob(None, None, 0, None) == inv
    lib.nvfp4_moe_destroy(None)  # no-op


def test_header_has_no_activation_scale():
    # weight-only: the forward takes logits, x and out, never an input scale
    text = open(P.binding.HEADER).read()
    fwd = text[text.index("nvfp4_moe_status nvfp4_moe_forward("):]
    fwd = fwd[:fwd.index(";")]
    assert "scale" not in fwd


def _create_linear(lib, **kw):
    base = dict(out_features=272, in_features=256, max_tokens=16, decode_max_tokens=16, out_dtype=0, device=0)
    base.update(kw)
    cfg = P.binding.LinearConfig(**base)
    h = ctypes.c_void_p()
    return lib.nvfp4_linear_create(ctypes.byref(cfg), ctypes.byref(h)), h


@pytest.mark.parametrize("kw", [
    dict(out_features=0), dict(out_features=8), dict(out_features=100), dict(out_features=16400),
    dict(in_features=64), dict(in_features=200), dict(max_tokens=0), dict(decode_max_tokens=17),
])
def test_linear_create_rejects_bad_shapes(lib, kw):
    st, h = _create_linear(lib, **kw)
    assert st == P.STATUS_CODE["NVFP4_MOE_ERR_UNSUPPORTED_SHAPE"]
    assert not h.value


def test_linear_null_and_bad_args(lib):
    inv = P.STATUS_CODE["NVFP4_MOE_ERR_INVALID_ARG"]
    st, h = _create_linear(lib, out_dtype=3)
    assert st == inv and not h.value
    assert lib.nvfp4_linear_create(None, None) == inv
    assert lib.nvfp4_linear_pack(None, None, None, None, None) == inv
    assert lib.nvfp4_linear_forward(None, 1, None, None, None) == inv


def test_linear_header_has_no_activation_scale():
    text = open(P.binding.HEADER).read()
    fwd = text[text.index("nvfp4_moe_status nvfp4_linear_forward("):]
    fwd = fwd[:fwd.index(";")]
    assert "scale" not in fwd


def test_status_word_decoding_on_the_host():
    """The device status word's bits map to status codes without a GPU: bit 0
    a bounded wait that gave up, bit 1 a device-side bounds check."""
    lib = P.binding.load_library()
    code = P.STATUS_CODE
    assert lib.nvfp4_moe_decode_status_word(0) == code["NVFP4_MOE_OK"]
    assert lib.nvfp4_moe_decode_status_word(1) == code["NVFP4_MOE_ERR_TIMEOUT"]
    assert lib.nvfp4_moe_decode_status_word(2) == code["NVFP4_MOE_ERR_DEVICE_CHECK"]
    assert lib.nvfp4_moe_decode_status_word(3) == code["NVFP4_MOE_ERR_TIMEOUT"]
