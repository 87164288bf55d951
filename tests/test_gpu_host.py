"""nvfp4_moe_forward_host: the decode forward with the router logits, x and
the output in page-locked host memory, read and written in place by the
decode kernel.  It must give exactly what nvfp4_moe_forward gives on device
buffers (the same kernel on the same values), and refuse, before launching
anything, memory the device cannot address in place and the other paths."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import nvfp4_weight_only_w4a16_gb300 as P
from synth import CONFIGS, make_inputs
from tests.test_gpu_parity import DEV, _layer, assert_layer_close

pytestmark = pytest.mark.gpu


def _pinned_io(inp):
    T, H = inp.x_bits.shape
    h_logits = torch.from_numpy(np.ascontiguousarray(inp.logits)).pin_memory()
    h_x = torch.from_numpy(inp.x_bits.view(np.int16)).pin_memory().view(torch.bfloat16)
    h_out = torch.full((T, H), -1, dtype=torch.int16).pin_memory().view(torch.bfloat16)
    return h_logits, h_x, h_out


def _device_forward(L, inp, k):
    T, H = inp.x_bits.shape
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    x = torch.from_numpy(inp.x_bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    L.nvfp4_moe_forward(torch.from_numpy(np.ascontiguousarray(inp.logits)).to(DEV), x, k, out)
    torch.cuda.synchronize()
    return out.cpu().view(torch.int16).numpy()


@pytest.mark.parametrize("name", ["tiny", "decode_mtp", "decode_c16"])
def test_forward_host_equals_device_forward(name):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg)
    L = _layer(cfg)
    L.nvfp4_moe_set_path(P.PATH_AUTO)
    h_logits, h_x, h_out = _pinned_io(inp)
    for _ in range(2):  # twice: the second call overwrites the first one's result in place
        L.nvfp4_moe_forward_host(h_logits, h_x, cfg.top_k, h_out)
        torch.cuda.synchronize()
    st, _ = L.nvfp4_moe_get_status()
    assert st == 0, P.STATUS[st]
    got = h_out.view(torch.int16).numpy().copy()
    np.testing.assert_array_equal(got, _device_forward(L, inp, cfg.top_k))
    if name == "tiny":
        ref = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k)
        assert_layer_close(O.bf16_bits_to_f64(got.view(np.uint16)), ref)


def test_forward_host_refuses_what_it_cannot_read_in_place():
    cfg = CONFIGS["tiny"]
    inp = make_inputs(cfg)
    L = _layer(cfg)
    T, H = inp.x_bits.shape
    k = cfg.top_k
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    invalid, unsupported = P.STATUS_CODE["NVFP4_MOE_ERR_INVALID_ARG"], P.STATUS_CODE["NVFP4_MOE_ERR_UNSUPPORTED_SHAPE"]
    h_logits, h_x, h_out = _pinned_io(inp)
    hp = [ctypes.c_void_p(t.data_ptr()) for t in (h_logits, h_x, h_out)]

    # device memory is not host memory
    d_logits = torch.from_numpy(np.ascontiguousarray(inp.logits)).to(DEV)
    d_x = torch.from_numpy(inp.x_bits.view(np.int16)).to(DEV)
    d_out = torch.empty((T, H), dtype=torch.int16, device=DEV)
    st = L.lib.nvfp4_moe_forward_host(L.h, ctypes.c_void_p(d_logits.data_ptr()), T, k,
                                      ctypes.c_void_p(d_x.data_ptr()), ctypes.c_void_p(d_out.data_ptr()), stream)
    assert st == invalid, P.STATUS.get(st, st)
    # one pinned buffer is not enough: every pointer is checked
    st = L.lib.nvfp4_moe_forward_host(L.h, hp[0], T, k, hp[1], ctypes.c_void_p(d_out.data_ptr()), stream)
    assert st == invalid, P.STATUS.get(st, st)

    # the prefill path copies x and the logits in bulk: refused
    L.nvfp4_moe_set_path(P.PATH_PREFILL)
    try:
        st = L.lib.nvfp4_moe_forward_host(L.h, hp[0], T, k, hp[1], hp[2], stream)
        assert st == unsupported, P.STATUS.get(st, st)
    finally:
        L.nvfp4_moe_set_path(P.PATH_AUTO)

    # the binding wants pinned CPU tensors
    with pytest.raises(ValueError):
        L.nvfp4_moe_forward_host(torch.from_numpy(np.ascontiguousarray(inp.logits)), h_x, k, h_out)

    # pageable memory: refused, unless this system reports it as mapped host memory -- then
    # the result must be the device forward's
    lg = np.ascontiguousarray(inp.logits)
    xb = np.ascontiguousarray(inp.x_bits)
    ob = np.zeros((T, H), np.uint16)
    st = L.lib.nvfp4_moe_forward_host(L.h, ctypes.c_void_p(lg.ctypes.data), T, k, ctypes.c_void_p(xb.ctypes.data),
                                      ctypes.c_void_p(ob.ctypes.data), stream)
    torch.cuda.synchronize()
    assert st in (invalid, P.STATUS_CODE["NVFP4_MOE_OK"]), P.STATUS.get(st, st)
    if st == P.STATUS_CODE["NVFP4_MOE_OK"]:
        np.testing.assert_array_equal(ob.view(np.int16), _device_forward(L, inp, k))

    # nothing above disturbed the handle
    st, _ = L.nvfp4_moe_get_status()
    assert st == 0, P.STATUS[st]
    L.nvfp4_moe_forward_host(h_logits, h_x, k, h_out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(h_out.view(torch.int16).numpy(), _device_forward(L, inp, k))
