"""The allocation-free decode forward, checked against the handle-based one
and against the float64 oracle.

nvfp4_moe_forward_decode_static serves callers that cannot call cudaMalloc
(global-mode graph capture, plugins inside a framework that owns all device
memory, static-memory runtimes): it takes only caller memory and keeps its
intermediates in a static device array.  Its device-side errors reach the
caller through nvfp4_moe_static_get_status.  This file runs last so that, if
it fails, a run that stops at the first failure has already run everything
else; it needs no state from the other tests.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import nvfp4_weight_only_w4a16_gb300 as P
import oracle as O
from synth import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _close(got, ref):
    # the layer tolerance of the parity tests, with the handle's output as reference
    err = np.abs(got - ref)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.all(err <= 2e-2 * rms + 2.0 ** -8 * np.abs(got)), (err.max(), rms)
    assert err.mean() / np.abs(ref).mean() <= 5e-3


def _assert_layer_bounds(got, ref):
    # the layer bounds against the oracle: max|err| <= 2e-2 RMS (plus the BF16
    # output rounding, 2^-8 of each value), mean relative error <= 5e-3
    err = np.abs(got - ref)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.all(err <= 2e-2 * rms + 2.0 ** -8 * np.abs(got)), (err.max(), rms)
    assert err.mean() / np.abs(ref).mean() <= 5e-3, err.mean() / np.abs(ref).mean()
    cos = float(np.sum(got * ref) / (np.linalg.norm(got) * np.linalg.norm(ref)))
    assert cos >= 0.9999 and 0.99 <= np.linalg.norm(got) / np.linalg.norm(ref) <= 1.01


def _static(blob, gscale, cfg, logits, x, out):
    st = P.binding.nvfp4_moe_forward_decode_static(blob, gscale, cfg.num_experts, cfg.hidden, cfg.inter,
                                                   logits, cfg.top_k, x, out)
    assert st == 0, P.STATUS[st]


def _run_both(name, token_slices):
    P.build()
    cfg = CONFIGS[name]
    inp = make_inputs(name)
    layer = P.MoELayer(cfg.num_experts, cfg.hidden, cfg.inter, cfg.tokens, cfg.top_k)
    P.upload_layer(layer, inp.weights, DEV)
    blob = layer.nvfp4_moe_debug_packed_blob()
    gscale = torch.from_numpy(inp.weights.gscale).to(DEV)
    for sl in token_slices:          # consecutive calls share the static scratch
        logits = torch.from_numpy(np.ascontiguousarray(inp.logits[sl])).to(DEV)
        x = torch.from_numpy(np.ascontiguousarray(inp.x_bits[sl]).view(np.int16)).to(DEV).view(torch.bfloat16)
        ref = torch.empty_like(x)
        got = torch.full_like(x, float("nan"))
        layer.nvfp4_moe_set_path(P.PATH_DECODE)
        layer.nvfp4_moe_forward(logits, x, cfg.top_k, ref)
        st = P.binding.nvfp4_moe_forward_decode_static(blob, gscale, cfg.num_experts, cfg.hidden, cfg.inter,
                                                       logits, cfg.top_k, x, got)
        assert st == 0, P.STATUS[st]
        torch.cuda.synchronize()
        got64 = got.float().cpu().numpy().astype(np.float64)
        _close(got64, ref.float().cpu().numpy().astype(np.float64))
        # and against the oracle itself (the whole-piece schedule for T > 8 is this path's own)
        _assert_layer_bounds(got64, O.moe_forward(inp.logits[sl], inp.x_bits[sl], inp.weights, cfg.top_k))
    st, nan = P.binding.nvfp4_moe_static_get_status()
    assert st == 0 and nan == 0, (P.STATUS[st], nan)
    layer.close()


def test_static_forward_matches_handle_forward_tiny():
    _run_both("tiny", [slice(0, 16), slice(3, 5)])


def test_static_forward_matches_handle_forward_mtp():
    _run_both("decode_mtp", [slice(0, 2), slice(1, 2)])


def test_static_forward_matches_handle_forward_c16():
    _run_both("decode_c16", [slice(0, 16), slice(4, 12)])


def test_static_forward_rejects_what_does_not_fit():
    # 16 tokens x top-16 x (2*16384 + 4*16384) bytes of intermediates > 16 MiB
    P.build()
    x = torch.zeros((16, 16384), dtype=torch.bfloat16, device=DEV)
    logits = torch.zeros((16, 256), dtype=torch.float32, device=DEV)
    blob = torch.zeros((16,), dtype=torch.uint8, device=DEV)
    gs = torch.ones((256, 3), dtype=torch.float32, device=DEV)
    st = P.binding.nvfp4_moe_forward_decode_static(blob, gs, 256, 16384, 16384, logits, 16, x, torch.empty_like(x))
    assert st == P.STATUS_CODE["NVFP4_MOE_ERR_UNSUPPORTED_SHAPE"]


def test_static_status_reports_nan_logits_and_timeouts():
    P.build()
    cfg = CONFIGS["tiny"]
    inp = make_inputs("tiny")
    layer = P.MoELayer(cfg.num_experts, cfg.hidden, cfg.inter, cfg.tokens, cfg.top_k)
    P.upload_layer(layer, inp.weights, DEV)
    blob = layer.nvfp4_moe_debug_packed_blob()
    gscale = torch.from_numpy(inp.weights.gscale).to(DEV)
    x = torch.from_numpy(inp.x_bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    out = torch.empty_like(x)
    P.binding.nvfp4_moe_static_get_status()          # start from a clean word
    # two NaN logits in one call, one in the next: the word accumulates until read
    bad = inp.logits.copy()
    bad[0, 1] = np.nan
    bad[5, 7] = np.nan
    _static(blob, gscale, cfg, torch.from_numpy(bad).to(DEV), x, out)
    _static(blob, gscale, cfg, torch.from_numpy(bad[4:6].copy()).to(DEV), x[4:6], out[4:6])
    st, nan = P.binding.nvfp4_moe_static_get_status()
    assert st == 0 and nan == 3, (P.STATUS[st], nan)
    assert P.binding.nvfp4_moe_static_get_status() == (0, 0)   # read clears it
    # a bounded wait that gives up: no copies are issued, the waits expire
    assert P.binding.nvfp4_moe_static_debug_set_fault(1) == 0
    try:
        _static(blob, gscale, cfg, torch.from_numpy(inp.logits).to(DEV), x, out)
        st, _ = P.binding.nvfp4_moe_static_get_status()
        assert st == P.STATUS_CODE["NVFP4_MOE_ERR_TIMEOUT"], P.STATUS[st]
    finally:
        P.binding.nvfp4_moe_static_debug_set_fault(0)
    # the context is still usable and the next call is right
    good = torch.full_like(x, float("nan"))
    _static(blob, gscale, cfg, torch.from_numpy(inp.logits).to(DEV), x, good)
    assert P.binding.nvfp4_moe_static_get_status() == (0, 0)
    _assert_layer_bounds(good.float().cpu().numpy().astype(np.float64),
                O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k))
    layer.close()
