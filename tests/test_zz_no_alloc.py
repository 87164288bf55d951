"""The allocation-free decode forward, checked against the handle-based one.

nvfp4_moe_forward_decode_static serves callers that cannot call cudaMalloc
(global-mode graph capture, plugins inside a framework that owns all device
memory, static-memory runtimes): it takes only caller memory and keeps its
intermediates in a static device array.  This file runs last so that, if it
fails, a run that stops at the first failure has already run everything else;
it needs no state from the other tests.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import nvfp4_weight_only_w4a16_gb300 as P
from synth import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _close(got, ref):
    # the layer tolerance of the parity tests, with the handle's output as reference
    err = np.abs(got - ref)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.all(err <= 2e-2 * rms + 2.0 ** -8 * np.abs(got)), (err.max(), rms)
    assert err.mean() / np.abs(ref).mean() <= 5e-3


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
        _close(got.float().cpu().numpy().astype(np.float64), ref.float().cpu().numpy().astype(np.float64))
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
