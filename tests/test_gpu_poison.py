"""Reads of memory a forward has not written, and the device-side checks.

Every workspace buffer that a forward rewrites is filled with 0xFF (NaN in
FP16, BF16 and FP32) before a second forward; its output must be
bit-identical to the first.  A kernel that read a stale or unwritten value --
the failure mode of the serving postmortem, where an uninitialised scale
zeroed every expert ("GLM-5.3-Flash on Blackwell", The model loaded, served
an API, and produced garbage) -- would change it.  Then the same forwards on
a handle created with NVFP4_MOE_CHECKS=1 (index checks in the kernels) must
report nothing and give the same bits.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import nvfp4_weight_only_w4a16_gb300 as P
from synth import CONFIGS, make_inputs, make_layer_weights, make_input_scales
from tests.test_gpu_parity import DEV, _dev

pytestmark = pytest.mark.gpu

CASES = [("tiny", P.PATH_DECODE, False), ("tiny", P.PATH_PREFILL, False), ("decode_mtp", P.PATH_DECODE, False),
         ("decode_c16", P.PATH_DECODE, False), ("tiny", P.PATH_DECODE, True), ("tiny", P.PATH_PREFILL, True)]


def _run(L, inp, path):
    cfg = inp.config
    L.nvfp4_moe_set_path(path)
    x = _dev(inp.x_bits.view(np.int16)).view(torch.bfloat16)
    out = torch.empty((cfg.tokens, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    L.nvfp4_moe_forward(_dev(inp.logits), x, cfg.top_k, out)
    torch.cuda.synchronize()
    st, _ = L.nvfp4_moe_get_status()
    assert st == 0, P.STATUS[st]
    return out.view(torch.int16).cpu().numpy().copy()


def _layer(cfg, checks):
    P.build()
    old = os.environ.get("NVFP4_MOE_CHECKS")
    os.environ["NVFP4_MOE_CHECKS"] = "1" if checks else "0"
    try:
        L = P.MoELayer(cfg.num_experts, cfg.hidden, cfg.inter, max(cfg.tokens, 16), cfg.top_k)
    finally:
        if old is None:
            os.environ.pop("NVFP4_MOE_CHECKS")
        else:
            os.environ["NVFP4_MOE_CHECKS"] = old
    P.upload_layer(L, make_layer_weights(cfg), DEV)
    return L


@pytest.mark.parametrize("name,path,w4a4", CASES)
def test_poisoned_workspace_changes_nothing(name, path, w4a4):
    inp = make_inputs(name)
    cfg = inp.config
    L = _layer(cfg, checks=False)
    try:
        if w4a4:
            L.nvfp4_moe_set_act_quant(_dev(make_input_scales(cfg)))
        first = _run(L, inp, path)
        L.nvfp4_moe_debug_poison_workspace(0xFF)
        second = _run(L, inp, path)
        assert np.array_equal(first, second)
        # and with the device checks on: silent, same bits
        C = _layer(cfg, checks=True)
        try:
            if w4a4:
                C.nvfp4_moe_set_act_quant(_dev(make_input_scales(cfg)))
            C.nvfp4_moe_debug_poison_workspace(0xFF)
            assert np.array_equal(_run(C, inp, path), first)
        finally:
            C.close()
    finally:
        L.close()
