"""Every variant at once, and the smallest shapes, on the GPU against the oracle.

One handle with the single shared expert, the router linear computed in the
library, sigmoid scoring with a choice bias, renormalisation and a scale, and
the W4A4 comparison variant on the routed experts -- on both paths.  The
oracle runs on the GPU's own logits (routing is an argmax over them, decided
in the same precision on both sides).  Plus the dense linear at its smallest
output width (N = 16: one 128-row block, 112 rows of it padding).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from synth import CONFIGS, LinearConfig, make_inputs, make_input_scales, make_linear_inputs, make_router_weight
import nvfp4_weight_only_w4a16_gb300 as P
from tests.test_gpu_parity import DEV, _dev
from tests.test_gpu_w4a4 import check_w4a4_layer
from tests.test_gpu_linear import _abs_sum, _check, _run

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path", [P.PATH_DECODE, P.PATH_PREFILL])
def test_shared_router_sigmoid_bias_w4a4_together(path):
    inp = make_inputs("tiny_shared")
    cfg = inp.config
    P.build()
    L = P.MoELayer(cfg.num_experts, cfg.hidden, cfg.inter, 64, cfg.top_k, num_shared_experts=1)
    try:
        P.upload_layer(L, inp.weights, DEV)
        wr = make_router_weight(cfg)
        L.nvfp4_moe_set_router(_dev(wr.view(np.int16)).view(torch.bfloat16))
        bias = (np.random.default_rng(9).standard_normal(cfg.num_experts) * 0.2).astype(np.float32)
        L.nvfp4_moe_set_scoring("sigmoid", True, 1.5, _dev(bias))
        iscale = make_input_scales(cfg)
        L.nvfp4_moe_set_act_quant(_dev(iscale))
        L.nvfp4_moe_set_path(path)
        x = _dev(inp.x_bits.view(np.int16)).view(torch.bfloat16)
        out = torch.empty((cfg.tokens, cfg.hidden), dtype=torch.bfloat16, device=DEV)
        L.nvfp4_moe_forward_routed(x, cfg.top_k, out)
        torch.cuda.synchronize()
        assert L.nvfp4_moe_get_status()[0] == 0
        logits = L.nvfp4_moe_debug_logits(cfg.tokens).cpu().numpy()
        sc = dict(score="sigmoid", renormalize=True, scale=1.5, bias=bias)
        check_w4a4_layer(out.float().cpu().numpy().astype(np.float64), inp, iscale, logits=logits, scoring=sc)
    finally:
        L.close()


@pytest.mark.parametrize("path", [P.PATH_DECODE, P.PATH_PREFILL])
def test_linear_smallest_width(path):
    cfg = LinearConfig("linear_n16", 16, 128, 9)
    inp = make_linear_inputs(cfg)
    P.build()
    L = P.Linear(cfg.out_features, cfg.in_features, 64)
    try:
        L.nvfp4_linear_pack(_dev(inp.w_q), _dev(inp.w_s), _dev(np.array([inp.gscale], np.float32)))
        gpu = _run(L, inp.x_bits, path)
        ref = O.linear_forward(inp.x_bits, inp.w_q, inp.w_s, inp.gscale)
        _check(gpu, ref, _abs_sum(inp.x_bits, inp), cfg.in_features, True)
    finally:
        L.close()
