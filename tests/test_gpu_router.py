"""The router linear inside the library (nvfp4_moe_forward_routed), on the
GPU, against the oracle.

The routers stay BF16 linears ("GLM-5.3-Flash on Blackwell", The
quantization); here logits = x W_r^T is computed on the GPU (a GEMV kernel for
T <= 16, the tcgen05 GEMM above) and fed to the layer.

Bars.  Logits: every BF16 product is exact in FP32, so the only error is the
FP32 summation over H terms: |gpu - float64| <= 4 (H + 1) 2^-24 sum_h |x w|
(the 4x margin covers the tensor core's accumulation order).  Routing is an
argmax over those logits, so it is checked on the GPU's own logits (the same
precision on both sides): ids, offsets and perm bit-exact against the
oracle's route of the GPU logits.  The layer output meets the MoE bars
against the oracle run on the GPU logits.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from synth import CONFIGS, LayerConfig, make_inputs, make_router_weight
import nvfp4_weight_only_w4a16_gb300 as P
from tests.test_gpu_parity import DEV, _dev, _layer, assert_layer_close

pytestmark = pytest.mark.gpu


def _routed(L, cfg, inp, T, path, out_f32=False):
    wr = make_router_weight(cfg)
    L.nvfp4_moe_set_router(_dev(wr.view(np.int16)).view(torch.bfloat16))
    L.nvfp4_moe_set_path(path)
    x = _dev(inp.x_bits[:T].view(np.int16)).view(torch.bfloat16)
    out = torch.empty((T, cfg.hidden), dtype=torch.float32 if out_f32 else torch.bfloat16, device=DEV)
    L.nvfp4_moe_forward_routed(x, cfg.top_k, out)
    torch.cuda.synchronize()
    st, _ = L.nvfp4_moe_get_status()
    assert st == 0, P.STATUS[st]
    logits = L.nvfp4_moe_debug_logits(T).cpu().numpy()
    L.nvfp4_moe_set_path(P.PATH_AUTO)
    return wr, logits, out.float().cpu().numpy().astype(np.float64)


def _check_logits(logits, x_bits, wr, rows=None):
    xb = x_bits if rows is None else x_bits[rows]
    lg = logits if rows is None else logits[rows]
    ref = O.router_logits(xb, wr)
    H = xb.shape[1]
    absum = np.abs(O.bf16_bits_to_f64(xb)) @ np.abs(O.bf16_bits_to_f64(wr)).T
    err = np.abs(lg - ref)
    assert np.all(err <= 4 * (H + 1) * 2.0 ** -24 * absum + 1e-30), (err.max(), (err / absum).max())


@pytest.mark.parametrize("T,path", [(1, P.PATH_DECODE), (16, P.PATH_DECODE), (16, P.PATH_PREFILL),
                                    (37, P.PATH_PREFILL), (300, P.PATH_PREFILL)])
def test_router_tiny(T, path):
    cfg = CONFIGS["tiny"].with_tokens(T)
    inp = make_inputs(cfg)
    L = _layer(CONFIGS["tiny"], max_tokens=512)
    wr, logits, out = _routed(L, cfg, inp, T, path)
    _check_logits(logits, inp.x_bits, wr)
    # the tables of the forward, re-derived from the GPU logits
    ids, w, off, perm = L.nvfp4_moe_debug_route(_dev(logits), T, cfg.top_k)
    r = O.route(logits, cfg.top_k)
    assert np.array_equal(ids.cpu().numpy(), r.ids)
    ref = O.moe_forward(logits, inp.x_bits, inp.weights, cfg.top_k)
    assert_layer_close(out, ref)


def test_router_decode_mtp_and_c16():
    for name in ("decode_mtp", "decode_c16"):
        inp = make_inputs(name)
        cfg = inp.config
        L = _layer(cfg, max_tokens=1024)
        wr, logits, out = _routed(L, cfg, inp, cfg.tokens, P.PATH_AUTO)
        _check_logits(logits, inp.x_bits, wr)
        tok = [0, cfg.tokens - 1]
        ref = O.moe_forward(logits, inp.x_bits, inp.weights, cfg.top_k, tokens=tok)
        assert_layer_close(out[tok], ref)


def test_router_prefill_1k_gemm():
    inp = make_inputs("prefill_1k")
    cfg = inp.config
    L = _layer(cfg)
    wr, logits, out = _routed(L, cfg, inp, cfg.tokens, P.PATH_AUTO)
    rows = np.arange(0, cfg.tokens, 7)
    _check_logits(logits, inp.x_bits, wr, rows)
    ids, _, off, perm = L.nvfp4_moe_debug_route(_dev(logits), cfg.tokens, cfg.top_k)
    r = O.route(logits, cfg.top_k)
    assert np.array_equal(ids.cpu().numpy(), r.ids)
    _, off_ref, perm_ref = O.permute(r.ids, cfg.num_experts)
    assert np.array_equal(off.cpu().numpy(), off_ref) and np.array_equal(perm.cpu().numpy(), perm_ref)
    tok = [0, 1, 511, 1023]
    assert_layer_close(out[tok], O.moe_forward(logits, inp.x_bits, inp.weights, cfg.top_k, tokens=tok))


def test_router_with_sigmoid_bias_scoring():
    inp = make_inputs("decode_mtp")
    cfg = inp.config
    L = _layer(cfg, max_tokens=1024)
    b = (np.random.default_rng(5).standard_normal(cfg.num_experts) * 0.3).astype(np.float32)
    L.nvfp4_moe_set_scoring("sigmoid", True, 2.5, _dev(b))
    try:
        wr, logits, out = _routed(L, cfg, inp, cfg.tokens, P.PATH_AUTO)
    finally:
        L.nvfp4_moe_set_scoring()
    sc = dict(score="sigmoid", renormalize=True, scale=2.5, bias=b)
    ref = O.moe_forward(logits, inp.x_bits, inp.weights, cfg.top_k, scoring=sc)
    assert_layer_close(out, ref)


def test_router_16k_sampled_256_experts():
    inp = make_inputs("prefill_16k")
    cfg = inp.config
    L = _layer(cfg)
    wr, logits, out = _routed(L, cfg, inp, cfg.tokens, P.PATH_AUTO, out_f32=False)
    rows = np.arange(0, cfg.tokens, 509)
    _check_logits(logits, inp.x_bits, wr, rows)
    ids, _, _, _ = L.nvfp4_moe_debug_route(_dev(logits), cfg.tokens, cfg.top_k)
    assert np.array_equal(ids.cpu().numpy(), O.route(logits, cfg.top_k).ids)


def test_router_errors():
    cfg = CONFIGS["tiny"]
    L = P.MoELayer(cfg.num_experts, cfg.hidden, cfg.inter, 64, cfg.top_k)
    from synth import make_layer_weights
    P.upload_layer(L, make_layer_weights(cfg), DEV)
    x = torch.zeros((4, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(x)
    with pytest.raises(P.Nvfp4MoeError) as ei:
        L.nvfp4_moe_forward_routed(x, cfg.top_k, out)
    assert ei.value.status == P.STATUS_CODE["NVFP4_MOE_ERR_INVALID_ARG"]
    with pytest.raises(P.Nvfp4MoeError) as ei:
        L.nvfp4_moe_debug_logits(4)
    assert ei.value.status == P.STATUS_CODE["NVFP4_MOE_ERR_INVALID_ARG"]
    L.close()
