"""The W4A4 comparison variant on the GPU, against the oracle.

The stock checkpoint's routed experts are W4A4 NVFP4: x and h are quantised
to NVFP4 against per-module input scales ("tenhkspark/GLM-5.3-Flash-NVFP4-
Wabi", opening summary).  nvfp4_moe_set_act_quant turns it on.

Bars, from the arithmetic.  Quantising x is decided in FP32 on identical
BF16 inputs on both sides, so the quantised x is identical.  h is rounded to
BF16 before it is quantised; the GPU's FP32 h and the oracle's float64 h
round to different BF16 values only within an FP32 error of a BF16 tie
point, so the quantised h agrees except for rare single-step flips:
  * per routed row, the GPU's quantised h (prefill) matches the oracle's on
    all but <= 0.1% of elements, each mismatch one E2M1 step of its block;
  * per routed row, y is within the FP32 summation bound of the oracle's
    down projection of the GPU's own (quantised) h;
  * the layer output: ||gpu - oracle|| <= (2^-8 + 1e-3) ||oracle|| (the BF16
    output rounding, at most 2^-8 of each value, plus 1e-3 for the rest:
    FP32 sums, the shared expert's BF16 h, rare flips), cosine >= 0.9999,
    norm ratio in [0.99, 1.01].
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from synth import CONFIGS, make_inputs, make_input_scales, f32_to_bf16_bits
import nvfp4_weight_only_w4a16_gb300 as P
from tests.test_gpu_parity import DEV, _dev, _layer, _forward

pytestmark = pytest.mark.gpu


def _mats(w, e):
    I = w.w13_q.shape[1] // 2
    return (O.dequant(w.w13_q[e, :I], w.w13_s[e, :I]), O.dequant(w.w13_q[e, I:], w.w13_s[e, I:]),
            O.dequant(w.w2_q[e], w.w2_s[e]), w.gscale[e].astype(np.float64))


def _row_ref(w, e, x_row, iscale):
    """Oracle pieces of one routed row: BF16 h (float64 values) and its quantisation."""
    wg, wu, wd, gs = _mats(w, e)
    is0, is1 = float(iscale[e, 0]), float(iscale[e, 1])
    xq, _ = O.quantize_act_nvfp4(x_row[None, :], is0)
    h = O.silu(gs[0] * is0 * (xq @ wg.T)) * (gs[1] * is0 * (xq @ wu.T))
    hb = O.bf16_bits_to_f64(f32_to_bf16_bits(h.astype(np.float32)))
    hq, _ = O.quantize_act_nvfp4(hb.astype(np.float32), is1)
    return hb[0], hq[0], wd, gs, is1


def _check_layer(gpu, ref):
    assert np.all(np.isfinite(gpu))
    rel = np.linalg.norm(gpu - ref) / np.linalg.norm(ref)
    assert rel <= 2.0 ** -8 + 1e-3, rel
    cos = float(np.sum(gpu * ref) / (np.linalg.norm(gpu) * np.linalg.norm(ref)))
    assert cos >= 0.9999, cos
    ratio = np.linalg.norm(gpu) / np.linalg.norm(ref)
    assert 0.99 <= ratio <= 1.01, ratio


def _check_rows(L, inp, iscale, path, rows_to_check):
    cfg = inp.config
    T, k = cfg.tokens, cfg.top_k
    hid, y = L.nvfp4_moe_debug_intermediates(T * k)
    hid = hid.float().cpu().numpy().astype(np.float64)
    y = y.cpu().numpy().astype(np.float64)
    r = O.route(inp.logits, k)
    _, _, perm = O.permute(r.ids, cfg.num_experts)
    x = O.bf16_bits_to_f64(inp.x_bits)
    mism = total = 0
    for p in rows_to_check:
        t, j = divmod(int(perm[p]), k)
        e = int(r.ids[t, j])
        hb, hq, wd, gs, is1 = _row_ref(inp.weights, e, x[t], iscale)
        if path == P.PATH_PREFILL:   # the stored h is already quantised
            hq_gpu = hid[p]
            d = hq_gpu != hq
            mism += int(d.sum())
            total += d.size
            # a mismatch is one E2M1 step of its block: at most a third of the block's largest value
            blk = np.abs(hq).reshape(-1, 16).max(axis=1).repeat(16)
            assert np.all(np.abs(hq_gpu - hq)[d] <= blk[d] / 3 + 1e-30)
        else:                        # decode stores BF16 h and quantises it in the down GEMV
            d = hid[p] != hb
            mism += int(d.sum())
            total += d.size
            assert np.all(np.abs(hid[p] - hb)[d] <= 2.0 ** -7 * np.abs(hb)[d] + 1e-30)
            hq_gpu, _ = O.quantize_act_nvfp4(hid[p][None, :].astype(np.float32), is1)
            hq_gpu = hq_gpu[0]
        y_ref = gs[2] * is1 * (wd @ hq_gpu)
        absum = gs[2] * is1 * (np.abs(wd) @ np.abs(hq_gpu))
        I = wd.shape[1]
        assert np.all(np.abs(y[p] - y_ref) <= 4 * (I + 2) * 2.0 ** -24 * absum + 1e-30), p
    assert mism <= 1e-3 * total, (mism, total)


@pytest.mark.parametrize("path", [P.PATH_DECODE, P.PATH_PREFILL])
def test_w4a4_tiny(path):
    inp = make_inputs("tiny")
    cfg = inp.config
    L = _layer(cfg, max_tokens=512)
    iscale = make_input_scales(cfg)
    L.nvfp4_moe_set_act_quant(_dev(iscale))
    try:
        gpu = _forward(L, inp.logits, inp.x_bits, cfg.top_k, path)
        _check_rows(L, inp, iscale, path, range(cfg.tokens * cfg.top_k))
    finally:
        L.nvfp4_moe_set_act_quant(None)
    ref = O.moe_forward_w4a4(inp.logits, inp.x_bits, inp.weights, cfg.top_k, iscale)
    _check_layer(gpu, ref)
    # W4A4 is not W4A16: the two differ by the activation quantisation
    a16 = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k)
    assert np.linalg.norm(gpu - a16) / np.linalg.norm(a16) > 1e-2
    # and switching it off gives the W4A16 layer back
    back = _forward(L, inp.logits, inp.x_bits, cfg.top_k, path)
    assert np.linalg.norm(back - a16) / np.linalg.norm(a16) < 5e-3


@pytest.mark.parametrize("name,path", [("decode_mtp", P.PATH_DECODE), ("decode_c16", P.PATH_DECODE),
                                       ("prefill_1k", P.PATH_PREFILL)])
def test_w4a4_full_size(name, path):
    inp = make_inputs(name)
    cfg = inp.config
    L = _layer(cfg)
    iscale = make_input_scales(cfg)
    L.nvfp4_moe_set_act_quant(_dev(iscale))
    try:
        gpu = _forward(L, inp.logits, inp.x_bits, cfg.top_k, path)
        R = cfg.tokens * cfg.top_k
        rows = range(R) if R <= 128 else np.random.default_rng(3).choice(R, 24, replace=False)
        _check_rows(L, inp, iscale, path, rows)
    finally:
        L.nvfp4_moe_set_act_quant(None)
    tok = list(range(cfg.tokens)) if cfg.tokens <= 16 else [0, 1, 2, 511, 1023]
    ref = O.moe_forward_w4a4(inp.logits, inp.x_bits, inp.weights, cfg.top_k, iscale, tokens=tok)
    _check_layer(gpu[tok], ref)


def test_w4a4_shared_expert_stays_w4a16():
    inp = make_inputs("tiny_shared")
    cfg = inp.config
    import tests.test_gpu_shared as S
    L = S._shared_layer(cfg)
    iscale = make_input_scales(cfg)
    L.nvfp4_moe_set_act_quant(_dev(iscale))
    try:
        for path in (P.PATH_DECODE, P.PATH_PREFILL):
            gpu = _forward(L, inp.logits, inp.x_bits, cfg.top_k, path)
            ref = O.moe_forward_w4a4(inp.logits, inp.x_bits, inp.weights, cfg.top_k, iscale, num_shared=1)
            _check_layer(gpu, ref)
    finally:
        L.nvfp4_moe_set_act_quant(None)


def test_w4a4_rejects_bad_input_scales():
    cfg = CONFIGS["tiny"]
    L = _layer(cfg, max_tokens=512)
    for bad in (0.0, -1.0, np.nan, np.inf):
        s = make_input_scales(cfg)
        s[3, 1] = bad
        with pytest.raises(P.Nvfp4MoeError) as ei:
            L.nvfp4_moe_set_act_quant(_dev(s))
        assert ei.value.status == P.STATUS_CODE["NVFP4_MOE_ERR_BAD_SCALE"]
    L.nvfp4_moe_set_act_quant(None)
