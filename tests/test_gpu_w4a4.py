"""The W4A4 comparison variant on the GPU, element by element against the oracle.

The stock checkpoint's routed experts are W4A4 NVFP4: x and h are quantised
to NVFP4 against per-module input scales ("tenhkspark/GLM-5.3-Flash-NVFP4-
Wabi", opening summary).  nvfp4_moe_set_act_quant turns it on.

The oracle quantises by the plain definition (both quotients in float64,
which decides as exact arithmetic does).  The kernels evaluate the same
quotients in FP32 as amax * fl(1 / fl(6 is)) and v * fl(1 / fl(scale * is)):
three roundings, so each quotient is within D = 4 * 2^-24 of its exact value,
relative.  A kernel's decision may therefore differ from the oracle's only
where the exact quotient lies within that distance of a rounding midpoint
(E2M1 or E4M3), and there either neighbour is valid.  The checks are interval
checks built on that, element by element, per routed row:

* x: the set of values the kernel may produce for each element of x^ (the
  oracle's, or the neighbour where the decision is that close);
* g, u: the oracle's dot products over that set, widened by the FP32
  summation bound 4 (K + 2) 2^-24 sum|x^ w| of the tensor-core accumulation
  and the FP32 products with the tensor scales;
* h: silu(g) u over those intervals, widened by 8 FP32 roundings (expf, the
  division, the product), then rounded to BF16 (monotone): decode stores this
  BF16 h, and every element must lie in its interval;
* h^ (prefill stores the quantised h): every block must be the quantisation,
  with some admissible scale, of values inside the BF16 h intervals;
* y: the down projection of the admissible h^ (from the GPU's own h), within
  the FP32 summation bound.
The layer output is checked element-wise at the W4A16 bounds (max|err| <=
2e-2 RMS plus the BF16 output rounding, mean relative error <= 5e-3) on the
error beyond a flip allowance: per element, the spread of every layer value
the admissible decisions can reach (the intervals above carried through the
combine).  The allowance is not small: with these input scales about 0.25% of
the x elements sit within D of a midpoint, and one flip moves a whole token's
expert output.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from synth import CONFIGS, make_inputs, make_input_scales
import nvfp4_weight_only_w4a16_gb300 as P
from tests.test_gpu_parity import DEV, _dev, _layer, _forward, assert_layer_close

pytestmark = pytest.mark.gpu

from tests.intervals import (D, U24, quant_box, assert_valid_quantisation, _mats, _dot_box,
                             hidden_bounds, w4a4_layer_allowance, assert_w4a4_layer)


def _check_rows(L, inp, iscale, path, rows_to_check):
    cfg = inp.config
    T, k = cfg.tokens, cfg.top_k
    hid, y = L.nvfp4_moe_debug_intermediates(T * k)
    rows = np.asarray(list(rows_to_check), dtype=np.int64)
    sel = torch.from_numpy(rows).to(hid.device)
    hid = hid[sel].float().cpu().numpy().astype(np.float64)
    y = y[sel].cpu().numpy().astype(np.float64)
    r = O.route(inp.logits, k)
    _, _, perm = O.permute(r.ids, cfg.num_experts)
    x = O.bf16_bits_to_f64(inp.x_bits)
    I = cfg.inter
    cache = {}
    for n, p in enumerate(rows):
        t, j = divmod(int(perm[p]), k)
        e = int(r.ids[t, j])
        if e not in cache:
            cache.clear()   # rows come in position order: one expert's rows are adjacent
            cache[e] = _mats(inp.weights, e)
        is1 = float(np.float32(iscale[e, 1]))
        hl, hh = hidden_bounds(cache[e], e, x[t], iscale)
        if path == P.PATH_PREFILL:   # the stored h is already quantised (code * scale)
            assert_valid_quantisation(hid[n], hl, hh, is1)
            vmin = vmax = hid[n]
        else:                        # decode stores BF16 h and quantises it inside the down GEMV
            bad = np.nonzero((hid[n] < hl) | (hid[n] > hh))[0]
            assert bad.size == 0, (p, bad[:8], hid[n][bad[:8]], hl[bad[:8]], hh[bad[:8]])
            vmin, vmax = quant_box(hid[n], hid[n], is1)
        _, _, wd, gs = cache[e]
        yl, yh = _dot_box(wd, vmin, vmax, gs[2] * is1, I)
        bad = np.nonzero((y[n] < yl) | (y[n] > yh))[0]
        assert bad.size == 0, (p, bad[:8], y[n][bad[:8]], yl[bad[:8]], yh[bad[:8]])


def check_w4a4_layer(gpu, inp, iscale, tokens=None, logits=None, scoring=None):
    """The layer against the oracle, element-wise, beyond the flip allowance
    (every output value the kernels' admissible quantiser decisions can reach)."""
    cfg = inp.config
    tok = np.arange(cfg.tokens) if tokens is None else np.asarray(tokens)
    lg = inp.logits if logits is None else logits
    ref = O.moe_forward_w4a4(lg, inp.x_bits, inp.weights, cfg.top_k, iscale, tokens=tok, num_shared=cfg.shared,
                             scoring=scoring)
    r = O.route(lg[tok], cfg.top_k) if scoring is None else O.route_scored(lg[tok], cfg.top_k, **scoring)
    ids, wts = r.ids, r.weights
    if cfg.shared:
        ids = np.concatenate([ids, np.full((len(tok), 1), cfg.num_experts, np.int32)], axis=1)
        wts = np.concatenate([wts, np.ones((len(tok), 1))], axis=1)
    A = w4a4_layer_allowance(inp.weights, inp.x_bits, ids, wts, iscale, cfg.num_experts, tok)
    assert_w4a4_layer(gpu, ref, A)
    return ref


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
    check_w4a4_layer(gpu, inp, iscale)
    # W4A4 is not W4A16: the two differ by the activation quantisation
    a16 = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k)
    assert np.linalg.norm(gpu - a16) / np.linalg.norm(a16) > 1e-2
    # and switching it off gives the W4A16 layer back
    back = _forward(L, inp.logits, inp.x_bits, cfg.top_k, path)
    assert_layer_close(back, a16)


@pytest.mark.parametrize("name,path", [("decode_mtp", P.PATH_DECODE), ("decode_c16", P.PATH_DECODE),
                                       ("prefill_1k", P.PATH_PREFILL), ("prefill_16k", P.PATH_PREFILL)])
def test_w4a4_full_size(name, path):
    inp = make_inputs(name)
    cfg = inp.config
    L = _layer(cfg)
    iscale = make_input_scales(cfg)
    L.nvfp4_moe_set_act_quant(_dev(iscale))
    try:
        gpu = _forward(L, inp.logits, inp.x_bits, cfg.top_k, path)
        R = cfg.tokens * cfg.top_k
        rows = range(R) if R <= 128 else np.sort(np.random.default_rng(3).choice(R, 24, replace=False))
        _check_rows(L, inp, iscale, path, rows)
    finally:
        L.nvfp4_moe_set_act_quant(None)
    if cfg.tokens <= 16:
        tok = list(range(cfg.tokens))
    else:
        tok = sorted({0, 1, 2, cfg.tokens // 2 - 1, cfg.tokens - 1})
    check_w4a4_layer(gpu[tok], inp, iscale, tokens=tok)


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
            check_w4a4_layer(gpu, inp, iscale)
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
