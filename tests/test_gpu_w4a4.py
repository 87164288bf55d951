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
2e-2 RMS plus the BF16 output rounding, mean relative error <= 5e-3), with
the norm ratio and cosine checks.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from synth import CONFIGS, make_inputs, make_input_scales
import nvfp4_weight_only_w4a16_gb300 as P
from tests.test_gpu_parity import DEV, _dev, _layer, _forward, assert_layer_close

pytestmark = pytest.mark.gpu

D = 4 * 2.0 ** -24          # relative error of the kernels' FP32 quantiser quotients
U24 = 2.0 ** -24            # FP32 unit roundoff


def _q_e2m1(v):
    """Signed E2M1 quantisation of float64 values (monotone non-decreasing)."""
    return O.decode_e2m1(O.encode_e2m1(v))


def _widen(v, rel):
    return v - rel * np.abs(v), v + rel * np.abs(v)


def _bf16(v):
    """float64 -> nearest BF16 value (via FP32, as the kernels hold h), float64."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint32) << 16
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def _scale_candidates(lo, hi, is_):
    """E4M3 scale values the kernel may pick for blocks whose inputs lie in
    [lo, hi] element-wise ([nb][16] each): the RNE of every amax in range,
    widened by D.  Returns a list (per block) of float64 scale values."""
    mlo = np.where((lo <= 0) & (hi >= 0), 0.0, np.minimum(np.abs(lo), np.abs(hi))).max(axis=-1)
    mhi = np.maximum(np.abs(lo), np.abs(hi)).max(axis=-1)
    c0 = O.encode_e4m3(mlo / (6.0 * is_) * (1 - D)).astype(np.int64)
    c1 = O.encode_e4m3(mhi / (6.0 * is_) * (1 + D)).astype(np.int64)
    return [O.decode_e4m3(np.arange(a, b + 1)) for a, b in zip(c0, c1)]


def _code_range(lo, hi, sv, is_):
    """Admissible code*scale values (min, max) per element for scale sv."""
    if sv == 0:
        z = np.zeros_like(lo)
        return z, z
    a, _ = _widen(lo / (sv * is_), D)
    _, b = _widen(hi / (sv * is_), D)
    return _q_e2m1(a) * sv, _q_e2m1(b) * sv


def quant_box(lo, hi, is_):
    """Element-wise bounds [vmin, vmax] (code * scale, without is) of every
    quantisation the kernel may produce for inputs in [lo, hi] ([..][K])."""
    shp = lo.shape
    lo = lo.reshape(-1, 16)
    hi = hi.reshape(-1, 16)
    vmin = np.empty_like(lo)
    vmax = np.empty_like(lo)
    for i, cands in enumerate(_scale_candidates(lo, hi, is_)):
        mins, maxs = zip(*(_code_range(lo[i], hi[i], sv, is_) for sv in cands))
        vmin[i] = np.min(mins, axis=0)
        vmax[i] = np.max(maxs, axis=0)
    return vmin.reshape(shp), vmax.reshape(shp)


def assert_valid_quantisation(V, lo, hi, is_):
    """Every 16-block of V (code * scale, float64) is the quantisation, with
    one admissible scale, of inputs inside [lo, hi]."""
    V = V.reshape(-1, 16)
    lo = lo.reshape(-1, 16)
    hi = hi.reshape(-1, 16)
    grid = O.decode_e2m1(np.arange(16))
    for i, cands in enumerate(_scale_candidates(lo, hi, is_)):
        ok = False
        for sv in cands:
            cmin, cmax = _code_range(lo[i], hi[i], sv, is_)
            on_grid = np.all(np.isin(V[i] / sv, grid)) if sv > 0 else np.all(V[i] == 0)
            if on_grid and np.all(V[i] >= cmin) and np.all(V[i] <= cmax):
                ok = True
                break
        assert ok, (i, V[i], lo[i], hi[i], cands)


def _silu_range(gl, gh):
    zs = -1.2784645427610738   # the minimum of silu
    a, b = O.silu(gl), O.silu(gh)
    lo = np.where((gl <= zs) & (zs <= gh), O.silu(np.float64(zs)), np.minimum(a, b))
    return lo, np.maximum(a, b)


def _mul_range(a1, a2, b1, b2):
    p = np.stack([a1 * b1, a1 * b2, a2 * b1, a2 * b2])
    return p.min(axis=0), p.max(axis=0)


def _mats(w, e):
    I = w.w13_q.shape[1] // 2
    return (O.dequant(w.w13_q[e, :I], w.w13_s[e, :I]), O.dequant(w.w13_q[e, I:], w.w13_s[e, I:]),
            O.dequant(w.w2_q[e], w.w2_s[e]), w.gscale[e].astype(np.float64))


def _dot_box(W, vmin, vmax, scale, K):
    """scale * W v over v in [vmin, vmax], widened by the FP32 accumulation and
    the FP32 products with the tensor scale."""
    mid, rad = (vmin + vmax) / 2, (vmax - vmin) / 2
    absw = np.abs(W)
    c = scale * (W @ mid)
    r = scale * (absw @ rad) + scale * 4 * (K + 2) * U24 * (absw @ np.maximum(np.abs(vmin), np.abs(vmax)))
    r = r + 3 * U24 * np.abs(c)
    return c - r, c + r


def hidden_bounds(mats, e, x_row, iscale):
    """BF16 h interval [lo, hi] of one routed row (expert e with its
    dequantised matrices, token row x)."""
    wg, wu, _, gs = mats
    is0 = float(np.float32(iscale[e, 0]))
    H = x_row.shape[-1]
    xmin, xmax = quant_box(x_row, x_row, is0)
    gl, gh = _dot_box(wg, xmin, xmax, gs[0] * is0, H)
    ul, uh = _dot_box(wu, xmin, xmax, gs[1] * is0, H)
    sl, sh = _silu_range(gl, gh)
    hl, hh = _mul_range(sl, sh, ul, uh)
    hl, _ = _widen(hl, 8 * U24)
    _, hh = _widen(hh, 8 * U24)
    return _bf16(hl), _bf16(hh)


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


def _check_layer(gpu, ref):
    assert np.all(np.isfinite(gpu))
    assert_layer_close(gpu, ref)


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
