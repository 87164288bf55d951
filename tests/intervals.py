"""Interval arithmetic for the element-wise GPU checks (test helpers).

A GPU result is accepted where it lies inside the interval of values that
the kernels' documented FP32 arithmetic can produce from the oracle's exact
values: tensor-core products of exact operands summed in FP32 (at most
4 (K + 2) 2^-24 sum|terms| away from the exact sum, whatever the order),
FP32 products with the tensor scales, silu and the SwiGLU product in FP32,
one rounding to BF16 (monotone), and -- for the W4A4 variant -- quantiser
quotients evaluated in FP32 within D = 4 * 2^-24 of the exact quotient.
Not collected by pytest (no test_ prefix).
"""
import numpy as np

import oracle as O

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
    """scale * W v over v in [vmin, vmax] (a row [K] or rows [m][K]), widened
    by the FP32 accumulation and the FP32 products with the tensor scale."""
    mid, rad = (vmin + vmax) / 2, (vmax - vmin) / 2
    c = scale * (mid @ W.T)
    # |W| (rad + 4 (K + 2) 2^-24 max(|vmin|, |vmax|)) in one product
    r = scale * ((rad + 4 * (K + 2) * U24 * np.maximum(np.abs(vmin), np.abs(vmax))) @ np.abs(W).T)
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




def prescale_slack(v):
    """Element-wise allowance for a row entering an FP16 MMA after a power-of-
    two prescale that puts its maximum in [2^13, 2^14): values more than 2^31
    below the maximum lose bits in FP16's subnormal range, by at most one
    subnormal step, max|v| * 2^-37 (generous) in the row's own units."""
    return np.max(np.abs(v), axis=-1, keepdims=True) * 2.0 ** -37


def hidden_bounds_w4a16(mats, x_row):
    """Interval [lo, hi] of the h values the down GEMM may consume for W4A16
    routed rows (x [K] or [m][K]): x enters exactly (BF16 operands, or FP16
    after a power-of-two prescale, within prescale_slack), g and u are FP32
    sums, and h is rounded once to 16 bits -- BF16 (8 significant bits, at most
    2^-9 of the value) or FP16 after a power-of-two prescale (11 bits, plus
    the subnormal slack of values far below the largest): 2^-8 of the value
    plus the slack covers either."""
    wg, wu, _, gs = mats
    H = x_row.shape[-1]
    eps = prescale_slack(x_row)
    gl, gh = _dot_box(wg, x_row - eps, x_row + eps, gs[0], H)
    ul, uh = _dot_box(wu, x_row - eps, x_row + eps, gs[1], H)
    sl, sh = _silu_range(gl, gh)
    hl, hh = _mul_range(sl, sh, ul, uh)
    hl, _ = _widen(hl, 8 * U24)
    _, hh = _widen(hh, 8 * U24)
    # the FP16 prescale 2^p of a row is at most its largest |h| (decode: per
    # chunk) or the row's Cauchy-Schwarz bound B = 2 gs_g gs_u max_f ||Wg_f||
    # ||Wu_f|| ||x||^2 (prefill) times 2^-13; FP16's subnormal spacing 2^-24
    # then stays below B 2^-37
    hb = np.max(np.linalg.norm(wg, axis=1) * np.linalg.norm(wu, axis=1))
    B = 2 * gs[0] * gs[1] * hb * np.sum(np.square(x_row), axis=-1, keepdims=True)
    slack = np.maximum(prescale_slack(np.maximum(np.abs(hl), np.abs(hh))), B * 2.0 ** -36)
    return hl - 2.0 ** -8 * np.abs(hl) - slack, hh + 2.0 ** -8 * np.abs(hh) + slack


def down_bounds_w4a16(mats, h_row):
    """Interval of y = gs_d Wd h for the h rows ([I] or [m][I]) the down GEMM
    consumed (the GPU's own, exactly)."""
    _, _, wd, gs = mats
    return _dot_box(wd, h_row, h_row, gs[2], wd.shape[1])


def assert_inside(v, lo, hi, what):
    bad = np.nonzero(((v < lo) | (v > hi)).reshape(-1))[0]
    v, lo, hi = v.reshape(-1), lo.reshape(-1), hi.reshape(-1)
    assert bad.size == 0, (what, bad.size, bad[:6], v[bad[:6]], lo[bad[:6]], hi[bad[:6]])


def w4a4_y_box(mats, x_rows, is0, is1):
    """[yl, yh] of y = gs_d is1 Wd h^ for W4A4 routed rows x_rows ([K] or
    [m][K]) of one expert: every value the kernels' arithmetic can produce --
    each quantiser decision within D of a midpoint either way, FP32 sums,
    BF16 h."""
    wg, wu, wd, gs = mats
    H = x_rows.shape[-1]
    xmin, xmax = quant_box(x_rows, x_rows, is0)
    gl, gh = _dot_box(wg, xmin, xmax, gs[0] * is0, H)
    ul, uh = _dot_box(wu, xmin, xmax, gs[1] * is0, H)
    sl, sh = _silu_range(gl, gh)
    hl, hh = _mul_range(sl, sh, ul, uh)
    hl, _ = _widen(hl, 8 * U24)
    _, hh = _widen(hh, 8 * U24)
    hmin, hmax = quant_box(_bf16(hl), _bf16(hh), is1)
    return _dot_box(wd, hmin, hmax, gs[2] * is1, wd.shape[1])


def w4a4_layer_allowance(weights, x_bits, ids, wts, iscale, num_routed, tokens):
    """Per output element, the spread of the W4A4 layer values the kernels may
    produce: sum over slots of |w| (yh - yl), yl/yh from w4a4_y_box (routed
    experts) or the W4A16 boxes (the shared expert, index num_routed).
    ids/wts [len(tokens)][slots] for the listed tokens."""
    x = O.bf16_bits_to_f64(np.asarray(x_bits)[tokens])
    A = np.zeros_like(x)
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        mats = _mats(weights, int(e))
        if e < num_routed:
            yl, yh = w4a4_y_box(mats, x[rows], float(np.float32(iscale[e, 0])), float(np.float32(iscale[e, 1])))
        else:
            hl, hh = hidden_bounds_w4a16(mats, x[rows])
            yl, yh = _dot_box(mats[2], hl, hh, mats[3][2], mats[2].shape[1])
        A[rows] += np.abs(wts[rows, slots])[:, None] * (yh - yl)
    return A


def assert_w4a4_layer(gpu, ref, allowance):
    """The layer bounds of the W4A16 checks (max|err| <= 2e-2 RMS plus the
    BF16 output rounding; mean relative error <= 5e-3), each on the error
    beyond the flip allowance."""
    assert np.all(np.isfinite(gpu))
    err = np.maximum(np.abs(gpu - ref) - allowance, 0.0)
    rms = np.sqrt(np.mean(ref ** 2))
    bad = err > 2e-2 * rms + 2.0 ** -8 * np.abs(gpu)
    assert not bad.any(), (int(bad.sum()), float(err.max()), rms)
    assert err.mean() / np.abs(ref).mean() <= 5e-3, err.mean() / np.abs(ref).mean()
