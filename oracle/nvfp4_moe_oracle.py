"""Float64 CPU oracle of the routed-expert MoE layer with weight-only NVFP4 experts.

TEST INFRASTRUCTURE ONLY.  The product (the CUDA library and its Python
binding) never imports, calls or links this file; only tests, the smoke check
and the benchmark's CPU-baseline leg do.

What the layer computes, as the GLM-5.3-Flash pages describe it:

* The routed experts are stored weight-only NVFP4: 4-bit values with one scale
  per group of 16 and one per-tensor global scale ("tenhkspark/GLM-5.3-Flash-
  NVFP4-Wabi", Config expectations: group_size = 16, weight_scale_2; "GLM-5.3-
  Flash on Blackwell", The quantization: the routed-expert tensors go to 4-bit).
* Activations stay BF16 and there is no activation scale: the weight-only path
  dequantises to BF16 and never consumes an input scale ("GLM-5.3-Flash on
  Blackwell", The model loaded, served an API, and produced garbage).
* Routers are BF16 linears whose logits are an input here (same page, The
  quantization: the routers stay BF16).

Value formats (public definitions, decoded from bit fields here):
* E2M1 (OCP Microscaling Formats v1.0, FP4): sign bit 3, exponent bits 2..1
  (bias 1), mantissa bit 0; exponent 0 is subnormal m*0.5.  Values
  {0, 0.5, 1, 1.5, 2, 3, 4, 6} x sign.
* E4M3 (OCP 8-bit Floating Point Specification): sign bit 7, exponent bits 6..3
  (bias 7), mantissa bits 2..0; exponent 0 is subnormal (m/8)*2**-6;
  S.1111.111 is NaN; there is no infinity; the largest value is 448.

Readings where the pages are silent (each is listed with its reason in the
design notes):
* nibble order: element 2j is the low nibble of byte j;
* scale groups run along K (the reduction axis) of each output row;
* three FP32 tensor scales per expert (gate, up, down), applied after the dot
  product;
* top-k: larger logit first, equal logits -> lower expert index first, NaN
  ranks below -inf;
* routing weights: softmax over the k selected logits, no extra factor (the
  sigmoid / bias-corrected / unnormalised / scaled variants: route_scored);
* permutation: expert-major, ascending flattened index t*k+j inside an expert;
* SwiGLU: h = silu(gate) * up with silu(z) = z / (1 + exp(-z));
* combine: out[t] = sum_j w[t][j] * y[t, j], summed in slot order j = 0..k-1.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "decode_e2m1", "decode_e4m3", "unpack_e2m1_codes", "dequant", "dequant_scaled_f32",
    "bf16_bits_to_f64", "route", "route_scored", "router_logits", "permute", "silu", "expert_ffn", "expert_hidden",
    "moe_forward", "linear_forward", "RouteResult", "encode_e2m1", "encode_e4m3", "quantize_act_nvfp4",
    "moe_forward_w4a4",
]


# ----------------------------------------------------------------------------
# Formats
# ----------------------------------------------------------------------------

def decode_e2m1(codes) -> np.ndarray:
    """E2M1 code (0..15) -> float64, from the bit fields."""
    c = np.asarray(codes).astype(np.int64)
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e - 1.0))
    return np.where(s == 1, -mag, mag)


def decode_e4m3(b) -> np.ndarray:
    """OCP E4M3 byte -> float64 (NaN for S.1111.111), from the bit fields."""
    c = np.asarray(b).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def unpack_e2m1_codes(q) -> np.ndarray:
    """[N][K/2] bytes -> [N][K] codes; element 2j is the low nibble of byte j."""
    q = np.asarray(q, dtype=np.uint8)
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = q & 0xF
    out[..., 1::2] = q >> 4
    return out


def dequant(q, s) -> np.ndarray:
    """W[n][k] = e2m1(code[n][k]) * e4m3(s[n][k // 16]) in float64 (exact).

    The per-tensor FP32 scale is not included; the FFN applies it after the
    dot product.  The bit-field decoders are evaluated once on all 16 / 256
    codes and the results looked up (same values, fewer passes over the data).
    """
    codes = unpack_e2m1_codes(q)
    vals = decode_e2m1(np.arange(16))[codes]
    scales = decode_e4m3(np.arange(256))[np.asarray(s, dtype=np.uint8)]
    return vals * np.repeat(scales, 16, axis=-1)


def dequant_scaled_f32(q, s, g) -> np.ndarray:
    """Dequantised weight including the tensor scale, as one FP32 product.

    e2m1 * e4m3 has at most 5 significant bits and lies in [2**-10, 2688], so
    it is exact in float32; the single float32 multiply by g (round to
    nearest even) is the only rounding.  This is the quantity the library's
    dequantisation check returns.
    """
    w = dequant(q, s).astype(np.float32)
    return (w * np.float32(g)).astype(np.float32)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """BF16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Route and permute
# ----------------------------------------------------------------------------

class RouteResult:
    def __init__(self, ids, weights, nan_count):
        self.ids = ids              # int32 [T][k]
        self.weights = weights      # float64 [T][k]
        self.nan_count = nan_count  # number of NaN logits seen


def route(logits, k: int) -> RouteResult:
    """Top-k of each token's router logits, then softmax over the k chosen.

    Order: larger logit first; equal logits -> lower expert index first; NaN
    ranks below every number including -inf.  Weights: exp(l_j - max) /
    sum_i exp(l_i - max) over the selected logits, with NaN taken as -inf.  If
    every selected logit is -inf/NaN the weights are 1/k each (the limit of
    equal logits); if the largest is +inf, the +inf entries share weight 1.
    """
    L = np.asarray(logits, dtype=np.float64)
    T, E = L.shape
    if not 1 <= k <= E:
        raise ValueError("top_k must be in 1..E")
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    nan = np.isnan(L)
    idx = np.arange(E)
    for t in range(T):
        clean = np.where(nan[t], 0.0, L[t])
        order = np.lexsort((idx, -clean, nan[t].astype(np.int8)))
        sel = order[:k]
        ids[t] = sel
        ls = np.where(nan[t, sel], -np.inf, L[t, sel])
        m = ls.max()
        if m == -np.inf:
            w[t] = 1.0 / k
        elif m == np.inf:
            hit = (ls == np.inf).astype(np.float64)
            w[t] = hit / hit.sum()
        else:
            ex = np.exp(ls - m)
            w[t] = ex / ex.sum()
    return RouteResult(ids, w, int(nan.sum()))


def route_scored(logits, k: int, score: str = "softmax", renormalize: bool = True, scale: float = 1.0,
                 bias=None) -> RouteResult:
    """Top-k routing with a choice of scoring rule (the router variants).

    The pages keep the routers as BF16 linears and say nothing more about how
    their outputs become expert choices and weights ("GLM-5.3-Flash on
    Blackwell", The quantization: the routers stay BF16; "tenhkspark/GLM-5.3-
    Flash-NVFP4-Wabi", Config expectations: the per-layer mlp.gate routers are
    excluded from quantisation).  The variants, each a plain reading:

    * score = "softmax": s_e = exp(l_e - max) / sum over ALL experts; with
      renormalize the chosen k weights are divided by their own sum, which is
      the same as softmax over the k chosen logits (route());
    * score = "sigmoid": s_e = 1 / (1 + exp(-l_e)); with renormalize the
      chosen weights are s_j / sum of the chosen s (1/k each if that sum is 0);
    * bias [E] (optional): added to s_e for the CHOICE only ("bias-
      corrected" selection); the weights use s_e without it;
    * scale: every final weight is multiplied by it.
    The choice orders experts by s_e + bias_e: larger first, equal values ->
    lower expert index first, a NaN logit below everything (its s counts as 0
    in the weights).  Softmax edge cases follow route(): all -inf -> equal s,
    any +inf -> the +inf entries share s = 1.
    """
    L = np.asarray(logits, dtype=np.float64)
    T, E = L.shape
    if not 1 <= k <= E:
        raise ValueError("top_k must be in 1..E")
    if score not in ("softmax", "sigmoid"):
        raise ValueError("score must be softmax or sigmoid")
    b = np.zeros(E) if bias is None else np.asarray(bias, dtype=np.float64)
    nan = np.isnan(L)
    idx = np.arange(E)
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        l = np.where(nan[t], -np.inf, L[t])
        if score == "sigmoid":
            with np.errstate(over="ignore"):
                s = 1.0 / (1.0 + np.exp(-l))
        else:
            m = l.max()
            if m == -np.inf:
                s = np.full(E, 1.0 / E)
            elif m == np.inf:
                hit = (l == np.inf).astype(np.float64)
                s = hit / hit.sum()
            else:
                ex = np.exp(l - m)
                s = ex / ex.sum()
        choice = s + b
        order = np.lexsort((idx, -np.where(nan[t], 0.0, choice), nan[t].astype(np.int8)))
        sel = order[:k]
        ids[t] = sel
        ws = np.where(nan[t, sel], 0.0, s[sel])
        if renormalize:
            tot = ws.sum()
            ws = ws / tot if tot > 0 else np.full(k, 1.0 / k)
        w[t] = scale * ws
    return RouteResult(ids, w, int(nan.sum()))


def router_logits(x_bits, w_router_bits) -> np.ndarray:
    """The router linear: logits[t][e] = sum_h x[t][h] * W[e][h] in float64.

    x [T][H] and W [E][H] are BF16 bit patterns (the routers stay BF16:
    "GLM-5.3-Flash on Blackwell", The quantization); no linear bias.
    """
    x = bf16_bits_to_f64(np.asarray(x_bits))
    wr = bf16_bits_to_f64(np.asarray(w_router_bits))
    return x @ wr.T


def permute(ids, num_experts: int):
    """Expert-major stable order of the T*k routed rows.

    Returns (counts [E], offsets [E+1], perm [T*k]) where perm[p] is the
    flattened index t*k+j of the row at position p; inside one expert the
    flattened indices ascend.
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    counts = np.bincount(flat, minlength=num_experts).astype(np.int32)
    offsets = np.zeros(num_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    return counts, offsets, perm


# ----------------------------------------------------------------------------
# Expert FFN and the layer
# ----------------------------------------------------------------------------

def silu(z):
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def _expert_mats(w, e):
    I = w.w13_q.shape[1] // 2
    wg = dequant(w.w13_q[e, :I], w.w13_s[e, :I])
    wu = dequant(w.w13_q[e, I:], w.w13_s[e, I:])
    wd = dequant(w.w2_q[e], w.w2_s[e])
    gs = w.gscale[e].astype(np.float64)
    return wg, wu, wd, gs


def expert_hidden(w, e: int, x) -> np.ndarray:
    """h = silu(gs_g * Wg x) * (gs_u * Wu x) for the rows of x [m][H], float64."""
    wg, wu, _, gs = _expert_mats(w, e)
    x = np.asarray(x, dtype=np.float64)
    return silu(gs[0] * (x @ wg.T)) * (gs[1] * (x @ wu.T))


def expert_ffn(w, e: int, x) -> np.ndarray:
    """FFN_e(x) = gs_d * Wd (silu(gs_g * Wg x) * (gs_u * Wu x)) for x [m][H]."""
    wg, wu, wd, gs = _expert_mats(w, e)
    x = np.asarray(x, dtype=np.float64)
    h = silu(gs[0] * (x @ wg.T)) * (gs[1] * (x @ wu.T))
    return gs[2] * (h @ wd.T)


def moe_forward(logits, x_bits, weights, k: int, tokens=None, return_parts=False, num_shared: int = 0,
                scoring=None):
    """out[t] = sum_{j<k} w[t][j] * FFN_{ids[t][j]}(x[t]) (+ FFN_E(x[t])) in float64.

    logits [T][E] (float32 or float64), x_bits [T][H] BF16 bit patterns,
    weights an ExpertWeights-like object with w13_q/w13_s/w2_q/w2_s/gscale.
    num_shared = 1: weights also hold expert E (E = logits.shape[1]), the
    layer's single shared expert, which every token uses with weight 1 on top
    of its routed experts ("GLM-5.3-Flash on Blackwell", The model loaded,
    served an API, and produced garbage: the model keeps running "on
    attention and the single shared expert" when every routed expert is
    zeroed; "GLM-5.3-Flash-NVFP4-h — W4A16 dense-side quantization": the shared
    experts' gate/up/down are W4A16 NVFP4 with 16-element groups).  Its output
    is added after the routed sum.
    tokens: optional subset of token indices (the output has one row per
    listed token, in that order).  With return_parts, also returns the route
    result and the per-slot expert outputs y [len(tokens)][k + num_shared][H]
    (the shared expert's in the last slot).
    scoring: None for route(), else the keyword arguments of route_scored
    (score, renormalize, scale, bias).
    """
    if num_shared not in (0, 1):
        raise ValueError("num_shared must be 0 or 1")
    logits = np.asarray(logits)
    T, E = logits.shape
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    r = route(logits[tok], k) if scoring is None else route_scored(logits[tok], k, **scoring)
    x = bf16_bits_to_f64(np.asarray(x_bits)[tok])
    H = x.shape[1]
    y = np.zeros((len(tok), k + num_shared, H), dtype=np.float64)
    for e in np.unique(r.ids):
        rows, slots = np.nonzero(r.ids == e)
        y[rows, slots] = expert_ffn(weights, int(e), x[rows])
    out = np.zeros((len(tok), H), dtype=np.float64)
    for j in range(k):
        out += r.weights[:, j:j + 1] * y[:, j]
    if num_shared:
        y[:, k] = expert_ffn(weights, E, x)
        out += y[:, k]
    if return_parts:
        return out, r, y
    return out


# ----------------------------------------------------------------------------
# W4A4 comparison variant: activations quantised to NVFP4 with an input scale
# ----------------------------------------------------------------------------
# The stock checkpoint's routed experts are W4A4 NVFP4: activations are also
# quantised to 4 bits with 16-element E4M3 block scales against a per-module
# FP32 `input_scale` ("tenhkspark/GLM-5.3-Flash-NVFP4-Wabi", opening summary:
# the routed experts keep the stock W4A4 NVFP4 quantisation; "GLM-5.3-Flash on
# Blackwell", The model loaded, served an API, and produced garbage: a W4A4
# MoE path consumed an uninitialised input_scale of 0.0 and zeroed every
# expert; "tacos4me/GLM-5.3-Flash-NVFP4-FP8ATTN-512K", Input-scales provenance:
# a placeholder input_scale of 1.0 made small-amax blocks underflow to zero).
# The block rule is the weight rule applied to activations: per 16 consecutive
# K elements, scale = E4M3(amax / (6 * input_scale)) and code = E2M1(v /
# (scale * input_scale)), both round-to-nearest-even and saturating; value =
# code * scale * input_scale.  The pages fix no precision or order of
# operations for these quotients, so the oracle takes the plain definition:
# both quotients in float64.  For float32 operands that decides exactly as
# real arithmetic does (a quotient of two floats with at most 28 significant
# bits is either exactly on a rounding midpoint or at least 2**-33 of its
# value away from it, far above float64's 2**-53 rounding).  h is rounded to
# BF16 before it is quantised, as it is between the GEMMs of the W4A16 layer.

_E2M1_POS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _rne_to_grid(a, grid):
    """Round |values| a (float64, >= 0) to the nearest of the increasing grid
    (index = code), ties to the even code, saturating at the top."""
    a = np.minimum(a, grid[-1])
    hi = np.searchsorted(grid, a, side="left")          # first grid value >= a
    hi = np.minimum(hi, len(grid) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - grid[lo], grid[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo)


def encode_e2m1(v) -> np.ndarray:
    """float -> E2M1 code, round-to-nearest-even, saturating at +-6."""
    v = np.asarray(v, dtype=np.float64)
    code = _rne_to_grid(np.abs(v), _E2M1_POS)
    return (code | (np.signbit(v).astype(np.int64) << 3)).astype(np.uint8)


def encode_e4m3(v) -> np.ndarray:
    """float >= 0 -> E4M3 code, round-to-nearest-even, saturating at 448."""
    grid = decode_e4m3(np.arange(127))                  # codes 0..126: 0 .. 448
    return _rne_to_grid(np.asarray(v, dtype=np.float64), grid).astype(np.uint8)


def quantize_act_nvfp4(v, input_scale: float):
    """v [..][K] (K % 16 == 0) -> its W4A4 value without the input scale,
    code * scale (float64, exact), plus the E4M3 scale codes [..][K/16].

    Per block of 16: scale = E4M3_RNE(amax / (6 * is)), then code =
    E2M1_RNE(v / (scale * is)) (a zero scale gives zero codes); every
    quotient in float64 from the exact float64 values of v and is.
    """
    v = np.asarray(v).astype(np.float64)
    isf = float(np.float32(input_scale))
    blk = v.reshape(v.shape[:-1] + (v.shape[-1] // 16, 16))
    amax = np.max(np.abs(blk), axis=-1)
    sc = encode_e4m3(amax / (6.0 * isf))
    sv = decode_e4m3(sc)
    step = sv * isf
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(step[..., None] > 0, blk / step[..., None], 0.0)
    codes = encode_e2m1(q)
    vals = decode_e2m1(codes) * sv[..., None]
    return vals.reshape(v.shape), sc


def moe_forward_w4a4(logits, x_bits, weights, k: int, input_scale, tokens=None, num_shared: int = 0,
                     scoring=None):
    """The layer with W4A4 routed experts: for routed row (t, e),
    x^ = Q(x[t]; is[e][0]), g = gs_g is0 Wg x^, u = gs_u is0 Wu x^,
    h = silu(g) u, h^ = Q(bf16(h); is[e][1]), y = gs_d is1 Wd h^, and
    out[t] = sum_j w_j y_j (+ the shared expert, which stays W4A16).
    input_scale [E][2] float32 (w13, w2), each finite and > 0."""
    iscale = np.asarray(input_scale, dtype=np.float32)
    if not np.all(np.isfinite(iscale)) or np.any(iscale <= 0):
        raise ValueError("every input_scale must be finite and > 0")
    logits = np.asarray(logits)
    T, E = logits.shape
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    r = route(logits[tok], k) if scoring is None else route_scored(logits[tok], k, **scoring)
    x = bf16_bits_to_f64(np.asarray(x_bits)[tok])
    out = np.zeros_like(x)
    for e in np.unique(r.ids):
        rows, slots = np.nonzero(r.ids == e)
        wg, wu, wd, gs = _expert_mats(weights, int(e))
        is0, is1 = float(iscale[e, 0]), float(iscale[e, 1])
        xq, _ = quantize_act_nvfp4(x[rows], is0)
        h = silu(gs[0] * is0 * (xq @ wg.T)) * (gs[1] * is0 * (xq @ wu.T))
        hq, _ = quantize_act_nvfp4(bf16_bits_to_f64(_round_bf16_bits(h)).astype(np.float32), is1)
        y = gs[2] * is1 * (hq @ wd.T)
        out[rows] += r.weights[rows, slots][:, None] * y
    if num_shared:
        out += expert_ffn(weights, E, x)
    return out


def _round_bf16_bits(v) -> np.ndarray:
    """float64 -> BF16 bit patterns: rounded to float32 first, as the kernels
    hold h, then to BF16 with round-to-nearest-even."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def linear_forward(x_bits, w_q, w_s, gscale: float) -> np.ndarray:
    """A W4A16 NVFP4 dense linear: out[t] = gs * W x[t] in float64.

    W [N][K] in the canonical NVFP4 layout (codes [N][K/2], E4M3 scales
    [N][K/16]) with one FP32 tensor scale gs, x [T][K] BF16 bit patterns.  The
    same weight-only format the routed experts use also covers the dense
    projections ("GLM-5.3-Flash-NVFP4-h — W4A16 dense-side quantization": the
    attention linears, shared experts and lm_head quantised to W4A16 NVFP4
    with 16-element groups, activations left in BF16).
    """
    x = bf16_bits_to_f64(np.asarray(x_bits))
    return float(gscale) * (x @ dequant(w_q, w_s).T)
