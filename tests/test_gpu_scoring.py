"""The route step's scoring variants, on the GPU, against the oracle.

Variants (nvfp4_moe_set_scoring; the oracle's route_scored): softmax over all
experts or sigmoid scores, an optional per-expert bias added for the choice
only, optional renormalisation of the chosen weights, a scaling factor.  The
pages keep the routers as BF16 linears and say no more ("GLM-5.3-Flash on
Blackwell", The quantization), so each variant is a plain reading.

Bars.  Without a bias the choice is made on the logits on both sides (both
scores are strictly increasing), so ids, offsets and perm are bit-exact.
With a bias the GPU compares FP32 scores and the oracle float64 ones: ids
must agree wherever the float64 gap around the k-th choice exceeds 1e-5 (an
FP32 score is within a few ulp, < 1e-6, of the float64 one), and elsewhere the
GPU's set must still be a valid top-k within that tolerance.  Weights: within
1e-6 relative + 1e-7 absolute of the float64 ones (FP32 expf and sums of <= 16
terms).  The layer meets the MoE bars against the oracle routed the same way.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from synth import CONFIGS, make_inputs
import nvfp4_weight_only_w4a16_gb300 as P
from tests.test_gpu_parity import DEV, _dev, _layer, assert_layer_close

pytestmark = pytest.mark.gpu

VARIANTS = {
    "sigmoid_bias_renorm_x2.5": dict(score="sigmoid", renormalize=True, scale=2.5, bias="normal0.3"),
    "sigmoid_plain": dict(score="sigmoid", renormalize=False, scale=1.0, bias=None),
    "softmax_full": dict(score="softmax", renormalize=False, scale=1.0, bias=None),
    "softmax_bias": dict(score="softmax", renormalize=True, scale=1.0, bias="normal0.02"),
}


def _bias(kind, E):
    if kind is None:
        return None
    std = float(kind.replace("normal", ""))
    return (np.random.default_rng(77).standard_normal(E) * std).astype(np.float32)


def _set(L, v, E):
    b = _bias(v["bias"], E)
    L.nvfp4_moe_set_scoring(v["score"], v["renormalize"], v["scale"], None if b is None else _dev(b))
    torch.cuda.synchronize()
    return dict(score=v["score"], renormalize=v["renormalize"], scale=v["scale"], bias=b)


def _scores64(logits, sc):
    L = np.asarray(logits, dtype=np.float64)
    if sc["score"] == "sigmoid":
        s = 1.0 / (1.0 + np.exp(-L))
    else:
        ex = np.exp(L - L.max(axis=1, keepdims=True))
        s = ex / ex.sum(axis=1, keepdims=True)
    return s + (0.0 if sc["bias"] is None else sc["bias"][None, :].astype(np.float64))


def _check_route(L, logits, k, E, sc, path):
    L.nvfp4_moe_set_path(path)
    T = logits.shape[0]
    ids, w, off, perm = L.nvfp4_moe_debug_route(_dev(logits), T, k)
    torch.cuda.synchronize()
    L.nvfp4_moe_set_path(P.PATH_AUTO)
    ids, w = ids.cpu().numpy(), w.cpu().numpy().astype(np.float64)
    r = O.route_scored(logits, k, **sc)
    if sc["bias"] is None:
        assert np.array_equal(ids, r.ids)
        _, off_ref, perm_ref = O.permute(r.ids, E)
        assert np.array_equal(off.cpu().numpy(), off_ref)
        assert np.array_equal(perm.cpu().numpy(), perm_ref)
        ref_w = r.weights
    else:
        ch = _scores64(logits, sc)
        tol = 1e-5
        ref_w = np.empty_like(w)
        for t in range(T):
            srt = np.sort(ch[t])[::-1]
            gap = srt[k - 1] - srt[k] if k < E else np.inf
            if gap > tol:
                assert np.array_equal(ids[t], r.ids[t]), t
            else:  # near-tie at the boundary: the GPU's choice must be a valid top-k
                assert len(set(ids[t].tolist())) == k
                assert ch[t, ids[t]].min() >= srt[k - 1] - tol, t
            ref_w[t] = O.route_scored(logits[t:t + 1], k, **sc).weights[0] if np.array_equal(ids[t], r.ids[t]) else \
                _weights_for(logits[t], ids[t], sc)
        _, off_ref, perm_ref = O.permute(ids, E)   # the permutation of the GPU's own choice
        assert np.array_equal(off.cpu().numpy(), off_ref)
        assert np.array_equal(perm.cpu().numpy(), perm_ref)
    assert np.all(np.abs(w - ref_w) <= 1e-6 * np.abs(ref_w) + 1e-7), np.abs(w - ref_w).max()
    return ids


def _weights_for(logit_row, chosen, sc):
    """float64 weights of a given choice (used only at near-ties)."""
    s = (1.0 / (1.0 + np.exp(-np.asarray(logit_row, np.float64))) if sc["score"] == "sigmoid" else
         np.exp(logit_row - logit_row.max()) / np.exp(logit_row - logit_row.max()).sum())
    ws = s[chosen]
    if sc["renormalize"]:
        ws = ws / ws.sum()
    return sc["scale"] * ws


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("path", [P.PATH_DECODE, P.PATH_PREFILL])
def test_scoring_route_and_layer_tiny(variant, path):
    inp = make_inputs("tiny")
    cfg = inp.config
    L = _layer(cfg, max_tokens=512)
    try:
        sc = _set(L, VARIANTS[variant], cfg.num_experts)
        _check_route(L, inp.logits, cfg.top_k, cfg.num_experts, sc, path)
        L.nvfp4_moe_set_path(path)
        x = _dev(inp.x_bits.view(np.int16)).view(torch.bfloat16)
        out = torch.empty((cfg.tokens, cfg.hidden), dtype=torch.bfloat16, device=DEV)
        L.nvfp4_moe_forward(_dev(inp.logits), x, cfg.top_k, out)
        torch.cuda.synchronize()
        assert L.nvfp4_moe_get_status()[0] == 0
        ref = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k, scoring=sc)
        assert_layer_close(out.float().cpu().numpy().astype(np.float64), ref)
    finally:
        L.nvfp4_moe_set_scoring()
        L.nvfp4_moe_set_path(P.PATH_AUTO)


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_scoring_route_full_size(variant):
    # 128 experts: decode (T = 16) and prefill (T = 1024) routing tables
    for name, path in (("decode_c16", P.PATH_DECODE), ("prefill_1k", P.PATH_PREFILL)):
        inp = make_inputs(name)
        cfg = inp.config
        L = _layer(cfg)
        try:
            sc = _set(L, VARIANTS[variant], cfg.num_experts)
            _check_route(L, inp.logits, cfg.top_k, cfg.num_experts, sc, path)
        finally:
            L.nvfp4_moe_set_scoring()


def test_scoring_layer_decode_mtp_sigmoid_bias():
    inp = make_inputs("decode_mtp")
    cfg = inp.config
    L = _layer(cfg, out_f32=True)
    try:
        sc = _set(L, VARIANTS["sigmoid_bias_renorm_x2.5"], cfg.num_experts)
        ids = _check_route(L, inp.logits, cfg.top_k, cfg.num_experts, sc, P.PATH_DECODE)
        assert np.array_equal(ids, O.route_scored(inp.logits, cfg.top_k, **sc).ids)
        x = _dev(inp.x_bits.view(np.int16)).view(torch.bfloat16)
        out = torch.empty((cfg.tokens, cfg.hidden), dtype=torch.float32, device=DEV)
        L.nvfp4_moe_forward(_dev(inp.logits), x, cfg.top_k, out)
        torch.cuda.synchronize()
        assert L.nvfp4_moe_get_status()[0] == 0
        ref = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k, scoring=sc)
        assert_layer_close(out.cpu().numpy().astype(np.float64), ref, bf16_out=False)
    finally:
        L.nvfp4_moe_set_scoring()


def test_scoring_errors():
    L = P.MoELayer(8, 256, 512, 16, 2)
    for bad in (dict(score="softmax", scale=0.0), dict(score="softmax", scale=float("nan")),
                dict(score="softmax", scale=-1.0)):
        with pytest.raises(P.Nvfp4MoeError) as ei:
            L.nvfp4_moe_set_scoring(**bad)
        assert ei.value.status == P.STATUS_CODE["NVFP4_MOE_ERR_INVALID_ARG"]
    assert L.lib.nvfp4_moe_set_scoring(L.h, 2, 1, 1.0, None, None) == P.STATUS_CODE["NVFP4_MOE_ERR_INVALID_ARG"]
    assert L.lib.nvfp4_moe_set_scoring(L.h, 0, 3, 1.0, None, None) == P.STATUS_CODE["NVFP4_MOE_ERR_INVALID_ARG"]
    L.close()
