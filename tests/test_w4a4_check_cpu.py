"""The W4A4 GPU tests' interval checks, exercised on the CPU.

The checks in tests/intervals.py (used by tests/test_gpu_w4a4.py) accept a kernel's quantisation where it
equals the oracle's, or where it is the neighbour and the exact quotient lies
within D = 4 * 2^-24 (relative) of a rounding midpoint.  Here: the oracle's
own result passes; an FP32 evaluation in the kernels' operation order (the
quotients as products with FP32 reciprocals) passes, including on exact
midpoints where it rounds the other way; a value one step off away from any
midpoint fails; a block quantised with the wrong scale fails.
"""
import numpy as np
import pytest

import oracle as O
from tests.intervals import assert_valid_quantisation, quant_box, D


def _fp32_order(v, input_scale):
    """Quantise like the kernels: scale = E4M3(fl(amax * fl(1 / fl(6 is)))),
    code = E2M1(fl(v * fl(1 / fl(scale * is)))), everything in FP32."""
    v = np.asarray(v, dtype=np.float32)
    isf = np.float32(input_scale)
    blk = v.reshape(-1, 16)
    amax = np.max(np.abs(blk), axis=-1)
    inv6 = np.float32(np.float32(1.0) / np.float32(np.float32(6.0) * isf))
    sc = O.encode_e4m3((amax * inv6).astype(np.float32))
    sv = O.decode_e4m3(sc)
    step = (sv.astype(np.float32) * isf).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        rcp = (np.float32(1.0) / step).astype(np.float32)
        q = (blk * rcp[:, None]).astype(np.float32)
    q = np.where(step[:, None] > 0, q, np.float32(0))
    return (O.decode_e2m1(O.encode_e2m1(q)) * sv[:, None]).reshape(v.shape)


def test_oracle_and_fp32_order_pass():
    rng = np.random.default_rng(4)
    v = rng.standard_normal(4096).astype(np.float32)
    for is_ in (float(np.float32(4.5 / 2688)), 1.0, float(np.float32(1e-3))):
        q, _ = O.quantize_act_nvfp4(v, is_)
        assert_valid_quantisation(q, v.astype(np.float64), v.astype(np.float64), is_)
        assert_valid_quantisation(_fp32_order(v, is_), v.astype(np.float64), v.astype(np.float64), is_)


def test_midpoint_where_the_two_orders_differ():
    is_ = float(np.float32(0.9012069702148438))
    blk = np.zeros(16)
    blk[0] = float(np.float32(6.0 * is_))
    blk[1] = 2.5 * is_
    q, _ = O.quantize_act_nvfp4(blk, is_)
    f = _fp32_order(blk, is_)
    assert q[1] == 2.0 and f[1] == 3.0       # the two decisions really differ here
    assert_valid_quantisation(q, blk, blk, is_)
    assert_valid_quantisation(f, blk, blk, is_)
    vmin, vmax = quant_box(blk, blk, is_)
    assert vmin[1] == 2.0 and vmax[1] == 3.0


def test_wrong_rounding_is_rejected():
    rng = np.random.default_rng(5)
    v = rng.standard_normal(16)
    is_ = float(np.float32(4.5 / 2688))
    q, sc = O.quantize_act_nvfp4(v, is_)
    sv = float(O.decode_e4m3(sc)[0])
    grid = O.decode_e2m1(np.arange(8))
    # an element whose quotient is far from every midpoint, moved one code up
    quot = np.abs(v) / (sv * is_)
    mids = (grid[1:] + grid[:-1]) / 2
    far = [i for i in range(16) if np.min(np.abs(quot[i] - mids)) > 1e-3 and abs(q[i]) / sv < 6]
    i = far[0]
    up = grid[np.searchsorted(grid, abs(q[i]) / sv) + 1] * sv * np.sign(v[i])
    bad = q.copy()
    bad[i] = up
    with pytest.raises(AssertionError):
        assert_valid_quantisation(bad, v, v, is_)
    # the whole block on a scale one E4M3 step away (the amax is far from its midpoint)
    sv2 = float(O.decode_e4m3(int(sc[0]) + 1))
    other = O.decode_e2m1(O.encode_e2m1(v / (sv2 * is_))) * sv2
    with pytest.raises(AssertionError):
        assert_valid_quantisation(other, v, v, is_)


def test_input_intervals_widen_the_admissible_set():
    # an input interval straddling a midpoint admits both neighbours
    is_ = 1.0
    blk = np.zeros(16)
    blk[0] = 6.0
    lo, hi = blk.copy(), blk.copy()
    lo[1], hi[1] = 2.4, 2.6
    vmin, vmax = quant_box(lo, hi, is_)
    assert vmin[1] == 2.0 and vmax[1] == 3.0
    assert D < 1e-6


def _layer_fp32_order(inp, iscale, monkeypatch):
    """The oracle's W4A4 layer with its quantiser evaluated in the kernels'
    FP32 operation order (a stand-in for a correct GPU result)."""
    import oracle.nvfp4_moe_oracle as OM
    monkeypatch.setattr(OM, "quantize_act_nvfp4",
                        lambda v, i: (_fp32_order(np.asarray(v, np.float32).reshape(-1, np.asarray(v).shape[-1]), i)
                                      .reshape(np.asarray(v).shape), None))
    cfg = inp.config
    out = O.moe_forward_w4a4(inp.logits, inp.x_bits, inp.weights, cfg.top_k, iscale, num_shared=cfg.shared)
    monkeypatch.undo()
    return out


@pytest.mark.parametrize("name", ["tiny", "tiny_shared"])
def test_layer_allowance_admits_fp32_order_and_rejects_a_wrong_scale(name, monkeypatch):
    from synth import make_inputs, make_input_scales
    from tests.intervals import w4a4_layer_allowance, assert_w4a4_layer
    inp = make_inputs(name)
    cfg = inp.config
    iscale = make_input_scales(cfg)
    ref = O.moe_forward_w4a4(inp.logits, inp.x_bits, inp.weights, cfg.top_k, iscale, num_shared=cfg.shared)
    r = O.route(inp.logits, cfg.top_k)
    ids, wts = r.ids, r.weights
    if cfg.shared:
        ids = np.concatenate([ids, np.full((cfg.tokens, 1), cfg.num_experts, np.int32)], axis=1)
        wts = np.concatenate([wts, np.ones((cfg.tokens, 1))], axis=1)
    A = w4a4_layer_allowance(inp.weights, inp.x_bits, ids, wts, iscale, cfg.num_experts, np.arange(cfg.tokens))
    got = _layer_fp32_order(inp, iscale, monkeypatch)
    assert np.abs(got - ref).max() > 1e-2 * np.sqrt(np.mean(ref ** 2))   # the flips are really there
    assert_w4a4_layer(got, ref, A)
    # one expert's x input scale off by a factor 1.37 (a power of two would
    # only move every block scale by that power: the values stay the same)
    bad_scale = iscale.copy()
    bad_scale[int(r.ids[0, 0]), 0] *= np.float32(1.37)
    wrong = O.moe_forward_w4a4(inp.logits, inp.x_bits, inp.weights, cfg.top_k, bad_scale, num_shared=cfg.shared)
    with pytest.raises(AssertionError):
        assert_w4a4_layer(wrong, ref, A)
