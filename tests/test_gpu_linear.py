"""The dense W4A16 NVFP4 linear, on the GPU, against the oracle.

out[t] = gs * W x[t] for one NVFP4 matrix W [N][K] ("GLM-5.3-Flash-NVFP4-h —
W4A16 dense-side quantization": the attention linears, shared experts and
lm_head in weight-only NVFP4 with 16-element groups).  Shapes: a small
matrix whose N is not a multiple of 128 (the library pads the last 128-row
block with zeros and must never write the padding out) and the fused KDA
in_proj, N = 12576, K = 4096 ("tacos4me/GLM-5.3-Flash-NVFP4-FP8ATTN-512K",
The kernel story), at a 2-token MTP step and a 1024-token prefill piece.

Bar, from the arithmetic: every weight is exact in FP16 and in BF16 (an E2M1
value times an E4M3 scale has at most 6 significant bits) and so is every
activation (BF16, or FP16 after an exact power-of-two prescale), so each
product is exact in FP32 and the only error is the FP32 summation of K
products plus the final scaling: |gpu - exact| <= (K + 2) * 2^-24 *
sum_k |gs x_k w_k|, taken here with a 4x margin for the tensor core's
accumulation order, plus the BF16 rounding of the output (2^-8 of each
value).  The layer bounds of the MoE tests (RMS, mean, norm ratio, cosine)
hold as well.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from synth import LINEAR_CONFIGS, make_linear_inputs
import nvfp4_weight_only_w4a16_gb300 as P
from tests.test_gpu_parity import DEV, _dev, assert_layer_close

pytestmark = pytest.mark.gpu

_LIN = {}


def _linear(cfg, max_tokens, out_f32=False):
    key = (cfg.out_features, cfg.in_features, cfg.weight_std, cfg.seed, max_tokens, out_f32)
    if key not in _LIN:
        for k in list(_LIN):
            _LIN.pop(k).close()
        P.build()
        L = P.Linear(cfg.out_features, cfg.in_features, max_tokens, out_f32=out_f32)
        inp = make_linear_inputs(cfg)
        L.nvfp4_linear_pack(_dev(inp.w_q), _dev(inp.w_s), _dev(np.array([inp.gscale], np.float32)))
        torch.cuda.synchronize()
        _LIN[key] = L
    return _LIN[key]


def _run(L, x_bits, path, out_f32=False):
    L.nvfp4_moe_set_path(path)
    T = x_bits.shape[0]
    x = _dev(x_bits.view(np.int16)).view(torch.bfloat16)
    # one spare row on each side: the library must write exactly [T][N]
    buf = torch.full((T + 2, L.N), float("nan"), dtype=torch.float32 if out_f32 else torch.bfloat16, device=DEV)
    out = buf[1:T + 1]
    L.nvfp4_linear_forward(x, out)
    torch.cuda.synchronize()
    st, _ = L.nvfp4_moe_get_status()
    assert st == 0, P.STATUS[st]
    L.nvfp4_moe_set_path(P.PATH_AUTO)
    b = buf.float().cpu().numpy()
    assert np.all(np.isnan(b[0])) and np.all(np.isnan(b[-1])), "wrote outside out"
    return b[1:T + 1].astype(np.float64)


def _abs_sum(x_bits, inp):
    """sum_k |gs x_k w_k| per output: the scale of the summation error."""
    x = np.abs(O.bf16_bits_to_f64(x_bits))
    return float(inp.gscale) * (x @ np.abs(O.dequant(inp.w_q, inp.w_s)).T)


def _check(gpu, ref, abs_sum, K, bf16_out):
    bound = 4.0 * (K + 2) * 2.0 ** -24 * abs_sum + (2.0 ** -8 * np.abs(gpu) if bf16_out else 0.0)
    err = np.abs(gpu - ref)
    assert np.all(np.isfinite(gpu))
    assert np.all(err <= bound), (err.max(), (err / np.maximum(bound, 1e-30)).max())
    assert_layer_close(gpu, ref, bf16_out=bf16_out)


@pytest.mark.parametrize("path", [P.PATH_DECODE, P.PATH_PREFILL])
@pytest.mark.parametrize("T", [1, 5, 8, 9, 16])
def test_linear_tiny(path, T):
    cfg = LINEAR_CONFIGS["linear_tiny"]
    inp = make_linear_inputs(cfg, tokens=T)
    L = _linear(cfg, 512)
    gpu = _run(L, inp.x_bits, path)
    ref = O.linear_forward(inp.x_bits, inp.w_q, inp.w_s, inp.gscale)
    _check(gpu, ref, _abs_sum(inp.x_bits, inp), cfg.in_features, True)


@pytest.mark.parametrize("T", [37, 128, 300])
def test_linear_tiny_prefill_ragged(T):
    cfg = LINEAR_CONFIGS["linear_tiny"]
    inp = make_linear_inputs(cfg, tokens=T)
    L = _linear(cfg, 512)
    gpu = _run(L, inp.x_bits, P.PATH_PREFILL)
    ref = O.linear_forward(inp.x_bits, inp.w_q, inp.w_s, inp.gscale)
    _check(gpu, ref, _abs_sum(inp.x_bits, inp), cfg.in_features, True)


def test_linear_tiny_f32_out_and_auto_path():
    cfg = LINEAR_CONFIGS["linear_tiny"]
    L = _linear(cfg, 512, out_f32=True)
    for T in (2, 37):  # AUTO: the decode kernel, then the GEMM
        inp = make_linear_inputs(cfg, tokens=T)
        gpu = _run(L, inp.x_bits, P.PATH_AUTO, out_f32=True)
        ref = O.linear_forward(inp.x_bits, inp.w_q, inp.w_s, inp.gscale)
        _check(gpu, ref, _abs_sum(inp.x_bits, inp), cfg.in_features, False)


def test_linear_packed_blob_is_the_down_layout_with_zero_padding():
    cfg = LINEAR_CONFIGS["linear_tiny"]
    inp = make_linear_inputs(cfg)
    L = _linear(cfg, 512)
    blob = L.nvfp4_moe_debug_packed_blob().cpu().numpy()
    N, K = cfg.out_features, cfg.in_features
    Np = (N + 127) // 128 * 128
    q = np.zeros((Np, K // 2), np.uint8)
    s = np.zeros((Np, K // 16), np.uint8)
    q[:N], s[:N] = inp.w_q, inp.w_s
    nch = K // 64
    # per tile [rb][c]: codes [sb 8][slot 32][half 2][8 bytes], then the scales in the same order;
    # segment t = 4 t4 + q of a 16-row sub-block sits at slot 8 q + (t4 + 2 q) % 8
    seg = q.reshape(Np // 128, 8, 2, 8, nch, 4, 8).transpose(0, 4, 1, 3, 5, 2, 6).reshape(Np // 128, nch, 8, 32, 16)
    sseg = s.reshape(Np // 128, 8, 2, 8, nch, 4).transpose(0, 4, 1, 3, 5, 2).reshape(Np // 128, nch, 8, 32, 2)
    t = np.arange(32)
    slot = 8 * (t % 4) + (t // 4 + 2 * (t % 4)) % 8
    nib_s, sc_s = np.empty_like(seg), np.empty_like(sseg)
    nib_s[:, :, :, slot] = seg
    sc_s[:, :, :, slot] = sseg
    nib, sc = nib_s.reshape(Np // 128, nch, 4096), sc_s.reshape(Np // 128, nch, 512)
    assert np.array_equal(blob, np.concatenate([nib, sc], axis=2).reshape(-1))


@pytest.mark.parametrize("out_f32", [False, True])
def test_linear_kda_in_proj_mtp_decode(out_f32):
    cfg = LINEAR_CONFIGS["kda_in_proj_mtp"]
    inp = make_linear_inputs(cfg)
    L = _linear(cfg, 1024, out_f32=out_f32)
    gpu = _run(L, inp.x_bits, P.PATH_AUTO, out_f32=out_f32)
    ref = O.linear_forward(inp.x_bits, inp.w_q, inp.w_s, inp.gscale)
    _check(gpu, ref, _abs_sum(inp.x_bits, inp), cfg.in_features, not out_f32)


def test_linear_kda_in_proj_1k_prefill_sampled():
    cfg = LINEAR_CONFIGS["kda_in_proj_1k"]
    inp = make_linear_inputs(cfg)
    L = _linear(cfg, 1024)
    gpu = _run(L, inp.x_bits, P.PATH_AUTO)
    rows = np.unique(np.concatenate([[0, 127, 128, 1023], np.random.default_rng(5).choice(1024, 28, replace=False)]))
    ref = O.linear_forward(inp.x_bits[rows], inp.w_q, inp.w_s, inp.gscale)
    _check(gpu[rows], ref, _abs_sum(inp.x_bits[rows], inp), cfg.in_features, True)


def test_linear_errors():
    cfg = LINEAR_CONFIGS["linear_tiny"]
    inp = make_linear_inputs(cfg)
    L = P.Linear(cfg.out_features, cfg.in_features, 64)
    x = torch.zeros((4, cfg.in_features), dtype=torch.bfloat16, device=DEV)
    out = torch.empty((4, cfg.out_features), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(P.Nvfp4MoeError) as ei:
        L.nvfp4_linear_forward(x, out)
    assert ei.value.status == P.STATUS_CODE["NVFP4_MOE_ERR_NOT_PACKED"]
    for bad in (0.0, -1.0, np.nan, np.inf):
        with pytest.raises(P.Nvfp4MoeError) as ei:
            L.nvfp4_linear_pack(_dev(inp.w_q), _dev(inp.w_s), _dev(np.array([bad], np.float32)))
        assert ei.value.status == P.STATUS_CODE["NVFP4_MOE_ERR_BAD_SCALE"]
    L.nvfp4_linear_pack(_dev(inp.w_q), _dev(inp.w_s), _dev(np.array([inp.gscale], np.float32)))
    big = torch.zeros((65, cfg.in_features), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(P.Nvfp4MoeError) as ei:
        L.nvfp4_linear_forward(big, torch.empty((65, cfg.out_features), dtype=torch.bfloat16, device=DEV))
    assert ei.value.status == P.STATUS_CODE["NVFP4_MOE_ERR_UNSUPPORTED_SHAPE"]
    # an MoE call on a linear handle, and a linear call on an MoE handle
    with pytest.raises(P.Nvfp4MoeError) as ei:
        L.nvfp4_moe_forward(torch.zeros((4, 1), device=DEV), x, 1, out)
    assert ei.value.status == P.STATUS_CODE["NVFP4_MOE_ERR_INVALID_ARG"]
    M = P.MoELayer(8, 256, 512, 16, 2)
    st = M.lib.nvfp4_linear_forward(M.h, 4, P.binding._ptr(x), P.binding._ptr(out), P.binding._stream())
    assert st == P.STATUS_CODE["NVFP4_MOE_ERR_INVALID_ARG"]
    M.close()
    L.close()
