"""The layer with its single shared expert, on the GPU, against the oracle.

The shared expert is expert E of the packed blob; every token uses it with
weight 1 after its top_k routed experts ("GLM-5.3-Flash on Blackwell", The
model loaded, served an API, and produced garbage: "the single shared
expert"; "GLM-5.3-Flash-NVFP4-h — W4A16 dense-side quantization": shared
experts in W4A16 NVFP4).  Routing (ids, weights, offsets, perm) is
bit-exact; the layer meets the same bounds as the routed-only layer.
"""
import numpy as np
import pytest
import torch

import nvfp4_weight_only_w4a16_gb300 as P
from oracle import nvfp4_moe_oracle as O
from synth import CONFIGS, LayerConfig, make_inputs, make_layer_weights
from tests.test_gpu_parity import check_rows, DEV, _dev, _forward, assert_layer_close

pytestmark = pytest.mark.gpu

_SHARED = {}


def _shared_layer(cfg: LayerConfig, max_tokens=None):
    key = (cfg.num_experts, cfg.hidden, cfg.inter, cfg.seed, max_tokens or cfg.tokens, cfg.top_k)
    if key not in _SHARED:
        for k in list(_SHARED):
            _SHARED.pop(k).close()
        P.build()
        L = P.MoELayer(cfg.num_experts, cfg.hidden, cfg.inter, max_tokens or cfg.tokens, cfg.top_k,
                       num_shared_experts=1)
        P.upload_layer(L, make_layer_weights(cfg), DEV)
        _SHARED[key] = L
    return _SHARED[key]


def _check_shared_route(L, logits, k, E, path):
    L.nvfp4_moe_set_path(path)
    T = logits.shape[0]
    ids, w, off, perm = L.nvfp4_moe_debug_route(_dev(logits), T, k)
    torch.cuda.synchronize()
    L.nvfp4_moe_set_path(P.PATH_AUTO)
    r = O.route(logits, k)
    ids_ref = np.concatenate([r.ids, np.full((T, 1), E, np.int32)], axis=1)
    _, off_ref, perm_ref = O.permute(ids_ref, E + 1)
    ids, w = ids.cpu().numpy(), w.cpu().numpy().astype(np.float64)
    assert np.array_equal(ids, ids_ref)
    assert np.all(w[:, k] == 1.0)
    assert np.all(np.abs(w[:, :k] - r.weights) <= 2e-6 * np.abs(r.weights) + 1e-30)
    assert np.array_equal(off.cpu().numpy(), off_ref)
    assert np.array_equal(perm.cpu().numpy(), perm_ref)


MID = LayerConfig("mid_shared", 16, 1024, 512, 4, 64, "normal0.5", shared=1)


@pytest.mark.parametrize("path", [P.PATH_DECODE, P.PATH_PREFILL])
def test_route_shared(path):
    for cfg in (CONFIGS["tiny_shared"], MID):
        inp = make_inputs(cfg)
        L = _shared_layer(cfg)
        logits = inp.logits[:16] if path == P.PATH_DECODE else inp.logits
        _check_shared_route(L, logits, cfg.top_k, cfg.num_experts, path)


@pytest.mark.parametrize("path", [P.PATH_DECODE, P.PATH_PREFILL])
def test_forward_shared_tiny(path):
    inp = make_inputs("tiny_shared")
    cfg = inp.config
    L = _shared_layer(cfg)
    gpu = _forward(L, inp.logits, inp.x_bits, cfg.top_k, path)
    ref = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k, num_shared=1)
    assert_layer_close(gpu, ref)
    # the shared expert really contributes: the routed-only result is far off
    routed = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k)
    assert np.abs(routed - ref).mean() > 0.5 * np.abs(ref).mean()


def test_forward_shared_mid_both_paths():
    inp = make_inputs(MID)
    cfg = inp.config
    L = _shared_layer(cfg)
    gpu = _forward(L, inp.logits, inp.x_bits, cfg.top_k, P.PATH_PREFILL)
    ref = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k, num_shared=1)
    assert_layer_close(gpu, ref)
    gpu16 = _forward(L, inp.logits[:16], inp.x_bits[:16], cfg.top_k, P.PATH_DECODE)
    assert_layer_close(gpu16, ref[:16])


def test_intermediates_shared_tiny():
    inp = make_inputs("tiny_shared")
    cfg = inp.config
    L = _shared_layer(cfg)
    _forward(L, inp.logits, inp.x_bits, cfg.top_k, P.PATH_DECODE)
    T, k, E = cfg.tokens, cfg.top_k, cfg.num_experts
    K = k + 1
    check_rows(L, inp, range(T * K))


def test_forward_shared_mtp_full_size():
    inp = make_inputs("decode_mtp_shared")
    cfg = inp.config
    L = _shared_layer(cfg, max_tokens=16)
    gpu = _forward(L, inp.logits, inp.x_bits, cfg.top_k)
    ref = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k, num_shared=1)
    assert_layer_close(gpu, ref)
