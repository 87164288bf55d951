"""The process-pool runner of the oracle's layer agrees with moe_forward.

oracle.pool distributes the oracle's own expert_ffn calls over processes and
sums the slots in the same order; the only admissible difference is BLAS
blocking at the float64 rounding level.
"""
import numpy as np

import oracle as O
from oracle.pool import moe_forward_pool
from synth import make_inputs


def test_pool_matches_moe_forward_tiny():
    inp = make_inputs("tiny")
    cfg = inp.config
    ref = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k)
    got, y = moe_forward_pool(inp.logits, inp.x_bits, inp.weights, cfg.top_k, procs=2, return_y=True)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    _, _, y_ref = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k, return_parts=True)
    assert np.allclose(y, y_ref, rtol=1e-12, atol=1e-12 * np.abs(y_ref).max())


def test_pool_matches_moe_forward_shared():
    inp = make_inputs("tiny_shared")
    cfg = inp.config
    ref = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k, num_shared=1)
    got = moe_forward_pool(inp.logits, inp.x_bits, inp.weights, cfg.top_k, num_shared=1, procs=2)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
