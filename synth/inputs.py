"""Seeded synthetic workloads for the weight-only NVFP4 (W4A16) MoE layer.

The five workloads are the shapes the GLM-5.3-Flash serving pages run the
routed-expert layer at: 2-token MTP decode steps ("tacos4me/GLM-5.3-Flash-
NVFP4-FP8ATTN-512K", TL;DR table: MTP k=1), eight 2-token streams, 1024-token
chunked-prefill pieces (same card, Quickstart: --max-num-batched-tokens 1024)
and a 16K-token prefill ("GLM-5.3-Flash NVFP4 W4A16 for 2x RTX PRO 6000
Blackwell", Measured results).  No dataset is involved; every value is drawn
from numpy's PCG64 from a fixed seed.

Draw order.  Activation-side values come from the stream
``SeedSequence(seed, spawn_key=(0,))``: router logits [T][E] (standard
normal, float32), then x [T][H] (standard normal, float32, rounded to BF16),
then the per-expert logit bias.  Expert e's weights come from their own stream
``SeedSequence(seed, spawn_key=(1, e))``, so the three E128 workloads share one
set of expert weights and any expert can be regenerated alone.

Weight encoding (input preparation, not the layer under test).  FP32 weights
~ N(0, std) are encoded to NVFP4 as the ModelOpt-style weight-only format the
pages ship ("tenhkspark/GLM-5.3-Flash-NVFP4-Wabi", Config expectations:
group_size = 16 plus a per-module weight_scale_2): per tensor g = amax/(6*448)
in FP32; per 16-element block along K the E4M3 scale s = RNE_sat((amax_blk/6)/g);
each element's E2M1 code = RNE_sat(w / (s*g)), ties to the even code.  A block
whose amax is 0, or whose scale rounds to 0, gets all-zero codes.

Canonical byte layout handed to the library (per expert, nn.Linear order, N
output rows by K reduction columns):
  w13_q [2I][H/2]  gate rows 0..I-1 then up rows I..2I-1; element 2j in the
                   low nibble of byte j, element 2j+1 in the high nibble
  w13_s [2I][H/16] E4M3 bytes, one per 16 consecutive K elements
  w2_q  [H][I/2], w2_s [H][I/16]  the down projection, same rules
  gscale [3]       FP32 tensor scales: gate, up, down
"""
from __future__ import annotations

import concurrent.futures as _cf
import multiprocessing as _mp
import os
from dataclasses import dataclass, field
from functools import lru_cache

import numpy as np

E2M1_MAX = 6.0
E4M3_MAX = 448.0


@dataclass(frozen=True)
class LayerConfig:
    name: str
    num_experts: int
    hidden: int
    inter: int
    top_k: int
    tokens: int
    logits_bias: str = "none"      # "none" | "normal0.5" | "zipf1.1"
    outlier_frac: float = 0.0       # share of weights multiplied by outlier_mult
    outlier_mult: float = 1.0
    weight_std: float = 0.02
    seed: int = 0
    shared: int = 0                 # 1: one shared expert (weights of expert index num_experts)

    def with_tokens(self, tokens: int) -> "LayerConfig":
        return LayerConfig(self.name, self.num_experts, self.hidden, self.inter,
                           self.top_k, tokens, self.logits_bias, self.outlier_frac,
                           self.outlier_mult, self.weight_std, self.seed, self.shared)

    @property
    def expert_bytes(self) -> int:
        """NVFP4 bytes of one expert: 3*H*I nibbles plus one scale byte per 16."""
        n = 3 * self.hidden * self.inter
        return n // 2 + n // 16


CONFIGS = {
    # E8 H256 I512 top-2, 16 tokens: small enough for brute force everywhere.
    "tiny": LayerConfig("tiny", 8, 256, 512, 2, 16),
    # One MTP decode step: the token plus one speculative token.
    "decode_mtp": LayerConfig("decode_mtp", 128, 4096, 1536, 8, 2),
    # Eight streams x 2-token MTP verify, uniform routing.
    "decode_c16": LayerConfig("decode_c16", 128, 4096, 1536, 8, 16),
    # A 1024-token chunked-prefill piece, mild imbalance from a N(0, 0.5) bias.
    "prefill_1k": LayerConfig("prefill_1k", 128, 4096, 1536, 8, 1024, "normal0.5"),
    # 16K-token prefill over 256 experts, Zipf(1.1) popularity, 1% x20 outliers.
    "prefill_16k": LayerConfig("prefill_16k", 256, 4096, 1536, 8, 16384, "zipf1.1",
                               0.01, 20.0),
    # The tiny layer and the MTP step with the layer's single shared expert.
    "tiny_shared": LayerConfig("tiny_shared", 8, 256, 512, 2, 16, shared=1),
    "decode_mtp_shared": LayerConfig("decode_mtp_shared", 128, 4096, 1536, 8, 2, shared=1),
}


@dataclass
class ExpertWeights:
    """Canonical NVFP4 bytes for all experts (see module docstring)."""
    w13_q: np.ndarray   # u8 [E][2I][H/2]
    w13_s: np.ndarray   # u8 [E][2I][H/16]
    w2_q: np.ndarray    # u8 [E][H][I/2]
    w2_s: np.ndarray    # u8 [E][H][I/16]
    gscale: np.ndarray  # f32 [E][3]  (gate, up, down)


@dataclass
class LayerInputs:
    config: LayerConfig
    logits: np.ndarray          # f32 [T][E]
    x_bits: np.ndarray          # u16 [T][H]  BF16 bit patterns
    weights: ExpertWeights
    expert_bias: np.ndarray = field(default=None)  # f32 [E] already added to logits


# ----------------------------------------------------------------------------
# Encoders (round-to-nearest-even, saturating).  Encoding only: nothing here
# turns a code back into a value.
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def encode_e4m3_rne(v: np.ndarray):
    """Encode non-negative float values as OCP E4M3 (bias 7, max 448).

    Returns (codes u8, rounded value float64).  Values above 448 saturate to
    448 (code 0x7E); subnormals are multiples of 2**-9.
    """
    v = np.asarray(v, dtype=np.float64)
    if np.any(v < 0) or np.any(~np.isfinite(v)):
        raise ValueError("E4M3 scale encoder expects finite non-negative values")
    code = np.zeros(v.shape, dtype=np.int64)
    val = np.zeros(v.shape, dtype=np.float64)
    sat = v >= E4M3_MAX
    sub = v < 2.0 ** -6
    nrm = ~sat & ~sub
    # subnormal range: step 2**-9; a result of 8 steps is the smallest normal
    m = np.rint(v[sub] * 2.0 ** 9)
    code[sub] = m.astype(np.int64)          # m == 8 is exponent field 1, mantissa 0
    val[sub] = m * 2.0 ** -9
    # normal range: 3 fraction bits
    mant, ex = np.frexp(v[nrm])             # v = mant * 2**ex, mant in [0.5, 1)
    e = ex - 1                              # v = (2*mant) * 2**e, 2*mant in [1, 2)
    q = np.rint(mant * 16.0)                # (2*mant)*8, in [8, 16]
    carry = q >= 16
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 8.0, q)
    code[nrm] = ((e + 7) << 3) | (q.astype(np.int64) - 8)
    val[nrm] = q / 8.0 * np.exp2(e.astype(np.float64))
    code[sat] = 0x7E
    val[sat] = E4M3_MAX
    return code.astype(np.uint8), val


def encode_e2m1_rne(v: np.ndarray) -> np.ndarray:
    """Encode float values as 4-bit E2M1 codes (sign in bit 3), ties to even code.

    Magnitude codes 0..7 stand for 0, 0.5, 1, 1.5, 2, 3, 4, 6; a magnitude
    above 6 saturates to code 7.  The midpoints between neighbours are the
    decision points; at a midpoint the even code wins.
    """
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v)
    code = ((a > 0.25).astype(np.uint8)
            + (a >= 0.75) + (a > 1.25) + (a >= 1.75)
            + (a > 2.5) + (a >= 3.5) + (a > 5.0)).astype(np.uint8)
    code |= (np.signbit(v).astype(np.uint8) << 3)
    return code


def quantize_nvfp4(w: np.ndarray):
    """Encode an FP32 matrix [N][K] (K % 16 == 0) as NVFP4.

    Returns (q u8 [N][K/2], s u8 [N][K/16], g float32).
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    if k % 16:
        raise ValueError("K must be a multiple of 16")
    amax = np.float32(np.max(np.abs(w))) if w.size else np.float32(0)
    g = np.float32(amax / np.float32(E2M1_MAX * E4M3_MAX)) if amax > 0 else np.float32(1.0)
    blk = w.reshape(n, k // 16, 16)
    amax_blk = np.max(np.abs(blk), axis=2)                         # f32
    s_target = (amax_blk / np.float32(E2M1_MAX)) / g               # f32 arithmetic
    s_code, s_val = encode_e4m3_rne(s_target.astype(np.float64))
    denom = (s_val.astype(np.float32) * g).astype(np.float32)      # exact scale, f32
    with np.errstate(divide="ignore", invalid="ignore"):
        r = blk / denom[:, :, None]
    r = np.where(denom[:, :, None] > 0, r, np.float32(0)).astype(np.float32)
    codes = encode_e2m1_rne(r).reshape(n, k)
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return q, s_code.reshape(n, k // 16), g


# ----------------------------------------------------------------------------
# Seeded draws
# ----------------------------------------------------------------------------

def _expert_rng(seed: int, e: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(1, e))))


def make_expert_weights(cfg: LayerConfig, e: int):
    """Draw expert e's FP32 weights and encode them.  Returns a tuple of
    (w13_q, w13_s, w2_q, w2_s, gscale[3])."""
    rng = _expert_rng(cfg.seed, e)
    H, I = cfg.hidden, cfg.inter
    w13 = rng.standard_normal((2 * I, H), dtype=np.float32) * np.float32(cfg.weight_std)
    w2 = rng.standard_normal((H, I), dtype=np.float32) * np.float32(cfg.weight_std)
    if cfg.outlier_frac > 0:
        m13 = rng.random((2 * I, H), dtype=np.float32) < cfg.outlier_frac
        m2 = rng.random((H, I), dtype=np.float32) < cfg.outlier_frac
        w13[m13] *= np.float32(cfg.outlier_mult)
        w2[m2] *= np.float32(cfg.outlier_mult)
    qg, sg, gg = quantize_nvfp4(w13[:I])
    qu, su, gu = quantize_nvfp4(w13[I:])
    qd, sd, gd = quantize_nvfp4(w2)
    return (np.concatenate([qg, qu]), np.concatenate([sg, su]), qd, sd,
            np.array([gg, gu, gd], dtype=np.float32))


def _worker(args):
    cfg, lo, hi = args
    return lo, [make_expert_weights(cfg, e) for e in range(lo, hi)]


def _weight_key(cfg: LayerConfig):
    # routed experts 0..E-1, then the shared expert (if any) as expert E
    return (cfg.num_experts + cfg.shared, cfg.hidden, cfg.inter, cfg.outlier_frac,
            cfg.outlier_mult, cfg.weight_std, cfg.seed)


@lru_cache(maxsize=2)
def _layer_weights_cached(key) -> ExpertWeights:
    E, H, I, of, om, std, seed = key
    cfg = LayerConfig("w", E, H, I, 1, 1, "none", of, om, std, seed)
    w13_q = np.empty((E, 2 * I, H // 2), np.uint8)
    w13_s = np.empty((E, 2 * I, H // 16), np.uint8)
    w2_q = np.empty((E, H, I // 2), np.uint8)
    w2_s = np.empty((E, H, I // 16), np.uint8)
    gs = np.empty((E, 3), np.float32)

    def put(lo, res):
        for i, (a, b, c, d, g) in enumerate(res):
            w13_q[lo + i], w13_s[lo + i], w2_q[lo + i], w2_s[lo + i], gs[lo + i] = a, b, c, d, g

    work = E * H * I
    nproc = min(len(os.sched_getaffinity(0)), 16)
    if work < (1 << 24) or nproc <= 1:
        put(0, [make_expert_weights(cfg, e) for e in range(E)])
    else:
        chunk = max(1, E // (4 * nproc))
        jobs = [(cfg, lo, min(E, lo + chunk)) for lo in range(0, E, chunk)]
        # spawn, never fork: the parent may already hold a CUDA context
        with _cf.ProcessPoolExecutor(nproc, mp_context=_mp.get_context("spawn")) as ex:
            for lo, res in ex.map(_worker, jobs):
                put(lo, res)
    return ExpertWeights(w13_q, w13_s, w2_q, w2_s, gs)


def make_layer_weights(cfg: LayerConfig) -> ExpertWeights:
    """All experts' NVFP4 bytes for cfg (cached per weight recipe); with a
    shared expert, num_experts + 1 of them."""
    return _layer_weights_cached(_weight_key(cfg))


def make_activations(cfg: LayerConfig):
    """Router logits (f32 [T][E], bias included), x BF16 bits [T][H], bias [E]."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(cfg.seed, spawn_key=(0,))))
    T, E, H = cfg.tokens, cfg.num_experts, cfg.hidden
    logits = rng.standard_normal((T, E), dtype=np.float32)
    x = rng.standard_normal((T, H), dtype=np.float32)
    if cfg.logits_bias == "none":
        bias = np.zeros(E, np.float32)
    elif cfg.logits_bias == "normal0.5":
        bias = (rng.standard_normal(E, dtype=np.float32) * np.float32(0.5)).astype(np.float32)
    elif cfg.logits_bias == "zipf1.1":
        rank = rng.permutation(E).astype(np.float64) + 1.0
        bias = (-1.1 * np.log(rank)).astype(np.float32)
    else:
        raise ValueError(cfg.logits_bias)
    logits = (logits + bias[None, :]).astype(np.float32)
    return logits, f32_to_bf16_bits(x), bias


def make_inputs(name_or_cfg, tokens: int | None = None) -> LayerInputs:
    cfg = CONFIGS[name_or_cfg] if isinstance(name_or_cfg, str) else name_or_cfg
    if tokens is not None:
        cfg = cfg.with_tokens(tokens)
    logits, x_bits, bias = make_activations(cfg)
    return LayerInputs(cfg, logits, x_bits, make_layer_weights(cfg), bias)


# ----------------------------------------------------------------------------
# Dense W4A16 linears
# ----------------------------------------------------------------------------
# The dense side of the model (attention linears, shared experts, lm_head) in
# the same weight-only NVFP4 format ("GLM-5.3-Flash-NVFP4-h — W4A16
# dense-side quantization", opening summary).  The one dense shape the pages
# print is the fused KDA in_proj, N = 12576 outputs over K = 4096
# ("tacos4me/GLM-5.3-Flash-NVFP4-FP8ATTN-512K", The kernel story); it runs at
# the MTP decode step (2 tokens) and at a 1024-token prefill piece.  Weights
# W ~ N(0, std) [N][K] are encoded by quantize_nvfp4 from the stream
# SeedSequence(seed, spawn_key=(2,)); x [T][K] (standard normal, rounded to
# BF16) from SeedSequence(seed, spawn_key=(3,)).

@dataclass(frozen=True)
class LinearConfig:
    name: str
    out_features: int   # N
    in_features: int    # K
    tokens: int         # T
    weight_std: float = 0.02
    seed: int = 0

    def with_tokens(self, tokens: int) -> "LinearConfig":
        return LinearConfig(self.name, self.out_features, self.in_features, tokens, self.weight_std, self.seed)

    @property
    def weight_bytes(self) -> int:
        n = self.out_features * self.in_features
        return n // 2 + n // 16


LINEAR_CONFIGS = {
    # small, N not a multiple of 128 (the last 128-row block is padded), ragged T
    "linear_tiny": LinearConfig("linear_tiny", 272, 256, 37),
    "kda_in_proj_mtp": LinearConfig("kda_in_proj_mtp", 12576, 4096, 2),
    "kda_in_proj_1k": LinearConfig("kda_in_proj_1k", 12576, 4096, 1024),
}


@dataclass
class LinearInputs:
    config: LinearConfig
    w_q: np.ndarray     # u8 [N][K/2]
    w_s: np.ndarray     # u8 [N][K/16]
    gscale: np.float32  # the tensor scale
    x_bits: np.ndarray  # u16 [T][K]  BF16 bit patterns


@lru_cache(maxsize=2)
def _linear_weights_cached(N: int, K: int, std: float, seed: int):
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(2,))))
    w = rng.standard_normal((N, K), dtype=np.float32) * np.float32(std)
    return quantize_nvfp4(w)


def make_linear_inputs(name_or_cfg, tokens: int | None = None) -> LinearInputs:
    cfg = LINEAR_CONFIGS[name_or_cfg] if isinstance(name_or_cfg, str) else name_or_cfg
    if tokens is not None:
        cfg = cfg.with_tokens(tokens)
    q, s, g = _linear_weights_cached(cfg.out_features, cfg.in_features, cfg.weight_std, cfg.seed)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(cfg.seed, spawn_key=(3,))))
    x = rng.standard_normal((cfg.tokens, cfg.in_features), dtype=np.float32)
    return LinearInputs(cfg, q, s, np.float32(g), f32_to_bf16_bits(x))


def make_router_weight(cfg: LayerConfig) -> np.ndarray:
    """BF16 bit patterns of a router linear W [E][H] (routed experts only),
    N(0, 1/H) from SeedSequence(seed, spawn_key=(4,)), so that the logits of
    N(0, 1) activations are about N(0, 1) like the given-logits workloads."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(cfg.seed, spawn_key=(4,))))
    w = rng.standard_normal((cfg.num_experts, cfg.hidden), dtype=np.float32) / np.float32(np.sqrt(cfg.hidden))
    return f32_to_bf16_bits(w)


def make_input_scales(cfg: LayerConfig) -> np.ndarray:
    """W4A4 input scales [E][2] (w13, w2) for the comparison variant: static
    calibration constants amax / (6 * 448) with amax = 4.5 for x ~ N(0, 1)
    and 0.125 * sqrt(H) for the hidden h (its typical largest magnitude for
    N(0, 0.02) weights); shared experts get 1.0 (unused, they stay W4A16)."""
    E = cfg.num_experts + cfg.shared
    s = np.ones((E, 2), np.float32)
    s[:cfg.num_experts, 0] = np.float32(4.5 / 2688.0)
    s[:cfg.num_experts, 1] = np.float32(0.125 * np.sqrt(cfg.hidden) / 2688.0)
    return s
