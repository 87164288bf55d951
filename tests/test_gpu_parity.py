"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Bars:
* dequantised weights, routing ids, offsets and the permutation: bit-exact;
* routing weights: |gpu - oracle| <= 2e-6 * oracle (FP32 softmax of <= 16
  logits against float64);
* layer output: max|err| <= 2e-2 * RMS(oracle) and mean|err| / mean|oracle|
  <= 5e-3 on the FP32 output; a BF16 output may in addition differ by the
  final rounding, at most 2^-8 of each output (BF16 keeps 8 significant
  bits; for heavy-tailed outputs, such as the 16K-token workload with x20
  outlier weights, rounding the exact result to BF16 alone exceeds 2e-2 *
  RMS); plus the magnitude check the weight-only serving postmortem asks
  for ("GLM-5.3-Flash on Blackwell", The model loaded, served an API, and
  produced garbage: an inverted scale kept cosine 0.996 at 25x the
  magnitude): ||gpu|| / ||oracle|| in [0.99, 1.01] and cosine >= 0.9999.
Every workload is compared on every token: the oracle's layer at 1K and 16K
tokens runs over a process pool (oracle.pool: the oracle's own expert FFNs,
one task per expert) once per session, cached in memory and under
tests/.oracle_cache (git-ignored).  Per routed row, h and y are checked
element-wise against intervals derived from the oracle and the kernels' FP32
arithmetic (tests/intervals.py): every row of the tiny layer and of the
decode workloads, and at 1K and 16K every row of the most-used expert (all
its 128-row m-tiles, the partial last one included) and of the three
least-used experts.
"""
import hashlib
import os
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O
from oracle.pool import moe_forward_pool
from synth import CONFIGS, make_inputs, make_layer_weights, LayerConfig, f32_to_bf16_bits
import nvfp4_weight_only_w4a16_gb300 as P
from tests.intervals import _mats, hidden_bounds_w4a16, down_bounds_w4a16, assert_inside

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
_LAYERS = {}


def _layer(cfg: LayerConfig, max_tokens=None, logits_bf16=False, out_f32=False):
    key = (cfg.num_experts, cfg.hidden, cfg.inter, cfg.outlier_frac, cfg.seed, max_tokens or cfg.tokens,
           cfg.top_k, logits_bf16, out_f32)
    if key not in _LAYERS:
        # keep at most one large layer resident
        if cfg.num_experts * cfg.hidden * cfg.inter > (1 << 26):
            for k in [k for k in _LAYERS if k[0] * k[1] * k[2] > (1 << 26)]:
                _LAYERS.pop(k).close()
        P.build()
        L = P.MoELayer(cfg.num_experts, cfg.hidden, cfg.inter, max_tokens or cfg.tokens, max(cfg.top_k, 1),
                       logits_bf16=logits_bf16, out_f32=out_f32)
        P.upload_layer(L, make_layer_weights(cfg), DEV)
        _LAYERS[key] = L
    return _LAYERS[key]


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


_REF = {}
_CACHE_DIR = os.path.join(os.path.dirname(__file__), ".oracle_cache")


def _source_key(name):
    h = hashlib.sha256(name.encode())
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for d in ("oracle", "synth"):
        for f in sorted(os.listdir(os.path.join(root, d))):
            if f.endswith(".py"):
                with open(os.path.join(root, d, f), "rb") as fh:
                    h.update(fh.read())
    return h.hexdigest()[:16]


def layer_reference(name):
    """The oracle's layer output [T][H] (float64) on every token of a
    workload, via the process pool; cached in memory and on disk."""
    if name in _REF:
        return _REF[name]
    path = os.path.join(_CACHE_DIR, f"{name}-{_source_key(name)}.npy")
    if os.path.exists(path):
        _REF[name] = np.load(path)
        return _REF[name]
    inp = make_inputs(name)
    out = moe_forward_pool(inp.logits, inp.x_bits, inp.weights, inp.config.top_k,
                           num_shared=inp.config.shared)
    os.makedirs(_CACHE_DIR, exist_ok=True)
    np.save(path + ".tmp.npy", out)
    os.replace(path + ".tmp.npy", path)
    _REF[name] = out
    return out


def _forward(L, logits, x_bits, k, path=P.PATH_AUTO):
    L.nvfp4_moe_set_path(path)
    T, H = x_bits.shape
    x = _dev(x_bits.view(np.int16)).view(torch.bfloat16)
    out = torch.empty((T, H), dtype=torch.float32 if L.out_f32 else torch.bfloat16, device=DEV)
    L.nvfp4_moe_forward(_dev(logits), x, k, out)
    torch.cuda.synchronize()
    st, nan = L.nvfp4_moe_get_status()
    assert st == 0, P.STATUS[st]
    L.nvfp4_moe_set_path(P.PATH_AUTO)
    return out.float().cpu().numpy().astype(np.float64)


def assert_layer_close(gpu, ref, bf16_out=True):
    err = np.abs(gpu - ref)
    rms = np.sqrt(np.mean(ref ** 2))
    allow = 2.0 ** -8 * np.abs(gpu) if bf16_out else 0.0
    assert np.all(err <= 2e-2 * rms + allow), (err.max(), rms)
    assert err.mean() / np.abs(ref).mean() <= 5e-3, err.mean() / np.abs(ref).mean()
    ratio = np.linalg.norm(gpu) / np.linalg.norm(ref)
    assert 0.99 <= ratio <= 1.01, ratio
    cos = float(np.sum(gpu * ref) / (np.linalg.norm(gpu) * np.linalg.norm(ref)))
    assert cos >= 0.9999, cos


def _check_route(L, logits, k, E, path=P.PATH_AUTO):
    L.nvfp4_moe_set_path(path)
    T = logits.shape[0]
    ids, w, off, perm = L.nvfp4_moe_debug_route(_dev(logits), T, k)
    torch.cuda.synchronize()
    L.nvfp4_moe_set_path(P.PATH_AUTO)
    r = O.route(logits, k)
    cnt, off_ref, perm_ref = O.permute(r.ids, E)
    assert np.array_equal(ids.cpu().numpy(), r.ids)
    assert np.array_equal(off.cpu().numpy(), off_ref)
    assert np.array_equal(perm.cpu().numpy(), perm_ref)
    wg = w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(wg - r.weights) <= 2e-6 * np.abs(r.weights) + 1e-30), np.abs(wg - r.weights).max()
    return r


# ---------------------------------------------------------------------------
# dequantisation (bit-exact)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("via_bf16", [False, True])
def test_dequant_bit_exact_tiny(via_bf16):
    cfg = CONFIGS["tiny"]
    L = _layer(cfg)
    w = make_layer_weights(cfg)
    I = cfg.inter
    for e in range(cfg.num_experts):
        for which, (q, s, g) in enumerate([(w.w13_q[e, :I], w.w13_s[e, :I], w.gscale[e, 0]),
                                           (w.w13_q[e, I:], w.w13_s[e, I:], w.gscale[e, 1]),
                                           (w.w2_q[e], w.w2_s[e], w.gscale[e, 2])]):
            got = L.nvfp4_moe_debug_dequant(e, which, via_bf16).cpu().numpy()
            ref = O.dequant_scaled_f32(q, s, g)
            assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), (e, which)


def test_dequant_bit_exact_full_layer():
    cfg = CONFIGS["decode_mtp"]
    L = _layer(cfg, max_tokens=1024)
    w = make_layer_weights(cfg)
    I = cfg.inter
    for e in (0, 77, 127):
        for which, (q, s, g) in enumerate([(w.w13_q[e, :I], w.w13_s[e, :I], w.gscale[e, 0]),
                                           (w.w13_q[e, I:], w.w13_s[e, I:], w.gscale[e, 1]),
                                           (w.w2_q[e], w.w2_s[e], w.gscale[e, 2])]):
            for via in (False, True):
                got = L.nvfp4_moe_debug_dequant(e, which, via).cpu().numpy()
                ref = O.dequant_scaled_f32(q, s, g)
                assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), (e, which, via)


def _host_repack_expert(w13_q, w13_s, w2_q, w2_s, H, I):
    """Independent numpy statement of the packed layout for one expert."""
    def pack(q, s, N, K, interleave):
        nch = K // 64
        rows = np.arange(N)
        if interleave:  # packed row 16g+r: gate feature 8g+r (r<8), up feature 8g+r-8
            g, r = rows // 16, rows % 16
            src = np.where(r < 8, 8 * g + r, N // 2 + 8 * g + (r - 8))
        else:
            src = rows
        qq, ss = q[src], s[src]                      # rows in packed order
        # [rb 128][sb 8][r 2][t4 8] x [c][q 4][8 bytes]; segment t = 4 t4 + q of a 16-row
        # sub-block is stored at slot 8 q + (t4 + 2 q) % 8
        qb = qq.reshape(N // 128, 8, 2, 8, nch, 4, 8)
        seg = qb.transpose(0, 4, 1, 3, 5, 2, 6).reshape(N // 128, nch, 8, 32, 16)   # rb, c, sb, t, 16 bytes
        sb_ = ss.reshape(N // 128, 8, 2, 8, nch, 4)
        sseg = sb_.transpose(0, 4, 1, 3, 5, 2).reshape(N // 128, nch, 8, 32, 2)     # rb, c, sb, t, 2 bytes
        t = np.arange(32)
        slot = 8 * (t % 4) + (t // 4 + 2 * (t % 4)) % 8
        nib = np.empty_like(seg)
        nib[:, :, :, slot] = seg
        sc = np.empty_like(sseg)
        sc[:, :, :, slot] = sseg
        # one tile per (rb, c): its 4096 code bytes, then its 512 scale bytes
        tiles = np.concatenate([nib.reshape(N // 128, nch, 4096), sc.reshape(N // 128, nch, 512)], axis=2)
        return tiles.reshape(-1)
    return np.concatenate([pack(w13_q, w13_s, 2 * I, H, True), pack(w2_q, w2_s, H, I, False)])


@pytest.mark.parametrize("name,experts", [("tiny", None), ("decode_mtp", (0, 64, 127))])
def test_packed_blob_matches_host_repack(name, experts):
    cfg = CONFIGS[name]
    L = _layer(cfg, max_tokens=1024 if cfg.num_experts == 128 else None)
    w = make_layer_weights(cfg)
    blob = L.nvfp4_moe_debug_packed_blob().cpu().numpy()
    H, I = cfg.hidden, cfg.inter
    stride = 3 * H * I * 9 // 16
    for e in (range(cfg.num_experts) if experts is None else experts):
        ref = _host_repack_expert(w.w13_q[e], w.w13_s[e], w.w2_q[e], w.w2_s[e], H, I)
        assert np.array_equal(blob[e * stride:(e + 1) * stride], ref), e


# ---------------------------------------------------------------------------
# routing and permutation (bit-exact ids/offsets/perm)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "decode_mtp", "decode_c16", "prefill_1k"])
def test_route_bit_exact(name):
    inp = make_inputs(name)
    cfg = inp.config
    L = _layer(cfg, max_tokens=1024 if cfg.num_experts == 128 else None)
    _check_route(L, inp.logits, cfg.top_k, cfg.num_experts)
    if cfg.tokens <= 16:  # the prefill routing kernels must agree too
        _check_route(L, inp.logits, cfg.top_k, cfg.num_experts, P.PATH_PREFILL)


def test_route_edge_cases():
    cfg = LayerConfig("edge", 40, 128, 128, 3, 48)
    L = _layer(cfg)
    rng = np.random.default_rng(1)
    logits = np.round(rng.standard_normal((48, 40)) * 2).astype(np.float32) / 2  # many ties
    logits[0, :] = 0.5                          # all equal -> ids 0,1,2, weights 1/3
    logits[1, 5] = np.nan
    logits[2, :] = -np.inf
    logits[3, 7] = np.inf
    logits[4, [3, 9]] = np.inf
    logits[5, :] = -1.0                         # -0 and +0 compare equal: lower index first
    logits[5, 6] = 0.0
    logits[5, 1] = -0.0
    for path in (P.PATH_PREFILL,):
        r = _check_route(L, logits, 3, 40, path)
    assert r.ids[0].tolist() == [0, 1, 2]
    assert r.ids[5].tolist()[:2] == [1, 6]
    for k in (1, 2, 3):
        _check_route(L, logits, k, 40, P.PATH_PREFILL)
        _check_route(L, logits[:16], k, 40, P.PATH_DECODE)
    # NaN logits are counted in the status word
    L.nvfp4_moe_get_status()
    L.nvfp4_moe_debug_route(_dev(logits), 48, 3)
    st, nan = L.nvfp4_moe_get_status()
    assert st == 0 and nan == 1


def test_route_full_size_zipf():
    inp = make_inputs("prefill_16k")
    cfg = inp.config
    L = _layer(cfg)
    r = _check_route(L, inp.logits, cfg.top_k, cfg.num_experts)
    counts = np.bincount(r.ids.reshape(-1), minlength=cfg.num_experts)
    assert counts.max() > 8 * counts.mean()  # the skew is really there


# ---------------------------------------------------------------------------
# the layer
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("path", [P.PATH_DECODE, P.PATH_PREFILL])
def test_forward_tiny(path):
    inp = make_inputs("tiny")
    cfg = inp.config
    L = _layer(cfg)
    gpu = _forward(L, inp.logits, inp.x_bits, cfg.top_k, path)
    ref = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k)
    assert_layer_close(gpu, ref)


def check_rows(L, inp, rows, k=None):
    """h and y of routed rows (positions, expert-major) against the interval
    checks: h inside the BF16 interval of the oracle's expert, y inside the
    down projection of the GPU's own h."""
    cfg = inp.config
    k = k or cfg.top_k
    T = cfg.tokens
    R = T * (k + cfg.shared)
    hid, y = L.nvfp4_moe_debug_intermediates(R)
    rows = np.asarray(rows, dtype=np.int64)
    sel = torch.from_numpy(rows).to(hid.device)
    hid = hid[sel].float().cpu().numpy().astype(np.float64)
    y = y[sel].cpu().numpy().astype(np.float64)
    r = O.route(inp.logits, k)
    ids = r.ids
    if cfg.shared:
        ids = np.concatenate([ids, np.full((T, 1), cfg.num_experts, np.int32)], axis=1)
    _, _, perm = O.permute(ids, cfg.num_experts + cfg.shared)
    flat = perm[rows]
    tok, slot = flat // ids.shape[1], flat % ids.shape[1]
    ex = ids[tok, slot]
    x = O.bf16_bits_to_f64(inp.x_bits)
    for e in np.unique(ex):
        m = ex == e
        mats = _mats(inp.weights, int(e))
        hl, hh = hidden_bounds_w4a16(mats, x[tok[m]])
        assert_inside(hid[m], hl, hh, ("h", int(e)))
        yl, yh = down_bounds_w4a16(mats, hid[m])
        assert_inside(y[m], yl, yh, ("y", int(e)))


@pytest.mark.parametrize("path", [P.PATH_DECODE, P.PATH_PREFILL])
def test_intermediates_tiny(path):
    inp = make_inputs("tiny")
    cfg = inp.config
    L = _layer(cfg)
    _forward(L, inp.logits, inp.x_bits, cfg.top_k, path)
    check_rows(L, inp, range(cfg.tokens * cfg.top_k))


@pytest.mark.parametrize("out_f32", [True, False])
@pytest.mark.parametrize("name", ["decode_mtp", "decode_c16"])
def test_forward_decode_full_size(name, out_f32):
    inp = make_inputs(name)
    cfg = inp.config
    L = _layer(cfg, max_tokens=1024, out_f32=out_f32)
    gpu = _forward(L, inp.logits, inp.x_bits, cfg.top_k)
    ref = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k)
    assert_layer_close(gpu, ref, bf16_out=not out_f32)
    if out_f32:
        check_rows(L, inp, range(cfg.tokens * cfg.top_k))


def _edge_rows(cfg, logits, k):
    """Positions of every row of the most-used expert and of the three
    least-used (touched) experts."""
    r = O.route(logits, k)
    cnt, off, _ = O.permute(r.ids, cfg.num_experts)
    used = np.nonzero(cnt)[0]
    picks = [int(used[np.argmax(cnt[used])])] + [int(e) for e in used[np.argsort(cnt[used], kind="stable")[:3]]]
    rows = np.concatenate([np.arange(off[e], off[e + 1]) for e in picks])
    return rows, picks, cnt


@pytest.mark.parametrize("out_f32", [True, False])
@pytest.mark.parametrize("name", ["prefill_1k", "prefill_16k"])
def test_forward_prefill_every_token(name, out_f32):
    inp = make_inputs(name)
    cfg = inp.config
    L = _layer(cfg, max_tokens=1024 if cfg.num_experts == 128 else None, out_f32=out_f32)
    gpu = _forward(L, inp.logits, inp.x_bits, cfg.top_k)
    assert np.all(np.isfinite(gpu))
    assert_layer_close(gpu, layer_reference(name), bf16_out=not out_f32)
    if out_f32:
        rows, picks, cnt = _edge_rows(cfg, inp.logits, cfg.top_k)
        assert cnt[picks[0]] > 128 and cnt[picks[0]] % 128 != 0   # several m-tiles and a partial last one
        check_rows(L, inp, rows)


# The decode kernel's code paths change with the token count: up to 4 tokens the signal warp
# that completes an output slice combines it, above that every consumer warp takes (slice,
# token) tasks; up to 8 tokens one 8-column MMA group, above that two; T consumer warps route
# and T convert x rows.  Every T of the decode range, on the tiny layer (small stages) and on
# a layer with the full H and I (8-chunk stages) but 8 experts, so the oracle stays quick.
DECODE_FULL_DIMS = LayerConfig("decode_full_dims", 8, 4096, 1536, 4, 16)


@pytest.mark.parametrize("T", range(1, 17))
def test_decode_every_token_count(T):
    for base in (CONFIGS["tiny"], DECODE_FULL_DIMS):
        cfg = base.with_tokens(T)
        inp = make_inputs(cfg)
        L = _layer(base, max_tokens=16)
        gpu = _forward(L, inp.logits, inp.x_bits, cfg.top_k, P.PATH_DECODE)
        ref = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k)
        assert_layer_close(gpu, ref)


@pytest.mark.parametrize("T,path", [(1, P.PATH_DECODE), (1, P.PATH_PREFILL), (37, P.PATH_PREFILL),
                                    (300, P.PATH_PREFILL), (16, P.PATH_DECODE)])
def test_forward_ragged_and_degenerate(T, path):
    cfg = CONFIGS["tiny"].with_tokens(T)
    inp = make_inputs(cfg)
    L = _layer(CONFIGS["tiny"], max_tokens=512)
    gpu = _forward(L, inp.logits, inp.x_bits, cfg.top_k, path)
    ref = O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k)
    assert_layer_close(gpu, ref)


@pytest.mark.parametrize("path", [P.PATH_DECODE, P.PATH_PREFILL])
def test_all_tokens_to_one_expert(path):
    T = 16 if path == P.PATH_DECODE else 300   # 300 rows of one expert: three 128-row m-tiles, the last partial
    cfg = CONFIGS["tiny"].with_tokens(T)
    inp = make_inputs(cfg)
    logits = inp.logits.copy()
    logits[:, 3] += 100.0
    L = _layer(CONFIGS["tiny"], max_tokens=512)
    gpu = _forward(L, logits, inp.x_bits, cfg.top_k, path)
    ref = O.moe_forward(logits, inp.x_bits, inp.weights, cfg.top_k)
    assert_layer_close(gpu, ref)


def test_top1_is_single_expert_ffn():
    cfg = CONFIGS["tiny"]
    inp = make_inputs(cfg)
    L = _layer(cfg)
    for path in (P.PATH_DECODE, P.PATH_PREFILL):
        gpu = _forward(L, inp.logits, inp.x_bits, 1, path)
        x = O.bf16_bits_to_f64(inp.x_bits)
        ref = np.stack([O.expert_ffn(inp.weights, int(np.argmax(inp.logits[t])), x[t:t + 1])[0]
                        for t in range(cfg.tokens)])
        assert_layer_close(gpu, ref)


def test_bf16_logits():
    cfg = CONFIGS["tiny"]
    inp = make_inputs(cfg)
    L = _layer(cfg, logits_bf16=True)
    lb = f32_to_bf16_bits(inp.logits)
    lf = O.bf16_bits_to_f64(lb).astype(np.float32)
    x = _dev(inp.x_bits.view(np.int16)).view(torch.bfloat16)
    out = torch.empty((cfg.tokens, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    L.nvfp4_moe_forward(_dev(lb.view(np.int16)), x, cfg.top_k, out)
    torch.cuda.synchronize()
    ref = O.moe_forward(lf, inp.x_bits, inp.weights, cfg.top_k)
    assert_layer_close(out.float().cpu().numpy().astype(np.float64), ref)


# ---------------------------------------------------------------------------
# errors and the bounded-wait status
# ---------------------------------------------------------------------------

def test_errors_are_reported():
    L = P.MoELayer(8, 256, 512, 16, 2)
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(x)
    logits = torch.zeros((4, 8), dtype=torch.float32, device=DEV)
    with pytest.raises(P.Nvfp4MoeError) as ei:
        L.nvfp4_moe_forward(logits, x, 2, out)
    assert ei.value.status == P.STATUS_CODE["NVFP4_MOE_ERR_NOT_PACKED"]
    w = make_layer_weights(CONFIGS["tiny"])
    bad = w.gscale.copy()
    bad[3, 1] = 0.0
    with pytest.raises(P.Nvfp4MoeError) as ei:
        L.nvfp4_moe_pack(_dev(w.w13_q), _dev(w.w13_s), _dev(w.w2_q), _dev(w.w2_s), _dev(bad))
    assert ei.value.status == P.STATUS_CODE["NVFP4_MOE_ERR_BAD_SCALE"]
    bad[3, 1] = np.nan
    with pytest.raises(P.Nvfp4MoeError):
        L.nvfp4_moe_pack(_dev(w.w13_q), _dev(w.w13_s), _dev(w.w2_q), _dev(w.w2_s), _dev(bad))
    P.upload_layer(L, w, DEV)
    big = torch.zeros((17, 256), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(P.Nvfp4MoeError) as ei:
        L.nvfp4_moe_forward(torch.zeros((17, 8), device=DEV), big, 2, torch.empty_like(big))
    assert ei.value.status == P.STATUS_CODE["NVFP4_MOE_ERR_UNSUPPORTED_SHAPE"]
    with pytest.raises(P.Nvfp4MoeError) as ei:
        L.nvfp4_moe_forward(logits, x, 3, out)
    assert ei.value.status == P.STATUS_CODE["NVFP4_MOE_ERR_UNSUPPORTED_SHAPE"]
    L.close()


@pytest.mark.parametrize("path", [P.PATH_PREFILL, P.PATH_DECODE])
def test_bounded_wait_reports_timeout(path):
    cfg = CONFIGS["tiny"]
    inp = make_inputs(cfg)
    L = P.MoELayer(cfg.num_experts, cfg.hidden, cfg.inter, 64, cfg.top_k)
    P.upload_layer(L, make_layer_weights(cfg), DEV)
    L.nvfp4_moe_set_path(path)
    L.nvfp4_moe_debug_set_fault(1)
    x = _dev(inp.x_bits.view(np.int16)).view(torch.bfloat16)
    out = torch.empty((cfg.tokens, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    L.nvfp4_moe_forward(_dev(inp.logits), x, cfg.top_k, out)
    st, _ = L.nvfp4_moe_get_status()
    assert st == P.STATUS_CODE["NVFP4_MOE_ERR_TIMEOUT"]
    # the context is still usable and the next forward is correct
    L.nvfp4_moe_debug_set_fault(0)
    gpu = _forward(L, inp.logits, inp.x_bits, cfg.top_k, path)
    assert_layer_close(gpu, O.moe_forward(inp.logits, inp.x_bits, inp.weights, cfg.top_k))
    L.close()
