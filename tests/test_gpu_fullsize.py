"""Parity at full size: the 0.5B prompt (512 tokens), the 1.5B prompt (2048
tokens), the 7B prompt (4096 tokens), the 1.5B append (1024 tokens after 3072
cached ones), the Qwen3 0.6B prompt and the tiny model, run by the CUDA
library exactly as it is timed, checked stage by stage on sampled rows.

A full oracle forward at these sizes takes the CPU many minutes, and over 28
layers any implementation that is not bit-identical to it drifts away from it
(each on-the-fly Q8_0 quantization turns a relative input difference d into
about 0.13*sqrt(d)).  So the check is teacher-forced: the library captures one
layer's intermediates from the real forward, and the oracle recomputes every
step of that layer (Qwen2 block: "09 · Prefill", section 3) from the GPU's own
input to the step, on sampled rows that span the first, interior and ragged
last row tiles.  Integer decisions (Q8_0 codes and scales of the norms, the
K/V rows written) must be bit-identical; sums must lie within the f32
rounding bound of the block sums; the attention and SwiGLU outputs within the
bound of their f32 arithmetic, with code flips only next to a rounding
boundary.  The last layer is teacher-forced down to the last-token logits.
"""
import numpy as np
import pytest

import synth
from helpers import U, check_logits, q8_sum_bound
from stagecheck import LayerWeights, check_row_layer
from helpers import check_q8_requant as _check_quantized
from helpers import check_q8_sum as _check_sum

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

@pytest.fixture(scope="module")
def qp():
    import quantized_transformer_prefill_gb300 as qp
    qp.lib()
    return qp


_MODELS = {}


def _gpu_model(qp, cfg):
    # one model at a time on the device: free the previous one
    if cfg.name not in _MODELS:
        for m in _MODELS.values():
            m.free()
        _MODELS.clear()
        from helpers import gpu_model
        _MODELS[cfg.name] = gpu_model(cfg)
    return _MODELS[cfg.name]


@pytest.fixture(scope="module", autouse=True)
def _release_models():
    yield
    for m in _MODELS.values():
        m.free()
    _MODELS.clear()


def _sample_rows(nt, k, seed):
    fixed = [0, 1, 2, 127, 128, 129, nt // 2, nt - 130, nt - 129, nt - 128, nt - 2, nt - 1]
    rng = np.random.default_rng(seed)
    extra = rng.choice(nt, size=max(0, k - len(fixed)), replace=False)
    return np.unique(np.clip(np.concatenate([fixed, extra]), 0, nt - 1)).astype(np.int64)


def _codes(g, name, nt, width):
    buf = np.empty((nt, width), np.float16)
    g.debug_read(name, buf)
    q = buf.astype(np.float32)
    assert np.array_equal(q, np.round(q)) and np.abs(q).max() <= 127
    return q.astype(np.int8)


def _scales(g, name, nb, ntp, rows):
    buf = np.empty((nb, ntp), np.float32)
    g.debug_read(name, buf)
    s = buf[:, rows].T.astype(np.float32)
    h = s.astype(np.float16)
    assert np.array_equal(h.astype(np.float32), s), "scale not an fp16 value"
    return h.view(np.uint16)


def _f32(g, name, nt, width):
    buf = np.empty((nt, width), np.float32)
    return g.debug_read(name, buf)


def _kv_rows(kv, layer, which, rows_pos):
    return np.stack([kv.read(layer, which, int(p), 1)[0] for p in rows_pos])


def _check_layer(oracle_mod, g, kv, cfg, layer, pos, rows, tail0=0):
    """Teacher-forced check of one layer on rows `rows`.  tail0 > 0: the last
    layer of a call that keeps the rows tail0.. past attention (their
    attention, FFN and SwiGLU captures start at row 0)."""
    nt = len(pos)
    ntp = (nt + 127) // 128 * 128
    H, hd, nh, nkv = cfg.n_embd, cfg.head_dim, cfg.n_head, cfg.n_head_kv
    q, kvw = nh * hd, nkv * hd
    nbH, nbq, nbF = (H + 31) // 32, (q + 31) // 32, (cfg.n_ff + 31) // 32
    Wt = LayerWeights(oracle_mod, cfg, layer)
    p = pos[rows]

    h_in = _f32(g, "h_in", nt, H)[rows]
    xq = _codes(g, "x_codes", nt, nbH * 32)[rows]
    xd = _scales(g, "x_scales", nbH, ntp, rows)
    oq, od = oracle_mod.q8_quantize(oracle_mod.rmsnorm(h_in, Wt.f32["attn_norm.weight"],
                                                       cfg.rms_eps))
    assert np.array_equal(xd, od) and np.array_equal(xq, oq), "attn_norm Q8_0 differs"

    qkv = _f32(g, "qkv", nt, q + 2 * kvw)[rows]
    _check_sum(oracle_mod, qkv, xq, xd, *Wt.q8["qkv"], H)
    full = Wt.qk_normed(oracle_mod, (qkv + Wt.bias).astype(np.float32))
    cos_t, sin_t = oracle_mod.rope_table(int(pos.max()) + 1, hd, cfg.rope_theta)
    want_q = oracle_mod.rope(full[:, :q], p, nh, hd, cos_t, sin_t)
    want_k = oracle_mod.rope(full[:, q:q + kvw], p, nkv, hd, cos_t, sin_t)
    assert np.array_equal(_f32(g, "qrot", nt, q)[rows], want_q), "rotated Q differs"
    assert np.array_equal(_kv_rows(kv, layer, 0, p), want_k), "K rows differ"
    assert np.array_equal(_kv_rows(kv, layer, 1, p), full[:, q + kvw:]), "V rows differ"

    # attention over the cache the GPU wrote (rows 0..max position)
    nctx = int(p.max()) + 1
    K = kv.read(layer, 0, 0, nctx)
    V = kv.read(layer, 1, 0, nctx)
    att_ref = oracle_mod.attention(want_q, p, K, V, nh, nkv, hd)
    att = _f32(g, "att", nt, q)[rows]
    err = np.abs(att - att_ref).max()
    assert err <= 2e-5 * max(1.0, np.abs(att_ref).max()), err
    aq = _codes(g, "att_codes", nt, nbq * 32)[rows - tail0]
    ad = _scales(g, "att_scales", nbq, ntp, rows - tail0)
    gq, gd = oracle_mod.q8_quantize(att)
    assert np.array_equal(ad, gd) and np.array_equal(aq, gq), "attention Q8_0 differs"

    h_mid = _f32(g, "h_mid", nt, H)[rows]
    _check_sum(oracle_mod, h_mid, aq, ad, *Wt.q8["attn_output.weight"], q, base=h_in)

    fq = _codes(g, "f_codes", nt, nbH * 32)[rows - tail0]
    fd = _scales(g, "f_scales", nbH, ntp, rows - tail0)
    oq, od = oracle_mod.q8_quantize(oracle_mod.rmsnorm(h_mid, Wt.f32["ffn_norm.weight"],
                                                       cfg.rms_eps))
    assert np.array_equal(fd, od) and np.array_equal(fq, oq), "ffn_norm Q8_0 differs"

    gate = oracle_mod.matmul_q8(fq, fd, *Wt.q8["ffn_gate.weight"], H).astype(np.float64)
    up = oracle_mod.matmul_q8(fq, fd, *Wt.q8["ffn_up.weight"], H).astype(np.float64)
    s_ref = oracle_mod.swiglu(gate, up)
    sq = _codes(g, "s_codes", nt, nbF * 32)[rows - tail0]
    sd = _scales(g, "s_scales", nbF, ntp, rows - tail0)
    # the GPU's gate/up are f32 block sums (error dg, du within their bounds);
    # silu' <= 1.1 and |silu(g)| <= |g| + 0.28 carry them into s = silu(g) u,
    # plus the f32 rounding of silu and of the product
    dg, du = (q8_sum_bound(oracle_mod, fq, fd, *Wt.q8[f"ffn_{x}.weight"], H) for x in ("gate", "up"))
    slack = 1.1 * np.abs(up) * dg + (np.abs(gate) + 0.28) * du + 16 * U * np.abs(s_ref)
    _check_quantized(oracle_mod, sq, sd, s_ref, slack)
    # the epilogue's own f32 values: within the same bound of the oracle's s,
    # and their Q8_0 (amax over the block, fp16 scale, rounded codes) is the
    # oracle's quantization of them, bit for bit
    s_gpu = _f32(g, "s_f32", nt, nbF * 32)[rows - tail0]
    assert not np.any(s_gpu[:, cfg.n_ff:]), "SwiGLU padding columns not zero"
    assert np.all(np.abs(s_gpu[:, :cfg.n_ff] - s_ref) <= slack), "SwiGLU f32 outside its bound"
    gq, gd = oracle_mod.q8_quantize(s_gpu[:, :cfg.n_ff])
    assert np.array_equal(sd, gd), "SwiGLU Q8_0 scales differ from the oracle's"
    assert np.array_equal(sq, gq), "SwiGLU Q8_0 codes differ from the oracle's"

    h_out = _f32(g, "h_out", nt, H)[rows]
    _check_sum(oracle_mod, h_out, sq, sd, *Wt.q8["ffn_down.weight"], cfg.n_ff, base=h_mid)
    return h_out


def _check_last_layer(oracle_mod, g, kv, cfg, pos, rows, logits):
    """Teacher-forced last layer: x codes, Q|K|V and the K/V rows of sampled
    rows, then the last token stage by stage through attention, FFN, output
    norm and head."""
    L = cfg.n_layer - 1
    nt = len(pos)
    ntp = (nt + 127) // 128 * 128
    H, hd, nh, nkv = cfg.n_embd, cfg.head_dim, cfg.n_head, cfg.n_head_kv
    q, kvw = nh * hd, nkv * hd
    nbH = (H + 31) // 32
    Wt = LayerWeights(oracle_mod, cfg, L)
    rows = np.union1d(rows, [nt - 1])
    p = pos[rows]
    h_in = _f32(g, "h_in", nt, H)[rows]
    xq = _codes(g, "x_codes", nt, nbH * 32)[rows]
    xd = _scales(g, "x_scales", nbH, ntp, rows)
    oq, od = oracle_mod.q8_quantize(oracle_mod.rmsnorm(h_in, Wt.f32["attn_norm.weight"],
                                                       cfg.rms_eps))
    assert np.array_equal(xd, od) and np.array_equal(xq, oq)
    qkv = _f32(g, "qkv", nt, q + 2 * kvw)[rows]
    _check_sum(oracle_mod, qkv, xq, xd, *Wt.q8["qkv"], H)
    full = Wt.qk_normed(oracle_mod, (qkv + Wt.bias).astype(np.float32))
    cos_t, sin_t = oracle_mod.rope_table(int(pos.max()) + 1, hd, cfg.rope_theta)
    want_k = oracle_mod.rope(full[:, q:q + kvw], p, nkv, hd, cos_t, sin_t)
    assert np.array_equal(_kv_rows(kv, L, 0, p), want_k)
    assert np.array_equal(_kv_rows(kv, L, 1, p), full[:, q + kvw:])

    # the last token, stage by stage from the GPU's own input to each stage,
    # then the logits from the GPU's output row of the layer
    t = nt - 1
    h_last = check_row_layer(oracle_mod, g, kv, cfg, Wt, L, int(pos[t]), h_in=h_in[-1:],
                             qkv=qkv[-1:], x_captured=False)
    specs = {sp.name: sp for sp in synth.tensor_specs(cfg)}
    yq, yd = oracle_mod.q8_quantize(
        oracle_mod.rmsnorm(h_last, synth.tensor_data(specs["output_norm.weight"]), cfg.rms_eps))
    head = specs["token_embd.weight" if cfg.tied else "output.weight"]
    wq, wd = oracle_mod.q8_quantize(synth.tensor_data(head))
    want = oracle_mod.matmul_q8(yq, yd, wq, wd, H)[0]
    check_logits(logits, want)


def _run(qp, oracle_mod, wl, layer_mid, n_rows, seed):
    cfg = wl.model
    g = _gpu_model(qp, cfg)
    ids, pos = wl.ids(), wl.positions()

    def fresh_cache():
        kv = g.kv(wl.n_ctx)
        if wl.prefill_tokens:
            g.prefill(kv, wl.prefill_ids(), np.arange(wl.prefill_tokens, dtype=np.int32))
        return kv

    rows = _sample_rows(wl.n_tokens, n_rows, seed)
    try:
        kv = fresh_cache()
        g.debug_layer(layer_mid)
        g.prefill(kv, ids, pos)
        _check_layer(oracle_mod, g, kv, cfg, layer_mid, pos, rows)
        kv.free()
        kv = fresh_cache()
        g.debug_layer(cfg.n_layer - 1)
        logits = g.prefill(kv, ids, pos)
        _check_last_layer(oracle_mod, g, kv, cfg, pos, rows, logits)
        kv.free()
    finally:
        g.debug_layer(-1)
    # the captured graph (the timed launch sequence) equals the eager forward
    kv = fresh_cache()
    assert np.array_equal(g.prefill(kv, ids, pos), logits), "graph replay differs"
    kv.free()


def test_tiny_32(qp, oracle_mod):
    """The tiny model (one ragged 32-row tile, partial Q8_0 blocks of the
    688-wide FFN), both layers."""
    _run(qp, oracle_mod, synth.WORKLOADS["tiny-32"], 0, 32, 5)


def test_qwen2_0_5b_512(qp, oracle_mod):
    """The benched workload: 24 layers of H 896, 14 query heads of 64 over 2
    KV heads (7 per group), tied lm_head over 151936 rows; a middle layer and
    the last layer down to the logits."""
    _run(qp, oracle_mod, synth.WORKLOADS["qwen2-0.5b-512"], 11, 40, 6)


def test_qwen2_1_5b_2048(qp, oracle_mod):
    _run(qp, oracle_mod, synth.WORKLOADS["qwen2-1.5b-2048"], 13, 40, 1)


def test_qwen2_1_5b_append_1024(qp, oracle_mod):
    """1024 new tokens at positions 3072..4095 attend over 3072 cached rows
    written by an earlier call (the split-KV attention path)."""
    _run(qp, oracle_mod, synth.WORKLOADS["qwen2-1.5b-append-1024"], 5, 40, 2)


def test_qwen2_7b_4096(qp, oracle_mod):
    _run(qp, oracle_mod, synth.WORKLOADS["qwen2-7b-4096"], 20, 32, 3)


def test_qwen3_0_6b_512(qp, oracle_mod):
    """The Qwen3 variant: per-head QK RMSNorm before RoPE, no Q/K/V bias,
    16 query / 8 KV heads of 128."""
    _run(qp, oracle_mod, synth.WORKLOADS["qwen3-0.6b-512"], 9, 40, 4)
