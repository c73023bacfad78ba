"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something it does not compute itself: a
library routine (numpy), a closed form, an invariant the pages state, brute
force on tiny inputs, or a size the pages print.  They are chosen so that a
plausible slip (a dropped term, a swapped pair, a wrong sign, a transposed
operand, a wrong head mapping) fails at least one of them.
"""
import math
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _ulp32(x):
    return np.spacing(np.abs(np.asarray(x, np.float32))).astype(np.float64)


# ---------------------------------------------------------------- fp16 scale

def test_fp16_conversion_matches_numpy(oracle_mod):
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.normal(0, 1, 2000), rng.normal(0, 1e-5, 2000),  # subnormal range
        np.ldexp(1.0 + np.arange(0, 2048) / 2048.0, -20),   # exact ties at several exponents
        [0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e9, 2.0 ** -25, 2.0 ** -24, 3 * 2.0 ** -26],
    ]).astype(np.float32)
    for v in vals:
        got = oracle_mod.f32_to_f16_bits(float(v))
        want = int(np.float32(v).astype(np.float16).view(np.uint16))
        assert got == want, (v, hex(got), hex(want))
    for h in list(range(0, 0x7C00, 7)) + [0x8001, 0x83FF, 0xFBFF]:
        assert oracle_mod.f16_bits_to_f32(h) == float(np.uint16(h).view(np.float16))


# ---------------------------------------------------------------- Q8_0 codec

def _q8_cases():
    rng = np.random.default_rng(2)
    rows = [rng.normal(0, 1, 64), rng.normal(0, 0.02, 64), rng.standard_cauchy(64),
            np.concatenate([np.zeros(32), rng.normal(0, 3, 32)]),
            rng.uniform(-1e-3, 1e-3, 64)]
    return np.array(rows, np.float32)


def test_q8_nearest_code_brute_force(oracle_mod):
    """Every code is (up to the f32 reciprocal) the nearest of all 255 codes."""
    x = _q8_cases()
    q, d = oracle_mod.q8_quantize(x)
    codes = np.arange(-127, 128, dtype=np.float64)
    for r in range(x.shape[0]):
        for b in range(2):
            blk = x[r, 32 * b:32 * b + 32].astype(np.float64)
            amax = np.max(np.abs(blk))
            dd = float(np.float32(np.float32(amax) / np.float32(127.0)))
            if dd == 0.0:
                assert np.all(q[r, 32 * b:32 * b + 32] == 0) and d[r, b] == 0
                continue
            err = np.abs(blk[:, None] - dd * codes[None, :])
            best = err.min(axis=1)
            mine = np.abs(blk - dd * q[r, 32 * b:32 * b + 32].astype(np.float64))
            assert np.all(mine <= best + dd * 2.0 ** -20), (r, b)
            # the element of largest magnitude maps to +-127
            k = int(np.argmax(np.abs(blk)))
            assert abs(int(q[r, 32 * b + k])) == 127
            # stored scale = round-to-nearest-even fp16 of amax/127 (numpy routine)
            assert d[r, b] == np.float16(np.float32(dd)).view(np.uint16)


def test_q8_roundtrip_within_half_scale(oracle_mod):
    """North-star pin: the Q8_0 round trip stays within scale/2 per element,
    the scale read as the fp16-rounded one (its rounding adds 127*|d - d16|)."""
    rng = np.random.default_rng(3)
    x = (rng.normal(0, 1, (50, 96)) * rng.uniform(1e-3, 1e2, (50, 1))).astype(np.float32)
    q, d = oracle_mod.q8_quantize(x)
    xr = oracle_mod.q8_dequantize(q, d, 96)
    for b in range(3):
        blk = x[:, 32 * b:32 * b + 32].astype(np.float64)
        dd = (np.max(np.abs(blk), axis=1).astype(np.float32) / np.float32(127)).astype(np.float64)
        d16 = d[:, b].view(np.float16).astype(np.float64)
        bound = dd / 2 + 127 * np.abs(dd - d16) + 4 * _ulp32(blk).max(axis=1)
        err = np.abs(blk - xr[:, 32 * b:32 * b + 32]).max(axis=1)
        assert np.all(err <= bound)


def test_q8_special_cases(oracle_mod):
    # amax 127 -> d = 1 exactly, id = 1: ties round away from zero
    x = np.zeros(32, np.float32)
    x[0], x[1], x[2], x[3], x[4] = 127.0, 2.5, -2.5, 0.5, -126.5
    q, d = oracle_mod.q8_quantize(x)
    assert list(q[0, :5]) == [127, 3, -3, 1, -127]
    assert d[0, 0] == np.float16(1.0).view(np.uint16)
    # sign symmetry
    y = _q8_cases()
    q1, d1 = oracle_mod.q8_quantize(y)
    q2, d2 = oracle_mod.q8_quantize(-y)
    assert np.array_equal(q1, -q2) and np.array_equal(d1, d2)
    # a partial final block (length not a multiple of 32) equals the zero-padded row
    z = np.random.default_rng(4).normal(0, 1, 48).astype(np.float32)
    qa, da = oracle_mod.q8_quantize(z)
    qb, db = oracle_mod.q8_quantize(np.concatenate([z, np.zeros(16, np.float32)]))
    assert np.array_equal(qa, qb) and np.array_equal(da, db)
    assert np.all(qa[0, 48:] == 0)


# ---------------------------------------------------------------- block dots / matmul

def test_block_dots_brute_force(oracle_mod):
    rng = np.random.default_rng(5)
    qa = rng.integers(-127, 128, (3, 96), dtype=np.int64).astype(np.int8)
    qw = rng.integers(-127, 128, (5, 96), dtype=np.int64).astype(np.int8)
    got = oracle_mod.block_dots(qa, qw)
    for m in range(3):
        for n in range(5):
            for b in range(3):
                s = sum(int(qa[m, 32 * b + i]) * int(qw[n, 32 * b + i]) for i in range(32))
                assert got[m, n, b] == s
    # extremes fit in int32 and are exact: 32 * 127 * 127
    full = np.full((1, 32), 127, np.int8)
    assert oracle_mod.block_dots(full, -full)[0, 0, 0] == -32 * 127 * 127


def test_matmul_equals_dequantized_float64_gemm(oracle_mod):
    rng = np.random.default_rng(6)
    M, N, K = 7, 11, 80  # K not a multiple of 32: partial final block
    x = rng.normal(0, 1, (M, K)).astype(np.float32)
    w = rng.normal(0, 0.02, (N, K)).astype(np.float32)
    bias = rng.normal(0, 0.02, N).astype(np.float32)
    xq, xd = oracle_mod.q8_quantize(x)
    wq, wd = oracle_mod.q8_quantize(w)
    y = oracle_mod.matmul_q8(xq, xd, wq, wd, K, bias)
    xr = oracle_mod.q8_dequantize(xq, xd, K).astype(np.float64)
    wr = oracle_mod.q8_dequantize(wq, wd, K).astype(np.float64)
    ref = (xr @ wr.T).astype(np.float32)  # closed form: numpy float64 GEMM
    ref = (ref + bias).astype(np.float32)
    assert np.all(np.abs(y.astype(np.float64) - ref) <= 2 * _ulp32(ref) + 1e-12)
    # a transposed weight operand would not match
    ref_t = (xr @ wr[::-1].T).astype(np.float32) + bias
    assert not np.allclose(y, ref_t, rtol=1e-3)


# ---------------------------------------------------------------- rmsnorm / swiglu

def test_rmsnorm_closed_form_and_scale_invariance(oracle_mod):
    rng = np.random.default_rng(7)
    x = rng.normal(0, 0.3, (5, 96)).astype(np.float32)
    w = (1 + rng.normal(0, 0.01, 96)).astype(np.float32)
    y = oracle_mod.rmsnorm(x, w, 1e-6)
    xd = x.astype(np.float64)
    ref = xd / np.sqrt(np.mean(xd * xd, axis=1, keepdims=True) + 1e-6) * w
    assert np.allclose(y, ref, rtol=3e-7, atol=0)
    y2 = oracle_mod.rmsnorm(x * np.float32(64.0), w, 1e-6)  # eps negligible at this scale
    assert np.allclose(y, y2, rtol=1e-5)


def test_swiglu_closed_form(oracle_mod):
    rng = np.random.default_rng(8)
    g = rng.normal(0, 2, 500).astype(np.float32)
    u = rng.normal(0, 2, 500).astype(np.float32)
    s = oracle_mod.swiglu(g, u)
    gd = g.astype(np.float64)
    ref = gd * (1.0 / (1.0 + np.exp(-gd))) * u
    assert np.allclose(s, ref, rtol=2e-7, atol=1e-30)
    assert oracle_mod.swiglu(np.zeros(3, np.float32), np.ones(3, np.float32)).tolist() == [0, 0, 0]


# ---------------------------------------------------------------- RoPE

def test_rope_table_matches_numpy(oracle_mod):
    c, s = oracle_mod.rope_table(64, 64, 1.0e6)
    i = np.arange(32, dtype=np.float64)
    ang = np.arange(64, dtype=np.float64)[:, None] * (1.0e6 ** (-2.0 * i / 64))[None, :]
    assert np.all(np.abs(c - np.cos(ang)) <= _ulp32(np.cos(ang)))
    assert np.all(np.abs(s - np.sin(ang)) <= _ulp32(np.sin(ang)) + 1e-45)
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)


def test_rope_neox_pairing_closed_form(oracle_mod):
    hd, theta = 64, 1.0e6
    c, s = oracle_mod.rope_table(100, hd, theta)
    for i in (0, 5, 31):
        e = np.zeros((1, hd), np.float32)
        e[0, i] = 1.0
        out = oracle_mod.rope(e, np.array([77], np.int32), 1, hd, c, s)
        a = 77 * theta ** (-2.0 * i / hd)
        want = np.zeros(hd)
        want[i], want[i + hd // 2] = math.cos(a), math.sin(a)
        assert np.allclose(out[0], want, atol=1e-6), i
        # the partner element rotates the other way
        e2 = np.zeros((1, hd), np.float32)
        e2[0, i + hd // 2] = 1.0
        out2 = oracle_mod.rope(e2, np.array([77], np.int32), 1, hd, c, s)
        want2 = np.zeros(hd)
        want2[i], want2[i + hd // 2] = -math.sin(a), math.cos(a)
        assert np.allclose(out2[0], want2, atol=1e-6), i


def test_rope_rotation_properties(oracle_mod):
    hd, nh = 128, 3
    c, s = oracle_mod.rope_table(400, hd, 1.0e6)
    rng = np.random.default_rng(9)
    q = rng.normal(0, 1, (1, nh * hd)).astype(np.float32)
    k = rng.normal(0, 1, (1, nh * hd)).astype(np.float32)
    half = hd // 2

    def R(v, p):
        return oracle_mod.rope(v, np.array([p], np.int32), nh, hd, c, s)

    # pair norms preserved
    r = R(q, 123).reshape(nh, hd)
    q3 = q.reshape(nh, hd)
    n0 = q3[:, :half] ** 2 + q3[:, half:] ** 2
    n1 = r[:, :half].astype(np.float64) ** 2 + r[:, half:].astype(np.float64) ** 2
    assert np.allclose(n0, n1, rtol=1e-5)
    # R(a) R(b) == R(a + b)
    assert np.allclose(R(R(q, 100), 150), R(q, 250), atol=2e-5)
    # position 0 is the identity, bit for bit
    assert np.array_equal(R(q, 0), q)
    # scores depend only on the relative position
    def score(p, t):
        return float(np.dot(R(q, p)[0, :hd].astype(np.float64), R(k, t)[0, :hd].astype(np.float64)))
    assert abs(score(30, 10) - score(230, 210)) < 1e-4
    assert abs(score(30, 10) - score(30, 20)) > 1e-3


# ---------------------------------------------------------------- attention

def _attention_brute(q, pos, K, V, nh, nkv, hd):
    nt = q.shape[0]
    out = np.zeros((nt, nh * hd))
    grp = nh // nkv
    for t in range(nt):
        for h in range(nh):
            g = h // grp
            qv = q[t, h * hd:(h + 1) * hd].astype(np.float64)
            Kg = K[:, g * hd:(g + 1) * hd].astype(np.float64)
            Vg = V[:, g * hd:(g + 1) * hd].astype(np.float64)
            sc = Kg @ qv / math.sqrt(hd)
            mask = np.arange(K.shape[0]) <= pos[t]  # explicit causal mask
            sc = np.where(mask, sc, -np.inf)
            p = np.exp(sc - sc.max())
            p /= p.sum()
            out[t, h * hd:(h + 1) * hd] = p @ Vg
    return out


def test_attention_brute_force_softmax(oracle_mod):
    rng = np.random.default_rng(10)
    nh, nkv, hd, n_ctx = 6, 2, 16, 24
    pos = np.array([3, 4, 5, 9, 10, 0], np.int32)
    q = rng.normal(0, 1, (6, nh * hd)).astype(np.float32)
    K = rng.normal(0, 1, (n_ctx, nkv * hd)).astype(np.float32)
    V = rng.normal(0, 1, (n_ctx, nkv * hd)).astype(np.float32)
    o = oracle_mod.attention(q, pos, K, V, nh, nkv, hd)
    ref = _attention_brute(q, pos, K, V, nh, nkv, hd)
    assert np.allclose(o, ref, rtol=1e-6, atol=1e-7)
    # GQA reduces to MHA when each KV head is repeated for its query group
    Kr = np.repeat(K.reshape(n_ctx, nkv, hd), nh // nkv, axis=1).reshape(n_ctx, nh * hd)
    Vr = np.repeat(V.reshape(n_ctx, nkv, hd), nh // nkv, axis=1).reshape(n_ctx, nh * hd)
    o_mha = oracle_mod.attention(q, pos, Kr, Vr, nh, nh, hd)
    assert np.allclose(o, o_mha, rtol=1e-6, atol=1e-7)
    # the token at position 0 sees only row 0: its output is V row 0 of its group
    assert np.allclose(o[5].reshape(nh, hd), Vr[0].reshape(nh, hd), atol=1e-7)


# ---------------------------------------------------------------- whole model invariants

@pytest.fixture(scope="module", params=["qwen2", "qwen3"])
def tiny(request, oracle_mod, synth_mod):
    """The tiny Qwen2-style model and its Qwen3 (QK-norm, no bias) variant:
    every model invariant below holds for both."""
    cfg = synth_mod.TINY if request.param == "qwen2" else synth_mod.QWEN3_TINY
    tensors = synth_mod.model_tensors(cfg)
    return cfg, tensors, oracle_mod.Model(cfg, tensors)


def _q8_model(oracle_mod, synth_mod, cfg, scale_qk: float):
    """cfg's model from Q8_0 blocks of its f32 tensors, with the Q and K
    projection block scales multiplied by scale_qk (exact for a power of two)."""
    m = oracle_mod.Model(cfg)
    for spec in synth_mod.tensor_specs(cfg):
        arr = synth_mod.tensor_data(spec)
        if spec.is_matrix:
            q, d = oracle_mod.q8_quantize(arr)
            if spec.name.endswith(("attn_q.weight", "attn_k.weight")):
                d = (d.view(np.float16) * np.float16(scale_qk)).view(np.uint16)
            nb = q.shape[1] // 32
            blocks = np.zeros((q.shape[0], nb, 34), np.uint8)
            blocks[:, :, :2] = d.reshape(q.shape[0], nb, 1).view(np.uint8)
            blocks[:, :, 2:] = q.reshape(q.shape[0], nb, 32).view(np.uint8)
            m.set_q8_0(spec.name, blocks.reshape(-1), spec.ne0, spec.ne1)
        else:
            m.set_f32(spec.name, arr)
    assert m.check()
    return m


def test_qk_norm_makes_attention_blind_to_the_qk_scale(oracle_mod, synth_mod):
    """QK-norm ("05 · Graph build", section 2.5 operation family: qk_norm for
    Qwen3; section 3.2, FusedQkvNorm: per-head Q/K RMSNorm before RoPE)
    normalizes each head: doubling every Q and K block scale leaves the
    logits bit-identical (with eps = 0 the doubling passes through the norm
    exactly), while the same change without QK-norm sharpens every softmax."""
    import dataclasses
    ids = synth_mod.token_ids(5, 24, 4096)
    pos = np.arange(24, dtype=np.int32)
    out = {}
    for qk in (True, False):
        cfg = dataclasses.replace(synth_mod.QWEN3_TINY, rms_eps=0.0, qk_norm=qk, qkv_bias=not qk)
        for scale in (1.0, 2.0):
            m = _q8_model(oracle_mod, synth_mod, cfg, scale)
            rc, lg, _ = m.prefill(m.kv(64), ids, pos)
            assert rc == 0
            out[qk, scale] = lg[0]
    assert np.array_equal(out[True, 1.0], out[True, 2.0])
    d = np.linalg.norm(out[False, 1.0] - out[False, 2.0]) / np.linalg.norm(out[False, 1.0])
    assert d > 1e-2, d


def test_model_causality(tiny, synth_mod):
    """Changing later tokens leaves earlier hidden states bit-identical (the
    causal rule of "09 · Prefill: the first forward", section 2.2)."""
    cfg, _, m = tiny
    ids = synth_mod.token_ids(0, 32, cfg.n_vocab)
    pos = np.arange(32, dtype=np.int32)
    _, _, h1 = m.prefill(m.kv(128), ids, pos, n_out=32, hidden=True)
    ids2 = ids.copy()
    ids2[20:] = (ids2[20:] + 17) % cfg.n_vocab
    _, _, h2 = m.prefill(m.kv(128), ids2, pos, n_out=32, hidden=True)
    for layer in range(cfg.n_layer + 1):
        assert np.array_equal(h1[layer, :20], h2[layer, :20]), layer
        assert not np.array_equal(h1[layer, 20:], h2[layer, 20:]), layer


def test_model_one_shot_equals_token_by_token(tiny, synth_mod):
    """One forward over the prompt equals nt single-token forwards at
    positions 0..nt-1 ("09 · Prefill: the first forward", section 2.3)."""
    cfg, _, m = tiny
    nt = 12
    ids = synth_mod.token_ids(0, nt, cfg.n_vocab)
    kv1, kv2 = m.kv(64), m.kv(64)
    rc, lg1, _ = m.prefill(kv1, ids, np.arange(nt, dtype=np.int32))
    assert rc == 0
    for t in range(nt):
        rc, lg2, _ = m.prefill(kv2, ids[t:t + 1], np.array([t], np.int32))
        assert rc == 0
    assert np.array_equal(lg1, lg2)
    for layer in range(cfg.n_layer):
        for which in (0, 1):
            assert np.array_equal(kv1.read(layer, which), kv2.read(layer, which))


def test_model_tail_equals_full_logits(tiny, synth_mod):
    """n_out=1 equals the last row of n_out=nt ("05 · Graph build", section 2.8)."""
    cfg, _, m = tiny
    ids = synth_mod.token_ids(3, 20, cfg.n_vocab)
    pos = np.arange(20, dtype=np.int32)
    _, lg1, _ = m.prefill(m.kv(64), ids, pos, n_out=1)
    _, lgf, _ = m.prefill(m.kv(64), ids, pos, n_out=20)
    assert np.array_equal(lg1[0], lgf[-1])
    _, lg5, _ = m.prefill(m.kv(64), ids, pos, n_out=5)
    assert np.array_equal(lg5, lgf[-5:])


def test_model_written_slots_and_errors(tiny, synth_mod):
    """Position p writes row p and nothing else; out-of-range positions or ids
    fail before anything is written ("09 · Prefill", sections 2.2 and 3.4)."""
    cfg, _, m = tiny
    kv = m.kv(64)
    w = cfg.n_head_kv * cfg.head_dim
    canary = np.full((64, w), np.float32(-7.25))
    for layer in range(cfg.n_layer):
        kv.write(layer, 0, 0, canary)
        kv.write(layer, 1, 0, canary)
    pos = np.array([5, 9, 10, 40, 63], np.int32)
    ids = synth_mod.token_ids(4, 5, cfg.n_vocab)
    assert m.prefill(kv, ids, np.array([5, 9, 10, 40, 64], np.int32))[0] == -2
    assert m.prefill(kv, ids, np.array([5, 9, -1, 40, 63], np.int32))[0] == -2
    bad = ids.copy(); bad[2] = cfg.n_vocab
    assert m.prefill(kv, bad, pos)[0] == -3
    for layer in range(cfg.n_layer):
        assert np.array_equal(kv.read(layer, 0), canary)
    # a repeated position is a bad argument (the pages give every token its
    # own slot): rejected before any write
    assert m.prefill(kv, ids, np.array([5, 9, 10, 9, 63], np.int32))[0] == -1
    for layer in range(cfg.n_layer):
        assert np.array_equal(kv.read(layer, 0), canary)
        assert np.array_equal(kv.read(layer, 1), canary)
    assert m.prefill(kv, ids, pos)[0] == 0
    for layer in range(cfg.n_layer):
        for which in (0, 1):
            r = kv.read(layer, which)
            changed = np.where(np.any(r != canary, axis=1))[0]
            assert changed.tolist() == pos.tolist()


def test_argmax_brute_force_with_ties(oracle_mod):
    """The argmax the acceptance bar compares: the largest value, ties to the
    lowest index (a plain loop over the vector decides)."""
    rng = np.random.default_rng(11)
    cases = [np.array([1.0, 3.0, 3.0, 2.0], np.float32),
             np.array([-5.0, -5.0, -7.0], np.float32),
             np.array([0.0], np.float32),
             np.array([2.0, -0.0, 0.0, 2.0], np.float32)]
    for _ in range(50):
        x = rng.integers(-4, 5, size=int(rng.integers(1, 300))).astype(np.float32)
        cases.append(x)
    cases.append(rng.standard_normal(151936).astype(np.float32))
    for x in cases:
        best = 0
        for i in range(1, x.size):
            if x[i] > x[best]:
                best = i
        assert oracle_mod.argmax(x) == best


def test_model_zero_weight_special_case(oracle_mod, synth_mod):
    """With every layer matrix and bias zero except the V bias, attention
    returns the V bias of each query head's group (softmax weights sum to 1),
    so h = embed + Q8_0(bv per head) . Wo and the FFN adds nothing: a closed
    form that pins the embedding, the residual adds, the GQA head mapping and
    the output projection."""
    cfg = synth_mod.TINY
    t = synth_mod.model_tensors(cfg)
    for name in list(t):
        if name.startswith("blk.") and not name.endswith("norm.weight") and "attn_output" not in name:
            t[name] = np.zeros_like(t[name])
    for i in range(cfg.n_layer):
        t[f"blk.{i}.attn_v.bias"] = synth_mod.normal(9, 100 + i, cfg.n_head_kv * cfg.head_dim, 0.0, 0.5)
    m = oracle_mod.Model(cfg, t)
    ids = synth_mod.token_ids(5, 6, cfg.n_vocab)
    rc, lg, hid = m.prefill(m.kv(16), ids, np.arange(6, dtype=np.int32), n_out=1, hidden=True)
    assert rc == 0
    H, hd, grp = cfg.n_embd, cfg.head_dim, cfg.n_head // cfg.n_head_kv
    eq, ed = m.get_q8("token_embd.weight", H, cfg.n_vocab)
    emb = eq[ids, :H].astype(np.float64) * np.repeat(ed[ids].view(np.float16).astype(np.float64), 32, axis=1)[:, :H]
    assert np.array_equal(hid[0], emb.astype(np.float32))
    h = emb.astype(np.float32)
    for i in range(cfg.n_layer):
        bv = t[f"blk.{i}.attn_v.bias"].reshape(cfg.n_head_kv, hd)
        att = np.concatenate([bv[hh // grp] for hh in range(cfg.n_head)])  # head hh reads group hh // grp
        aq, ad = oracle_mod.q8_quantize(att[None, :])
        wq, wd = m.get_q8(f"blk.{i}.attn_output.weight", cfg.n_head * hd, H)
        ar = oracle_mod.q8_dequantize(aq, ad, cfg.n_head * hd).astype(np.float64)
        wr = oracle_mod.q8_dequantize(wq, wd, cfg.n_head * hd).astype(np.float64)
        o = (ar @ wr.T).astype(np.float32)
        h = (h + o).astype(np.float32)
        rows = 6 if i < cfg.n_layer - 1 else 1
        assert np.allclose(hid[i + 1, :rows], h[-rows:], rtol=1e-6, atol=1e-7), i
        if i == cfg.n_layer - 1:
            h = h[-1:]
    # final norm + lm_head against the dequantized float64 closed form
    xn = h.astype(np.float64) / np.sqrt(np.mean(h.astype(np.float64) ** 2) + 1e-6) * t["output_norm.weight"]
    xq, xd = oracle_mod.q8_quantize(xn.astype(np.float32))
    oq, od = m.get_q8("output.weight", H, cfg.n_vocab)
    ref = oracle_mod.q8_dequantize(xq, xd, H).astype(np.float64) @ oracle_mod.q8_dequantize(oq, od, H).astype(np.float64).T
    # the normed row may differ from the oracle's f32 rounding by an ulp, which can move a code by one
    assert np.allclose(lg[0], ref[0], atol=0.02 * np.abs(ref).max())
    assert np.corrcoef(lg[0], ref[0])[0, 1] > 0.9999


# ---------------------------------------------------------------- sizes printed on the pages

def _golden_sizes():
    vals = {}
    with open(os.path.join(HERE, "golden", "pages_sizes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                name, v, tol = line.split()
                vals[name] = (float(v), float(tol))
    return vals


def test_sizes_printed_on_pages(oracle_mod, synth_mod):
    g = _golden_sizes()
    cfg = synth_mod.QWEN2_0_5B
    kvw = cfg.n_head_kv * cfg.head_dim
    per_token = 2 * kvw * 4 * cfg.n_layer
    got = {"kv_bytes_per_token": per_token, "kv_bytes_nctx4096": per_token * 4096,
           "k_region_bytes_per_layer": kvw * 4096 * 4, "logits_bytes": cfg.n_vocab * 4,
           "lm_head_macs_last_row": cfg.n_embd * cfg.n_vocab,
           "lm_head_macs_30_rows": 30 * cfg.n_embd * cfg.n_vocab}
    for k, (v, tol) in g.items():
        assert abs(got[k] - v) <= tol * v, (k, got[k], v)
    # and the oracle's own regions and logits have those sizes
    small = synth_mod.ModelConfig("kvsize", 1, cfg.n_embd, cfg.n_head, cfg.n_head_kv, cfg.head_dim,
                                  64, 8, tied=True)
    m = oracle_mod.Model(small)
    kv = m.kv(16)
    assert kv.read(0, 0).nbytes == 16 * kvw * 4


def test_attention_f32_variant_is_the_same_attention(oracle_mod):
    """The float32 rounding variant (used only to measure the drift floor)
    computes the same masked softmax attention to float32 accuracy."""
    rng = np.random.default_rng(12)
    nh, nkv, hd, n_ctx = 4, 2, 32, 40
    pos = np.array([0, 3, 17, 39, 20], np.int32)
    q = rng.normal(0, 1, (5, nh * hd)).astype(np.float32)
    K = rng.normal(0, 1, (n_ctx, nkv * hd)).astype(np.float32)
    V = rng.normal(0, 1, (n_ctx, nkv * hd)).astype(np.float32)
    ref = _attention_brute(q, pos, K, V, nh, nkv, hd)
    oracle_mod.set_attention_f32(True)
    try:
        o32 = oracle_mod.attention(q, pos, K, V, nh, nkv, hd)
    finally:
        oracle_mod.set_attention_f32(False)
    assert np.allclose(o32, ref, rtol=2e-5, atol=2e-6)
    assert not np.array_equal(o32, oracle_mod.attention(q, pos, K, V, nh, nkv, hd))


def test_committed_drift_floor_is_the_oracles(oracle_mod):
    """tests/golden/drift_floors.json (the bound the deep end-to-end GPU test
    scales) is what the oracle gives today: recomputed here, equal within the
    spread that the host's libm may introduce (last-bit differences of exp /
    cos / pow grow through the Q8_0 re-quantizations like any other)."""
    import json
    sys.path.insert(0, os.path.join(HERE, "golden"))
    try:
        import make_drift_floors
    finally:
        sys.path.pop(0)
    with open(os.path.join(HERE, "golden", "drift_floors.json")) as f:
        want = json.load(f)
    got = make_drift_floors.floors(want["workload"])
    assert got["argmax"] == want["argmax"]
    for a, b in zip(got["hidden_rel_l2"][1:], want["hidden_rel_l2"][1:]):
        assert 0.75 * b <= a <= 1.25 * b, (a, b)
    assert got["hidden_rel_l2"][0] == 0.0
    for k in ("logits_max_abs", "logits_rel_l2"):
        assert 0.75 * want[k] <= got[k] <= 1.25 * want[k], (k, got[k], want[k])
