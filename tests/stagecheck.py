"""Stage-level (teacher-forced) checks shared by the GPU parity tests: one
layer's weights quantized by the oracle as the model loader does, and the
one-row check that recomputes every stage of a layer from the GPU's own input
to that stage (the Qwen2 block of "09 · Prefill", section 3)."""
import numpy as np

import synth
from helpers import U, check_q8_requant, check_q8_sum, q8_sum_bound


class LayerWeights:
    """One layer's tensors, quantized by the oracle as the model loader does."""

    def __init__(self, oracle_mod, cfg, layer):
        specs = {s.name: s for s in synth.tensor_specs(cfg)}
        self.f32 = {}
        self.q8 = {}
        for kind in ("attn_norm.weight", "attn_q.weight", "attn_q.bias", "attn_k.weight",
                     "attn_k.bias", "attn_v.weight", "attn_v.bias", "attn_output.weight",
                     "ffn_norm.weight", "ffn_gate.weight", "ffn_up.weight", "ffn_down.weight",
                     "attn_q_norm.weight", "attn_k_norm.weight"):
            spec = specs.get(f"blk.{layer}.{kind}")
            if spec is None:  # a bias of a QK-norm model, or QK-norm of a plain one
                continue
            arr = synth.tensor_data(spec)
            if spec.is_matrix:
                self.q8[kind] = oracle_mod.q8_quantize(arr)
            else:
                self.f32[kind] = arr
        q, k, v = (self.q8[f"attn_{x}.weight"] for x in "qkv")
        self.q8["qkv"] = (np.concatenate([q[0], k[0], v[0]]), np.concatenate([q[1], k[1], v[1]]))
        nq, nkv = cfg.n_head * cfg.head_dim, cfg.n_head_kv * cfg.head_dim
        self.bias = (np.concatenate([self.f32[f"attn_{x}.bias"] for x in "qkv"]) if cfg.qkv_bias
                     else np.zeros(nq + 2 * nkv, np.float32))
        self.cfg = cfg

    def qk_normed(self, oracle_mod, full):
        """Q|K|V after the bias -> Q and K heads RMS-normalized (Qwen3), V as is."""
        cfg = self.cfg
        if not cfg.qk_norm:
            return full
        hd, nq, nkv = cfg.head_dim, cfg.n_head * cfg.head_dim, cfg.n_head_kv * cfg.head_dim
        out = full.copy()
        rows = full.shape[0]
        out[:, :nq] = oracle_mod.rmsnorm(full[:, :nq].reshape(-1, hd), self.f32["attn_q_norm.weight"],
                                         cfg.rms_eps).reshape(rows, nq)
        out[:, nq:nq + nkv] = oracle_mod.rmsnorm(full[:, nq:nq + nkv].reshape(-1, hd),
                                                 self.f32["attn_k_norm.weight"],
                                                 cfg.rms_eps).reshape(rows, nkv)
        return out


def check_row_layer(oracle_mod, g, kv, cfg, Wt, layer, p, h_in=None, qkv=None, x_captured=True):
    """Teacher-forced check of one layer for one row in the one-row (GEMV)
    layouts: every stage recomputed by the oracle from the GPU's own input to
    that stage.  h_in / qkv: that row's input and Q|K|V sums when the capture
    holds them for all rows (the last layer of a prompt); x_captured: the
    attn_norm codes were captured in the one-row layout.  Returns the GPU's
    output row of the layer."""
    H, hd, nh, nkv, F = cfg.n_embd, cfg.head_dim, cfg.n_head, cfg.n_head_kv, cfg.n_ff
    q, kvw = nh * hd, nkv * hd
    nbH, nbq, nbF = (H + 31) // 32, (q + 31) // 32, (F + 31) // 32
    pos = np.array([p], np.int32)

    def f32(name, n):
        return g.debug_read(name, np.empty((1, n), np.float32))

    def q8(name, nb):
        codes = g.debug_read(name + "_q8", np.empty((1, nb * 32), np.int8))
        sc = g.debug_read(name + "_s8", np.empty((1, nb), np.float32))
        assert np.array_equal(sc.astype(np.float16).astype(np.float32), sc)
        return codes, sc.astype(np.float16).view(np.uint16)

    oq, od = None, None
    if h_in is None:
        h_in = f32("h_in", H)
    if x_captured:
        xq, xd = q8("x", nbH)
        oq, od = oracle_mod.q8_quantize(oracle_mod.rmsnorm(h_in, Wt.f32["attn_norm.weight"], cfg.rms_eps))
        assert np.array_equal(xq, oq) and np.array_equal(xd, od), "attn_norm Q8_0"
    if qkv is None:
        qkv = f32("qkv", q + 2 * kvw)
        check_q8_sum(oracle_mod, qkv, xq, xd, *Wt.q8["qkv"], H)
    full = Wt.qk_normed(oracle_mod, (qkv + Wt.bias).astype(np.float32))
    c, s_ = oracle_mod.rope_table(p + 1, hd, cfg.rope_theta)
    want_q = oracle_mod.rope(full[:, :q], pos, nh, hd, c, s_)
    if x_captured:
        assert np.array_equal(f32("qrot", q), want_q), "rotated Q"
    K, V = kv.read(layer, 0, 0, p + 1), kv.read(layer, 1, 0, p + 1)
    assert np.array_equal(K[p:], oracle_mod.rope(full[:, q:q + kvw], pos, nkv, hd, c, s_)), "K row"
    assert np.array_equal(V[p:], full[:, q + kvw:]), "V row"
    att = f32("att", q)
    ref = oracle_mod.attention(want_q, pos, K, V, nh, nkv, hd)
    assert np.abs(att - ref).max() <= 2e-5 * max(1.0, np.abs(ref).max()), "attention"
    aq, ad = q8("att", nbq)
    gq, gd = oracle_mod.q8_quantize(att)
    assert np.array_equal(aq, gq) and np.array_equal(ad, gd), "attention Q8_0"
    h_mid = f32("h_mid", H)
    check_q8_sum(oracle_mod, h_mid, aq, ad, *Wt.q8["attn_output.weight"], q, base=h_in)
    fq, fd = q8("f", nbH)
    oq, od = oracle_mod.q8_quantize(oracle_mod.rmsnorm(h_mid, Wt.f32["ffn_norm.weight"], cfg.rms_eps))
    assert np.array_equal(fq, oq) and np.array_equal(fd, od), "ffn_norm Q8_0"
    gate = oracle_mod.matmul_q8(fq, fd, *Wt.q8["ffn_gate.weight"], H).astype(np.float64)
    up = oracle_mod.matmul_q8(fq, fd, *Wt.q8["ffn_up.weight"], H).astype(np.float64)
    s_ref = oracle_mod.swiglu(gate, up)
    dg, du = (q8_sum_bound(oracle_mod, fq, fd, *Wt.q8[f"ffn_{x}.weight"], H) for x in ("gate", "up"))
    sq, sd = q8("s", nbF)
    check_q8_requant(oracle_mod, sq, sd, s_ref,
                     1.1 * np.abs(up) * dg + (np.abs(gate) + 0.28) * du + 16 * U * np.abs(s_ref))
    check_q8_sum(oracle_mod, f32("h_out", H), sq, sd, *Wt.q8["ffn_down.weight"], F, base=h_mid)
    return f32("h_out", H)
