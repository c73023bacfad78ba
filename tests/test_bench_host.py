"""Host-side arithmetic of the measurement (CPU): the work counts behind the
roofline fractions and the DRAM traffic read from the committed ncu summaries."""
import bench
import synth


def _brute_force_macs(cfg, nt, p0, n_out):
    """Walk layers and rows one by one: every layer projects Q|K|V for all rows;
    the last layer carries only the last n_out rows through attention, Wo and
    the FFN; each attending row t reads keys 0..p0+t."""
    H, q = cfg.n_embd, cfg.n_head * cfg.head_dim
    kv = cfg.n_head_kv * cfg.head_dim
    mm = attn = 0
    for layer in range(cfg.n_layer):
        last = layer == cfg.n_layer - 1
        for t in range(nt):
            mm += H * q + 2 * H * kv                     # Q, K, V projections
            if last and t < nt - n_out:
                continue
            keys = p0 + t + 1
            attn += keys * q + keys * q                  # Q.K^T and P.V
            mm += q * H                                  # Wo
            mm += 2 * H * cfg.n_ff + cfg.n_ff * H        # gate, up, down
    return mm, n_out * H * cfg.n_vocab, attn


def test_forward_macs_equals_a_row_by_row_count():
    tiny = synth.WORKLOADS["qwen3-tiny-32"].model
    for nt, p0, n_out in [(32, 0, 1), (17, 5, 1), (9, 40, 3), (1, 100, 1), (12, 0, 12)]:
        assert bench.forward_macs(tiny, nt, p0, n_out) == _brute_force_macs(tiny, nt, p0, n_out)


def test_per_token_matmul_work_and_lm_head_of_the_shapes():
    """Per token and layer H(q+2kv) + qH + 3HF: 14.9 M (0.5B), 46.8 M (1.5B),
    233 M (7B); the 0.5B lm_head on one row is 896 x 151936 MACs (the pages'
    1.4e8 for the last-row-only head)."""
    want = {"qwen2-0.5b-512": 14.9e6, "qwen2-1.5b-2048": 46.8e6, "qwen2-7b-4096": 233e6}
    for name, per_tok in want.items():
        cfg = synth.WORKLOADS[name].model
        mm_one, _, _ = bench.forward_macs(cfg, 1, 0, 1)
        assert abs(mm_one / cfg.n_layer - per_tok) < 0.005 * per_tok  # 3-digit figures
    cfg = synth.WORKLOADS["qwen2-0.5b-512"].model
    assert bench.forward_macs(cfg, 512, 0, 1)[1] == 896 * 151936 == 136134656


def test_profiled_traffic_reads_the_committed_summaries():
    for kernel in ("gemm_gate_up_swiglu", "attention", "rmsnorm_quant", "gemm_qkv", "gemm_o",
                   "gemm_down", "rope_kv_store", "lm_head_gemv"):
        t = bench.profiled_traffic(kernel, "qwen2-0.5b-512")
        assert isinstance(t, int) and t > 1_000_000
    assert bench.profiled_traffic("embed", "qwen2-0.5b-512") is None
    assert bench.profiled_traffic("gemm_gate_up_swiglu", "no-such-workload") is None


def test_forward_roofline_limits():
    """T* with unlimited bandwidth is the forward's flops at the tensor peak
    (GEMMs, attention and the lm_head); with unlimited compute it is the
    algorithmic bytes at the bandwidth, counted here step by step."""
    for name in ("tiny-32", "qwen2-0.5b-512", "qwen2-1.5b-append-1024"):
        w = synth.WORKLOADS[name]
        cfg = w.model
        nt, p0, n_out = w.n_tokens, w.p0, w.n_out
        mm, lm, attn = bench.forward_macs(cfg, nt, p0, n_out)
        t, parts = bench.forward_roofline(cfg, nt, p0, n_out, 1e30, 1.0)
        assert abs(t - 2 * (mm + lm + attn) / 1e12) <= 1e-9 * t
        assert parts["memory"] < 1e-12 * t
        # bytes, one step at a time
        H, q = cfg.n_embd, cfg.n_head * cfg.head_dim
        kv, F, L, V = cfg.n_head_kv * cfg.head_dim, cfg.n_ff, cfg.n_layer, cfg.n_vocab
        e = 34 / 32
        b = nt * H * 5
        for layer in range(L):
            r = n_out if layer == L - 1 else nt
            b += nt * H * (4 + e)                                      # attn_norm
            b += (q + 2 * kv) * H * e + nt * H * e + nt * (q + 2 * kv) * 4  # QKV GEMM
            b += 2 * nt * (q + 2 * kv) * 4                             # RoPE + store
            b += r * q * 4 + (p0 + nt) * 2 * kv * 4 + r * q * e        # attention
            b += H * q * e + r * q * e + r * H * 4                     # Wo
            b += r * H * (12 + e)                                      # residual + ffn_norm
            b += 2 * F * H * e + r * H * e + r * F * e                 # gate/up + SwiGLU out
            b += H * F * e + r * F * e + r * H * 4                     # down
            b += 2 * r * H * 4                                         # residual
        b += n_out * H * (4 + e) + V * H * e + n_out * V * 4           # final norm, lm_head
        t, _ = bench.forward_roofline(cfg, nt, p0, n_out, 1.0, 1e30)
        assert abs(t * 1e9 - b) <= 1e-9 * b, (name, t * 1e9, b)
