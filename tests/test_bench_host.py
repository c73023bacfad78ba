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
    for kernel in ("gemm_gate_up_swiglu", "attention", "rmsnorm_quant"):
        t = bench.profiled_traffic(kernel, "qwen2-0.5b-512")
        assert isinstance(t, int) and t > 1_000_000
    assert bench.profiled_traffic("gemm_down", "qwen2-0.5b-512") is None
    assert bench.profiled_traffic("gemm_gate_up_swiglu", "no-such-workload") is None
