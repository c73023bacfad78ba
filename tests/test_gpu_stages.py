"""Stage-by-stage parity of the CUDA kernels (through the C ABI) against the
oracle on identical inputs.

Bit-exact where the work decides integers: Q8_0 codes and fp16 scale bits,
per-32-block int32 dots, the set of KV rows written.  Float results within
tolerances derived from f32 arithmetic.
"""
import numpy as np
import pytest

from helpers import U, check_q8_requant, q8_sum_bound

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def qp():
    import quantized_transformer_prefill_gb300 as qp
    qp.lib()
    return qp


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _rows(seed, rows, n, kind="normal"):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        x = rng.normal(0, 1, (rows, n))
    elif kind == "wide":
        x = rng.normal(0, 1, (rows, n)) * np.exp(rng.uniform(-8, 8, (rows, 1)))
    elif kind == "cauchy":
        x = rng.standard_cauchy((rows, n))
    else:
        x = rng.normal(0, 1, (rows, n))
        x[:, ::7] = 0.0
        x[0] = 0.0
    return x.astype(np.float32)


@pytest.mark.parametrize("n", [32, 256, 688, 896, 1536, 3584])
@pytest.mark.parametrize("kind", ["normal", "wide", "cauchy", "zeros"])
def test_quantize_bit_exact(qp, oracle_mod, n, kind):
    x = _rows(n, 67, n, kind)
    q, d = qp.op_quantize(_dev(x))
    oq, od = oracle_mod.q8_quantize(x)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), od)


@pytest.mark.parametrize("n", [256, 896, 1536, 3584, 688])
def test_rmsnorm_quantize_bit_exact(qp, oracle_mod, n):
    x = _rows(n + 1, 131, n, "wide")
    w = (1 + np.random.default_rng(n).normal(0, 0.01, n)).astype(np.float32)
    q, d = qp.op_rmsnorm_quantize(_dev(x), _dev(w), 1e-6)
    oq, od = oracle_mod.q8_quantize(oracle_mod.rmsnorm(x, w, 1e-6))
    assert np.array_equal(d.cpu().numpy().view(np.uint16), od)
    assert np.array_equal(q.cpu().numpy(), oq)


def _q8_pair(oracle_mod, seed, M, N, K):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 1, (M, K)).astype(np.float32)
    w = rng.normal(0, 0.02, (N, K)).astype(np.float32)
    return oracle_mod.q8_quantize(x) + oracle_mod.q8_quantize(w)


@pytest.mark.parametrize("M,N,K", [(200, 300, 896), (37, 128, 224), (128, 1152, 256),
                                   (300, 520, 688), (1, 64, 64)])
def test_gemm_block_dots_bit_exact(qp, oracle_mod, M, N, K):
    xq, xd, wq, wd = _q8_pair(oracle_mod, M + N + K, M, N, K)
    y, dots = qp.op_gemm(_dev(xq), _dev(xd.view(np.int16)), _dev(wq), _dev(wd.view(np.int16)), K,
                         dots=True)
    assert np.array_equal(dots.cpu().numpy(), oracle_mod.block_dots(xq, wq))
    ref = oracle_mod.matmul_q8(xq, xd, wq, wd, K)
    np.testing.assert_allclose(y.cpu().numpy(), ref, rtol=2e-6, atol=2e-6 * np.abs(ref).max())


@pytest.mark.parametrize("M,N,K", [(512, 896, 4864), (512, 9728, 896), (2048, 1536, 1536),
                                   (130, 896, 896)])
def test_gemm_shapes_and_split_k(qp, oracle_mod, M, N, K):
    """Shapes of the 0.5B/1.5B layers: split-K (down/o), a wide N (gate/up),
    several M tiles with a ragged tail."""
    xq, xd, wq, wd = _q8_pair(oracle_mod, 7 * M + N, M, N, K)
    y = qp.op_gemm(_dev(xq), _dev(xd.view(np.int16)), _dev(wq), _dev(wd.view(np.int16)), K)
    rows = np.unique(np.concatenate([np.arange(0, M, max(1, M // 23)), [M - 1]]))
    ref = oracle_mod.matmul_q8(xq[rows], xd[rows], wq, wd, K)
    got = y.cpu().numpy()[rows]
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-5 * np.abs(ref).max())


@pytest.mark.parametrize("M,F,K", [(100, 688, 256), (257, 4864, 896)])
def test_gemm_swiglu_quantize(qp, oracle_mod, M, F, K):
    rng = np.random.default_rng(M + F)
    x = rng.normal(0, 1, (M, K)).astype(np.float32)
    g = rng.normal(0, 0.02, (F, K)).astype(np.float32)
    u = rng.normal(0, 0.02, (F, K)).astype(np.float32)
    xq, xd = oracle_mod.q8_quantize(x)
    gq, gd = oracle_mod.q8_quantize(g)
    uq, ud = oracle_mod.q8_quantize(u)
    sq, sd = qp.op_gemm_swiglu(_dev(xq), _dev(xd.view(np.int16)), _dev(gq), _dev(gd.view(np.int16)),
                               _dev(uq), _dev(ud.view(np.int16)), F, K)
    gg = oracle_mod.matmul_q8(xq, xd, gq, gd, K).astype(np.float64)
    uu = oracle_mod.matmul_q8(xq, xd, uq, ud, K).astype(np.float64)
    s_ref = oracle_mod.swiglu(gg, uu)
    oq, od = oracle_mod.q8_quantize(s_ref)
    sq = sq.cpu().numpy()
    sd = sd.cpu().numpy().view(np.uint16)
    # the GPU's gate/up are f32 block sums (error dg, du within their bounds);
    # silu' <= 1.1 and |silu(g)| <= |g| + 0.28 carry them into s = silu(g) u,
    # plus the f32 arithmetic of silu and of the product (10 units of
    # roundoff; 16 allowed): a code or a scale may then differ from the
    # oracle's own quantization only across a rounding boundary within that
    # bound
    dg = q8_sum_bound(oracle_mod, xq, xd, gq, gd, K)
    du = q8_sum_bound(oracle_mod, xq, xd, uq, ud, K)
    slack = 1.1 * np.abs(uu) * dg + (np.abs(gg) + 0.28) * du + 16 * U * np.abs(s_ref)
    check_q8_requant(oracle_mod, sq, sd, s_ref, slack)
    deq = oracle_mod.q8_dequantize(sq, sd, F)
    ref = oracle_mod.q8_dequantize(oq, od, F)
    assert np.linalg.norm(deq - ref) <= 1e-3 * np.linalg.norm(ref)


@pytest.mark.parametrize("nh,nkv,hd,nt,n_ctx,p0", [(4, 2, 64, 37, 64, 0), (14, 2, 64, 100, 160, 0),
                                                    (12, 2, 128, 50, 200, 120),
                                                    (28, 4, 128, 33, 64, 7),
                                                    # 64 rows and more: the tensor-core kernel
                                                    (14, 2, 64, 300, 512, 0),
                                                    (12, 2, 128, 257, 640, 200),
                                                    (16, 8, 128, 129, 256, 7),
                                                    (28, 4, 128, 640, 704, 0)])
def test_attention_vs_oracle(qp, oracle_mod, nh, nkv, hd, nt, n_ctx, p0):
    rng = np.random.default_rng(nh * hd + nt)
    q = rng.normal(0, 1, (nt, nh * hd)).astype(np.float32)
    K = rng.normal(0, 1, (n_ctx, nkv * hd)).astype(np.float32)
    V = rng.normal(0, 1, (n_ctx, nkv * hd)).astype(np.float32)
    pos = (p0 + np.arange(nt)).astype(np.int32)
    if p0 == 7:  # scattered, non-monotone positions
        pos = rng.permutation(n_ctx)[:nt].astype(np.int32)
    o = qp.op_attention(_dev(q), _dev(pos), _dev(K), _dev(V), nh, nkv, hd).cpu().numpy()
    ref = oracle_mod.attention(q, pos, K, V, nh, nkv, hd)
    err = np.abs(o - ref).max()
    assert err <= 2e-5 * max(1.0, np.abs(ref).max()), err


@pytest.mark.parametrize("nh,nkv,hd,n_ctx,p,grow", [
    (14, 2, 64, 4096, 0, False), (14, 2, 64, 4096, 31, False), (14, 2, 64, 4096, 32, False),
    (14, 2, 64, 4096, 512, False), (14, 2, 64, 4096, 4095, True),
    (14, 2, 64, 16384, 16383, True),   # 128 CTAs of 128 keys: two chunks each
    (28, 4, 128, 8192, 8191, True),    # 76 CTAs of ~108 keys
    (28, 4, 128, 8192, 700, False), (12, 2, 128, 600, 599, False), (16, 8, 128, 256, 200, False),
    (4, 2, 64, 64, 63, False), (16, 16, 64, 100, 57, True)])
def test_attention_one_row_vs_oracle(qp, oracle_mod, nh, nkv, hd, n_ctx, p, grow):
    """One query row (a single-token call, the last row of a prompt): the keys
    0..p of each KV head are dealt to many CTAs, each keeps an online softmax
    over chunks of keys, and the last CTA of the head merges the shares.  Keys
    that grow along the sequence make the chunk rescaling and the merge
    weights differ from one."""
    rng = np.random.default_rng(n_ctx + p + hd)
    q = rng.normal(0, 1, (1, nh * hd)).astype(np.float32)
    scale = (1.0 + np.arange(n_ctx) / 256.0).astype(np.float32)[:, None] if grow else 1.0
    K = (rng.normal(0, 1, (n_ctx, nkv * hd)) * scale).astype(np.float32)
    V = rng.normal(0, 1, (n_ctx, nkv * hd)).astype(np.float32)
    pos = np.array([p], np.int32)
    o = qp.op_attention(_dev(q), _dev(pos), _dev(K), _dev(V), nh, nkv, hd).cpu().numpy()
    ref = oracle_mod.attention(q, pos, K, V, nh, nkv, hd)
    err = np.abs(o - ref).max()
    assert err <= 2e-5 * max(1.0, np.abs(ref).max()), err


@pytest.mark.parametrize("nh,nkv,hd,nt", [(14, 2, 64, 384), (12, 2, 128, 300)])
def test_attention_rising_scores_vs_oracle(qp, oracle_mod, nh, nkv, hd, nt):
    """Keys that grow with their position push every row's running max up
    tile after tile, so the tensor-core kernel's rescaling of the O it keeps
    in TMEM (and of the sum) runs many times, next to its periodic folds."""
    rng = np.random.default_rng(hd + nt)
    n_ctx = nt
    q = rng.normal(0, 1, (nt, nh * hd)).astype(np.float32)
    grow = (1.0 + np.arange(n_ctx) / 32.0).astype(np.float32)[:, None]
    K = (rng.normal(0, 1, (n_ctx, nkv * hd)) * grow).astype(np.float32)
    V = rng.normal(0, 1, (n_ctx, nkv * hd)).astype(np.float32)
    pos = np.arange(nt, dtype=np.int32)
    o = qp.op_attention(_dev(q), _dev(pos), _dev(K), _dev(V), nh, nkv, hd).cpu().numpy()
    ref = oracle_mod.attention(q, pos, K, V, nh, nkv, hd)
    err = np.abs(o - ref).max()
    assert err <= 2e-5 * max(1.0, np.abs(ref).max()), err


def test_rope_store_vs_oracle(qp, oracle_mod):
    nh, nkv, hd, nt, n_ctx, theta = 14, 2, 64, 40, 96, 1.0e6
    rng = np.random.default_rng(11)
    W = (nh + 2 * nkv) * hd
    qkv = rng.normal(0, 1, (nt, W)).astype(np.float32)
    bias = rng.normal(0, 0.02, W).astype(np.float32)
    pos = rng.permutation(n_ctx)[:nt].astype(np.int32)
    canary = np.full((n_ctx, nkv * hd), -3.5, np.float32)
    Kd, Vd = _dev(canary), _dev(canary)
    q_out = qp.op_rope_store(_dev(qkv), _dev(bias), _dev(pos), nh, nkv, hd, theta, Kd, Vd)
    c, s = oracle_mod.rope_table(n_ctx, hd, theta)
    full = (qkv + bias).astype(np.float32)
    qr = oracle_mod.rope(full[:, :nh * hd], pos, nh, hd, c, s)
    kr = oracle_mod.rope(full[:, nh * hd:(nh + nkv) * hd], pos, nkv, hd, c, s)
    assert np.array_equal(q_out.cpu().numpy(), qr)
    Kh, Vh = Kd.cpu().numpy(), Vd.cpu().numpy()
    want_k, want_v = canary.copy(), canary.copy()
    want_k[pos] = kr
    want_v[pos] = full[:, (nh + nkv) * hd:]
    assert np.array_equal(Kh, want_k)
    assert np.array_equal(Vh, want_v)


@pytest.mark.parametrize("nh,nkv,hd", [(4, 2, 64), (16, 8, 128)])
def test_qknorm_rope_store_vs_oracle(qp, oracle_mod, nh, nkv, hd):
    """Qwen3: per-head RMSNorm of Q and K between the bias and RoPE, bit-exact
    against the oracle's rmsnorm and rope on the same sums."""
    nt, n_ctx, theta, eps = 37, 80, 1.0e6, 1e-6
    rng = np.random.default_rng(nh + hd)
    W = (nh + 2 * nkv) * hd
    qkv = (rng.normal(0, 1, (nt, W)) * np.exp(rng.uniform(-3, 3, (nt, 1)))).astype(np.float32)
    qn = (1 + rng.normal(0, 0.01, hd)).astype(np.float32)
    kn = (1 + rng.normal(0, 0.01, hd)).astype(np.float32)
    pos = rng.permutation(n_ctx)[:nt].astype(np.int32)
    Kd = _dev(np.zeros((n_ctx, nkv * hd), np.float32))
    Vd = _dev(np.zeros((n_ctx, nkv * hd), np.float32))
    q_out = qp.op_qknorm_rope_store(_dev(qkv), None, _dev(qn), _dev(kn), eps, _dev(pos), nh, nkv,
                                    hd, theta, Kd, Vd)
    c, s = oracle_mod.rope_table(n_ctx, hd, theta)
    qh = oracle_mod.rmsnorm(qkv[:, :nh * hd].reshape(-1, hd), qn, eps).reshape(nt, nh * hd)
    kh = oracle_mod.rmsnorm(qkv[:, nh * hd:(nh + nkv) * hd].reshape(-1, hd), kn, eps).reshape(nt, -1)
    assert np.array_equal(q_out.cpu().numpy(), oracle_mod.rope(qh, pos, nh, hd, c, s))
    Kh, Vh = Kd.cpu().numpy(), Vd.cpu().numpy()
    assert np.array_equal(Kh[pos], oracle_mod.rope(kh, pos, nkv, hd, c, s))
    assert np.array_equal(Vh[pos], qkv[:, (nh + nkv) * hd:])
