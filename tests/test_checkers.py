"""The tolerance checkers used by the full-size parity tests must reject the
mistakes they exist to catch.  Each mistake is planted on the CPU in values
produced by the oracle itself."""
import numpy as np

from helpers import check_q8_requant, check_q8_sum


def _raises(fn, *args, **kw):
    try:
        fn(*args, **kw)
    except AssertionError:
        return True
    return False


def _operands(oracle_mod, seed, M=6, N=40, K=896):
    rng = np.random.default_rng(seed)
    aq, ad = oracle_mod.q8_quantize(rng.normal(0, 1, (M, K)).astype(np.float32))
    wq, wd = oracle_mod.q8_quantize(rng.normal(0, 0.02, (N, K)).astype(np.float32))
    return aq, ad, wq, wd, K


def test_sum_checker_accepts_reordered_f32_sum(oracle_mod):
    aq, ad, wq, wd, K = _operands(oracle_mod, 1)
    dots = oracle_mod.block_dots(aq, wq).astype(np.float32)      # [M][N][nb]
    da = oracle_mod.q8_dequantize(np.ones_like(aq), ad, K)[:, ::32]
    dw = oracle_mod.q8_dequantize(np.ones_like(wq), wd, K)[:, ::32]
    # f32 accumulation in reverse block order: a legal rounding order
    acc = np.zeros(dots.shape[:2], np.float32)
    for b in reversed(range(dots.shape[2])):
        acc = (acc + dots[:, :, b] * (da[:, None, b] * dw[None, :, b])).astype(np.float32)
    check_q8_sum(oracle_mod, acc, aq, ad, wq, wd, K)
    base = np.random.default_rng(2).normal(0, 3, acc.shape).astype(np.float32)
    check_q8_sum(oracle_mod, (acc + base).astype(np.float32), aq, ad, wq, wd, K, base=base)


def test_sum_checker_rejects_dropped_block_and_scale(oracle_mod):
    aq, ad, wq, wd, K = _operands(oracle_mod, 3)
    good = oracle_mod.matmul_q8(aq, ad, wq, wd, K)
    # one block of one row dropped
    aq2 = aq.copy()
    aq2[2, 64:96] = 0
    assert _raises(check_q8_sum, oracle_mod, oracle_mod.matmul_q8(aq2, ad, wq, wd, K),
                   aq, ad, wq, wd, K)
    # one block's activation scale off by one fp16 step
    ad2 = ad.copy()
    ad2[4, 5] += 1
    assert _raises(check_q8_sum, oracle_mod, oracle_mod.matmul_q8(aq, ad2, wq, wd, K),
                   aq, ad, wq, wd, K)
    # a missing residual
    base = np.ones_like(good)
    assert _raises(check_q8_sum, oracle_mod, good, aq, ad, wq, wd, K, base=base)


def test_requant_checker(oracle_mod):
    rng = np.random.default_rng(5)
    ref = rng.normal(0, 0.1, (8, 700))
    slack = 4e-6 * np.abs(ref)
    x = (ref * (1 + rng.normal(0, 1e-6, ref.shape))).astype(np.float32)
    q, d = oracle_mod.q8_quantize(x)
    check_q8_requant(oracle_mod, q, d, ref, slack)
    q2 = q.copy()
    q2[3, 100] += 1           # a flip away from any boundary
    assert _raises(check_q8_requant, oracle_mod, q2, d, ref, slack)
    q3, d3 = oracle_mod.q8_quantize((ref * 1.01).astype(np.float32))   # a scaled output
    assert _raises(check_q8_requant, oracle_mod, q3, d3, ref, slack)
    # one block's scale one fp16 step off, its d far from a rounding boundary
    f16 = lambda b: np.asarray(b, dtype=np.uint16).view(np.float16).astype(np.float64)
    amax = np.abs(np.pad(ref, ((0, 0), (0, 4)))).reshape(8, 22, 32).max(axis=2)
    frac = (amax / 127.0 - f16(d)) / (f16(d + 1) - f16(d))
    r, b = np.argwhere(np.abs(frac) < 0.2)[0]
    d4 = d.copy()
    d4[r, b] += 1
    assert _raises(check_q8_requant, oracle_mod, q, d4, ref, slack)
    # the same step where d sits on the boundary within the slack passes
    ref5 = ref.copy()
    blk = ref5[r, 32 * b:32 * b + 32]
    k = int(np.argmax(np.abs(blk)))
    mid = 0.5 * (f16(d[r, b]) + f16(d[r, b] + 1))
    blk[k] = np.sign(blk[k]) * mid * 127.0   # amax / 127 exactly on the boundary
    q5, d5 = oracle_mod.q8_quantize(ref5.astype(np.float32))
    d6 = d5.copy()
    d6[r, b] = d5[r, b] + 1 if f16(d5[r, b]) < mid else d5[r, b] - 1
    check_q8_requant(oracle_mod, q5, d6, ref5, 4e-6 * np.abs(ref5))
