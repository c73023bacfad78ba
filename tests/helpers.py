"""Shared test helpers: build models from the seeded synthetic recipe on both
sides (the CUDA library and the oracle) and compare results."""
from __future__ import annotations

import numpy as np

import synth


def f32_tensors(cfg, seed: int = 0):
    """(name, array, ne0, ne1, MINFER_F32) for every tensor of cfg."""
    for spec in synth.tensor_specs(cfg):
        yield spec.name, synth.tensor_data(spec, seed), spec.ne0, spec.ne1, 0


def gpu_model(cfg, seed: int = 0):
    import quantized_transformer_prefill_gb300 as qp
    return qp.load_model(cfg, f32_tensors(cfg, seed))


def oracle_model(cfg, seed: int = 0):
    import oracle
    m = oracle.Model(cfg)
    for name, arr, _, _, _ in f32_tensors(cfg, seed):
        m.set_f32(name, arr)
    assert m.check()
    return m


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def check_logits(got, want, atol=2e-2, rtol_l2=1e-3):
    """The float acceptance bar: max-abs <= 2e-2 and rel-L2 <= 1e-3; argmax
    equal unless the reference's top-2 gap is below the measured error."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    err = float(np.max(np.abs(got - want)))
    rl2 = rel_l2(got, want)
    assert err <= atol, f"logits max-abs {err:.3e} > {atol}"
    assert rl2 <= rtol_l2, f"logits rel-L2 {rl2:.3e} > {rtol_l2}"
    import oracle
    top2 = np.sort(want)[-2:]
    if top2[1] - top2[0] > err:
        # the oracle's argmax (ties to the lowest index) on both sides
        assert oracle.argmax(got.astype(np.float32)) == oracle.argmax(want.astype(np.float32)), \
            "argmax differs"
    return err, rl2


U = 2.0 ** -24  # f32 unit roundoff


def check_q8_sum(oracle_mod, got, aq, ad, wq, wd, K, base=None):
    """got = base + (Q8_0 matmul) within the f32 bound of summing the nb block
    terms S_b * d_a * d_w (and the residual add); the bound uses
    sum_b sum_i |qa_i||qw_i| d_a d_w, an upper bound of sum_b |term_b|."""
    want = oracle_mod.matmul_q8(aq, ad, wq, wd, K)
    tol = q8_sum_bound(oracle_mod, aq, ad, wq, wd, K)
    if base is not None:
        want = (want.astype(np.float64) + base).astype(np.float32)
        tol = tol + 4 * U * np.abs(base)
    tol = tol + 4 * U * np.abs(want)
    err = np.abs(got.astype(np.float64) - want)
    bad = err > tol
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outside the f32 bound; worst "
                           f"{(err / np.maximum(tol, 1e-30)).max():.2f}x")
    return want


def q8_sum_bound(oracle_mod, aq, ad, wq, wd, K):
    """The f32 rounding bound of a Q8_0 matmul's block sums (see check_q8_sum)."""
    bound = oracle_mod.matmul_q8(np.abs(aq.astype(np.int16)).astype(np.int8), ad,
                                 np.abs(wq.astype(np.int16)).astype(np.int8), wd, K)
    return (aq.shape[1] // 32 + 8) * U * bound.astype(np.float64)


def check_q8_requant(oracle_mod, codes, scales, ref, slack):
    """Q8_0 of a value the GPU computed in f32 (codes/scales) against the
    oracle's value ref (Q8_0 block: d = amax/127 kept as fp16, codes round(x/d)).
    The dequantized GPU value lies within the Q8_0 error of ref (half a step
    plus 127 times the fp16 rounding of d) plus the f32 error `slack`; a code
    that differs from the oracle's own quantization differs by one step and
    only where ref lies within `slack` of a rounding boundary."""
    rows, n = ref.shape
    oq, od = oracle_mod.q8_quantize(ref)
    deq = oracle_mod.q8_dequantize(codes, scales, n).astype(np.float64)
    step = np.abs(oracle_mod.q8_dequantize(np.ones_like(codes), scales, n).astype(np.float64))
    assert np.all(np.abs(deq - ref) <= (0.5 + 128 * 2.0 ** -11) * step * (1 + 1e-3) + slack)
    diff = np.abs(codes[:, :n].astype(np.int32) - oq[:, :n].astype(np.int32))
    same_scale = np.repeat(scales == od, 32, axis=1)[:, :n]
    assert diff[same_scale].max(initial=0) <= 1
    nb = (n + 31) // 32
    padded = np.zeros((rows, nb * 32))
    padded[:, :n] = ref
    amax = np.abs(padded.reshape(rows, nb, 32)).max(axis=2, keepdims=True)
    d32 = np.maximum(amax, 1e-30) / 127.0
    t = (padded.reshape(rows, nb, 32) / d32).reshape(rows, nb * 32)[:, :n]
    dist = np.abs(t - np.floor(t) - 0.5)
    sl = np.zeros((rows, nb * 32))
    sl[:, :n] = slack
    tol_t = (sl.reshape(rows, nb, 32).max(axis=2, keepdims=True) / d32)
    tol_t = np.broadcast_to(tol_t, (rows, nb, 32)).reshape(rows, nb * 32)[:, :n] + 1e-4 * np.abs(t)
    flips = (diff > 0) & same_scale
    assert np.all(dist[flips] <= tol_t[flips] + 1e-3), "code flip away from a rounding boundary"
    assert flips.mean() <= 2e-3, flips.mean()
    # a block's fp16 scale may differ from the oracle's only by one fp16 step,
    # and only where the oracle's d = amax/127 lies within the f32 error of
    # amax (the block's largest slack, over 127) of the rounding boundary
    # between the two fp16 values
    sc = np.asarray(scales)[:, :nb]
    off = sc != od[:, :nb]
    if off.any():
        g16, o16 = sc[off].astype(np.int32), od[:, :nb][off].astype(np.int32)
        assert np.all(np.abs(g16 - o16) == 1), "scale off by more than one fp16 step"
        f16 = lambda b: np.asarray(b, dtype=np.uint16).view(np.float16).astype(np.float64)
        mid = 0.5 * (f16(sc[off]) + f16(od[:, :nb][off]))
        dref = amax[:, :, 0][off] / 127.0
        smax = sl.reshape(rows, nb, 32).max(axis=2)[off]
        assert np.all(np.abs(dref - mid) <= smax / 127.0 * (1 + 1e-3) + 2.0 ** -22 * dref), \
            "scale differs away from an fp16 rounding boundary"
