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
    top2 = np.sort(want)[-2:]
    if top2[1] - top2[0] > err:
        assert int(np.argmax(got)) == int(np.argmax(want)), "argmax differs"
    return err, rl2
