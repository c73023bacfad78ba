"""Write drift_floors.json: how far the oracle moves from itself over a deep
model when one step is rounded differently.

The oracle's attention is evaluated in double; its float32 variant
(oracle.set_attention_f32) is the same attention rounded in float32.  Run
over the 24-layer Qwen2-0.5B-shaped workload (512 tokens at positions
0..511), the two differ per hidden slot and in the logits by the amount that
an independent, correct rounding of one step grows to after every on-the-fly
Q8_0 re-quantization: the chaos floor against which an end-to-end
comparison of any non-bit-identical implementation is judged.

Only the oracle and the seeded inputs are used.  Run from the repository
root:  python tests/golden/make_drift_floors.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

WORKLOAD = "qwen2-0.5b-512"


def rel_l2(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def floors(workload: str = WORKLOAD) -> dict:
    oracle.build()
    w = synth.WORKLOADS[workload]
    cfg = w.model
    m = oracle.Model(cfg)
    for spec in synth.tensor_specs(cfg):
        m.set_f32(spec.name, synth.tensor_data(spec))
    ids, pos = w.ids(), w.positions()
    rc, lo, ho = m.prefill(m.kv(w.n_ctx), ids, pos, 1, hidden=True)
    assert rc == 0
    oracle.set_attention_f32(True)
    try:
        rc, l32, h32 = m.prefill(m.kv(w.n_ctx), ids, pos, 1, hidden=True)
    finally:
        oracle.set_attention_f32(False)
    assert rc == 0
    nt = w.n_tokens
    hidden = []
    for layer in range(cfg.n_layer + 1):
        rows = nt if layer < cfg.n_layer else 1
        hidden.append(rel_l2(h32[layer, :rows], ho[layer, :rows]))
    return {"workload": workload,
            "hidden_rel_l2": hidden,
            "logits_max_abs": float(np.abs(l32[0] - lo[0]).max()),
            "logits_rel_l2": rel_l2(l32[0], lo[0]),
            "argmax": oracle.argmax(lo[0]),
            "argmax_f32_attention": oracle.argmax(l32[0])}


if __name__ == "__main__":
    out = floors()
    with open(os.path.join(HERE, "drift_floors.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print(json.dumps(out))
