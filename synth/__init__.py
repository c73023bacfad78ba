"""Seeded synthetic inputs shared by the tests, the oracle runs and the bench.

This module only draws numbers (see ``synth.c`` for the generator's published
definition) and describes the five model shapes.  It holds none of the
forward pass's arithmetic: no quantization, normalisation or matmul.

The shapes follow the Qwen2 family as the "Graph build" page of the minfer
walkthrough describes it (section 2.5: hidden 896, 14 query heads of dim 64,
2 KV heads, FFN 4864, vocabulary 151936 for the 0.5B model), extended to the
1.5B and 7B shapes and a tiny 2-layer model for fast oracle runs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``libsynth.so`` next to it (plain gcc)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               src, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.synth_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                             ctypes.c_double, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_void_p]
            lib.synth_ids.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int32,
                                      ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
            lib.synth_q8_0_blocks.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                              ctypes.c_double, ctypes.c_int64, ctypes.c_void_p]
            lib.synth_u64.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
            lib.synth_u64.restype = ctypes.c_uint64
            _lib = lib
    return _lib


def normal(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0,
           first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().synth_normal_f32(seed, stream, mean, std, first, n, out.ctypes.data)
    return out


def token_ids(seed: int, n: int, vocab: int, stream: int = 1_000_000, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().synth_ids(seed, stream, vocab, first, n, out.ctypes.data)
    return out


def q8_0_blocks(seed: int, stream: int, nblocks: int, lo: float = 2.0 ** -12,
                hi: float = 2.0 ** -7) -> np.ndarray:
    """Random bytes in the 34-byte Q8_0 block format (scale bits, 32 codes)."""
    out = np.empty(nblocks * 34, dtype=np.uint8)
    _load().synth_q8_0_blocks(seed, stream, lo, hi, nblocks, out.ctypes.data)
    return out


def u64(seed: int, stream: int, i: int) -> int:
    return int(_load().synth_u64(seed, stream, i))


@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layer: int
    n_embd: int
    n_head: int
    n_head_kv: int
    head_dim: int
    n_ff: int
    n_vocab: int
    tied: bool
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6
    max_seq_len: int = 32768
    weight_std: float = 0.02
    bias_std: float = 0.02
    norm_std: float = 0.01
    qk_norm: bool = False   # Qwen3: per-head RMSNorm of Q and K before RoPE
    qkv_bias: bool = True   # Qwen2 carries Q/K/V biases, Qwen3 none


@dataclass(frozen=True)
class Workload:
    """One prefill call (or a pre-fill call followed by the timed append)."""
    name: str
    model: ModelConfig
    n_tokens: int
    p0: int
    n_ctx: int
    prompt_seed: int = 0
    prefill_tokens: int = 0      # tokens pre-filled (untimed) at positions 0..prefill_tokens-1
    prefill_seed: int = 0
    n_out: int = 1               # logits rows returned (the last n_out tokens)

    def positions(self) -> np.ndarray:
        return np.arange(self.p0, self.p0 + self.n_tokens, dtype=np.int32)

    def ids(self) -> np.ndarray:
        return token_ids(self.prompt_seed, self.n_tokens, self.model.n_vocab)

    def prefill_ids(self) -> np.ndarray:
        return token_ids(self.prefill_seed, self.prefill_tokens, self.model.n_vocab)


TINY = ModelConfig("tiny", 2, 256, 4, 2, 64, 688, 4096, tied=False, max_seq_len=128)
QWEN2_0_5B = ModelConfig("qwen2-0.5b", 24, 896, 14, 2, 64, 4864, 151936, tied=True)
QWEN2_1_5B = ModelConfig("qwen2-1.5b", 28, 1536, 12, 2, 128, 8960, 151936, tied=False)
QWEN2_7B = ModelConfig("qwen2-7b", 28, 3584, 28, 4, 128, 18944, 152064, tied=False)
# Qwen3 variant (per-head QK RMSNorm, no Q/K/V bias): a tiny model for strict
# parity and the 0.6B shape (28 layers, H 1024, 16/8 heads of 128, FFN 3072)
QWEN3_TINY = ModelConfig("qwen3-tiny", 2, 256, 4, 2, 64, 688, 4096, tied=True, max_seq_len=128,
                         qk_norm=True, qkv_bias=False)
QWEN3_0_6B = ModelConfig("qwen3-0.6b", 28, 1024, 16, 8, 128, 3072, 151936, tied=True,
                         qk_norm=True, qkv_bias=False)

WORKLOADS = {
    "tiny-32": Workload("tiny-32", TINY, 32, 0, 128),
    "qwen2-0.5b-512": Workload("qwen2-0.5b-512", QWEN2_0_5B, 512, 0, 4096),
    "qwen2-1.5b-2048": Workload("qwen2-1.5b-2048", QWEN2_1_5B, 2048, 0, 4096),
    "qwen2-7b-4096": Workload("qwen2-7b-4096", QWEN2_7B, 4096, 0, 8192),
    "qwen2-1.5b-append-1024": Workload("qwen2-1.5b-append-1024", QWEN2_1_5B, 1024, 3072, 4096,
                                       prompt_seed=1, prefill_tokens=3072, prefill_seed=0),
    # decode-shaped calls: one token after a 512-token turn already in the cache
    "qwen2-0.5b-decode-1": Workload("qwen2-0.5b-decode-1", QWEN2_0_5B, 1, 512, 4096,
                                    prompt_seed=2, prefill_tokens=512, prefill_seed=0),
    "qwen2-7b-decode-1": Workload("qwen2-7b-decode-1", QWEN2_7B, 1, 512, 8192,
                                  prompt_seed=2, prefill_tokens=512, prefill_seed=0),
    # every prompt token's logits (n_out = n_tokens)
    "qwen2-0.5b-512-all-logits": Workload("qwen2-0.5b-512-all-logits", QWEN2_0_5B, 512, 0, 4096,
                                          n_out=512),
    "qwen3-tiny-32": Workload("qwen3-tiny-32", QWEN3_TINY, 32, 0, 128),
    "qwen3-0.6b-512": Workload("qwen3-0.6b-512", QWEN3_0_6B, 512, 0, 4096),
}

# stream ids of the per-tensor generators
_GLOBAL_STREAMS = {"token_embd.weight": 1, "output_norm.weight": 2, "output.weight": 3}
_LAYER_KINDS = ["attn_norm.weight", "attn_q.weight", "attn_q.bias", "attn_k.weight", "attn_k.bias",
                "attn_v.weight", "attn_v.bias", "attn_output.weight", "ffn_norm.weight",
                "ffn_gate.weight", "ffn_up.weight", "ffn_down.weight", "attn_q_norm.weight",
                "attn_k_norm.weight"]


@dataclass(frozen=True)
class TensorSpec:
    name: str
    ne0: int          # contiguous (input) dimension
    ne1: int          # rows (output dimension); 1 for vectors
    stream: int
    mean: float
    std: float

    @property
    def numel(self) -> int:
        return self.ne0 * self.ne1

    @property
    def is_matrix(self) -> bool:
        return self.ne1 > 1 and not self.name.endswith(".bias")


def tensor_specs(cfg: ModelConfig) -> list[TensorSpec]:
    """Every tensor of the model with its GGUF-style name and its draw recipe."""
    H, q, kv, F, V = (cfg.n_embd, cfg.n_head * cfg.head_dim, cfg.n_head_kv * cfg.head_dim,
                      cfg.n_ff, cfg.n_vocab)
    w, b, nrm = cfg.weight_std, cfg.bias_std, cfg.norm_std
    specs = [TensorSpec("token_embd.weight", H, V, 1, 0.0, w),
             TensorSpec("output_norm.weight", H, 1, 2, 1.0, nrm)]
    if not cfg.tied:
        specs.append(TensorSpec("output.weight", H, V, 3, 0.0, w))
    shapes = {"attn_norm.weight": (H, 1, 1.0, nrm), "attn_q.weight": (H, q, 0.0, w),
              "attn_q.bias": (q, 1, 0.0, b), "attn_k.weight": (H, kv, 0.0, w),
              "attn_k.bias": (kv, 1, 0.0, b), "attn_v.weight": (H, kv, 0.0, w),
              "attn_v.bias": (kv, 1, 0.0, b), "attn_output.weight": (q, H, 0.0, w),
              "ffn_norm.weight": (H, 1, 1.0, nrm), "ffn_gate.weight": (H, F, 0.0, w),
              "ffn_up.weight": (H, F, 0.0, w), "ffn_down.weight": (F, H, 0.0, w),
              "attn_q_norm.weight": (cfg.head_dim, 1, 1.0, nrm),
              "attn_k_norm.weight": (cfg.head_dim, 1, 1.0, nrm)}
    for i in range(cfg.n_layer):
        for k, kind in enumerate(_LAYER_KINDS):
            if kind.endswith(".bias") and not cfg.qkv_bias:
                continue
            if kind.endswith("_norm.weight") and kind.startswith("attn_") and kind != "attn_norm.weight" \
                    and not cfg.qk_norm:
                continue
            ne0, ne1, mean, std = shapes[kind]
            specs.append(TensorSpec(f"blk.{i}.{kind}", ne0, ne1, 16 + 16 * i + k, mean, std))
    return specs


def tensor_data(spec: TensorSpec, seed: int = 0) -> np.ndarray:
    """The f32 values of one tensor, row-major [ne1][ne0]."""
    return normal(seed, spec.stream, spec.numel, spec.mean, spec.std).reshape(spec.ne1, spec.ne0) \
        if spec.ne1 > 1 else normal(seed, spec.stream, spec.numel, spec.mean, spec.std)


def model_tensors(cfg: ModelConfig, seed: int = 0) -> dict[str, np.ndarray]:
    """All tensors as f32 arrays (only for shapes small enough to hold on the host)."""
    return {s.name: tensor_data(s, seed) for s in tensor_specs(cfg)}
