"""ctypes binding of the CPU oracle (``oracle.cpp``).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``.  The product library never
imports, links or runs anything in this directory.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {0: "ok", -1: "bad arguments", -2: "position out of range", -3: "token id out of range",
          -4: "missing tensor"}


def build(force: bool = False) -> str:
    """Compile the oracle with plain g++ (-O3, OpenMP, no FMA contraction)."""
    src = os.path.join(_HERE, "oracle.cpp")
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(src):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O3", "-std=c++17", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-fno-fast-math", src, "-o", tmp])
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


class Hparams(ctypes.Structure):
    _fields_ = [("n_layer", ctypes.c_int), ("n_embd", ctypes.c_int), ("n_head", ctypes.c_int),
                ("n_head_kv", ctypes.c_int), ("head_dim", ctypes.c_int), ("n_ff", ctypes.c_int),
                ("n_vocab", ctypes.c_int), ("max_seq_len", ctypes.c_int),
                ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("tied_embeddings", ctypes.c_int), ("qk_norm", ctypes.c_int)]


def _lib_handle():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(LIB_PATH)
            P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            sig = {
                "orc_f32_to_f16": ([ctypes.c_float], ctypes.c_uint16),
                "orc_f16_to_f32": ([ctypes.c_uint16], ctypes.c_float),
                "orc_q8_quantize": ([P, I64, I64, P, P], None),
                "orc_q8_dequantize": ([P, P, I64, I64, P], None),
                "orc_block_dots": ([P, I64, P, I64, I64, P], None),
                "orc_matmul_q8": ([P, P, I64, P, P, I64, I64, P, P], None),
                "orc_rmsnorm": ([P, P, I64, I64, ctypes.c_float, P], None),
                "orc_rope_table": ([I, I, ctypes.c_float, P, P], None),
                "orc_rope": ([P, I64, I, I, P, P, P], None),
                "orc_attention": ([P, I64, P, P, P, I, I, I, P], None),
                "orc_swiglu": ([P, P, I64, P], None),
                "orc_model_create": ([ctypes.POINTER(Hparams)], P),
                "orc_model_free": ([P], None),
                "orc_model_set_f32": ([P, ctypes.c_char_p, P, I64, I64], I),
                "orc_model_set_q8_0": ([P, ctypes.c_char_p, P, I64, I64], I),
                "orc_model_get_q8": ([P, ctypes.c_char_p, P, P], I),
                "orc_model_check": ([P], I),
                "orc_kv_create": ([P, I], P),
                "orc_kv_free": ([P], None),
                "orc_kv_ctx": ([P], I),
                "orc_kv_read": ([P, I, I, I, I, P, I64], I),
                "orc_kv_write": ([P, I, I, I, I, P, I64], I),
                "orc_prefill": ([P, P, P, P, I, I, P, P], I),
                "orc_argmax": ([P, I64], I64),
                "orc_set_attention_f32": ([I], I),
            }
            for name, (args, res) in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


# ---------------- stage functions ----------------

def f32_to_f16_bits(x: float) -> int:
    return int(_lib_handle().orc_f32_to_f16(float(x)))


def f16_bits_to_f32(h: int) -> float:
    return float(_lib_handle().orc_f16_to_f32(int(h)))


def q8_quantize(x: np.ndarray):
    """Rows of x [rows][n] -> (codes int8 [rows][nb*32], scale bits uint16 [rows][nb])."""
    x, px = _c(np.atleast_2d(x), np.float32)
    rows, n = x.shape
    nb = (n + 31) // 32
    q = np.zeros((rows, nb * 32), np.int8)
    d = np.zeros((rows, nb), np.uint16)
    _lib_handle().orc_q8_quantize(px, rows, n, q.ctypes.data, d.ctypes.data)
    return q, d


def q8_dequantize(q: np.ndarray, d: np.ndarray, n: int) -> np.ndarray:
    q, pq = _c(q, np.int8)
    d, pd = _c(d, np.uint16)
    rows = q.shape[0]
    x = np.zeros((rows, n), np.float32)
    _lib_handle().orc_q8_dequantize(pq, pd, rows, n, x.ctypes.data)
    return x


def block_dots(qa: np.ndarray, qw: np.ndarray) -> np.ndarray:
    qa, pa = _c(qa, np.int8)
    qw, pw = _c(qw, np.int8)
    M, N, nb = qa.shape[0], qw.shape[0], qa.shape[1] // 32
    out = np.zeros((M, N, nb), np.int32)
    _lib_handle().orc_block_dots(pa, M, pw, N, nb, out.ctypes.data)
    return out


def matmul_q8(xq, xd, wq, wd, K: int, bias=None) -> np.ndarray:
    xq, pxq = _c(xq, np.int8)
    xd, pxd = _c(xd, np.uint16)
    wq, pwq = _c(wq, np.int8)
    wd, pwd = _c(wd, np.uint16)
    M, N = xq.shape[0], wq.shape[0]
    pb = None
    if bias is not None:
        bias, pb = _c(bias, np.float32)
    y = np.zeros((M, N), np.float32)
    _lib_handle().orc_matmul_q8(pxq, pxd, M, pwq, pwd, N, K, pb, y.ctypes.data)
    return y


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    x, px = _c(np.atleast_2d(x), np.float32)
    w, pw = _c(w, np.float32)
    y = np.zeros_like(x)
    _lib_handle().orc_rmsnorm(px, pw, x.shape[0], x.shape[1], eps, y.ctypes.data)
    return y


def rope_table(n_ctx: int, hd: int, theta: float):
    c = np.zeros((n_ctx, hd // 2), np.float32)
    s = np.zeros((n_ctx, hd // 2), np.float32)
    _lib_handle().orc_rope_table(n_ctx, hd, theta, c.ctypes.data, s.ctypes.data)
    return c, s


def rope(x: np.ndarray, pos: np.ndarray, nheads: int, hd: int, cos_t, sin_t) -> np.ndarray:
    x = np.array(x, dtype=np.float32, copy=True, order="C")
    pos, pp = _c(pos, np.int32)
    cos_t, pc = _c(cos_t, np.float32)
    sin_t, ps = _c(sin_t, np.float32)
    _lib_handle().orc_rope(x.ctypes.data, x.shape[0], nheads, hd, pp, pc, ps)
    return x


def attention(q, pos, K, V, nh: int, nkv: int, hd: int) -> np.ndarray:
    q, pq = _c(q, np.float32)
    pos, pp = _c(pos, np.int32)
    K, pk = _c(K, np.float32)
    V, pv = _c(V, np.float32)
    o = np.zeros_like(q)
    _lib_handle().orc_attention(pq, q.shape[0], pp, pk, pv, nh, nkv, hd, o.ctypes.data)
    return o


def swiglu(g, u) -> np.ndarray:
    g, pg = _c(g, np.float32)
    u, pu = _c(u, np.float32)
    s = np.zeros_like(g)
    _lib_handle().orc_swiglu(pg, pu, g.size, s.ctypes.data)
    return s


def set_attention_f32(on: bool) -> bool:
    """Switch the attention between float64 (default) and float32 rounding."""
    return bool(_lib_handle().orc_set_attention_f32(int(on)))


def argmax(x: np.ndarray) -> int:
    x, px = _c(x, np.float32)
    return int(_lib_handle().orc_argmax(px, x.size))


# ---------------- model ----------------

def hparams_of(cfg) -> Hparams:
    return Hparams(cfg.n_layer, cfg.n_embd, cfg.n_head, cfg.n_head_kv, cfg.head_dim, cfg.n_ff,
                   cfg.n_vocab, cfg.max_seq_len, cfg.rope_theta, cfg.rms_eps, int(cfg.tied),
                   int(getattr(cfg, "qk_norm", False)))


class Model:
    """The oracle model: weights quantized by the oracle's own Q8_0 codec."""

    def __init__(self, cfg, tensors: dict | None = None, q8_blocks: dict | None = None):
        self.cfg = cfg
        self._hp = hparams_of(cfg)
        self.ptr = _lib_handle().orc_model_create(ctypes.byref(self._hp))
        if not self.ptr:
            raise ValueError("oracle: bad hparams")
        for name, arr in (tensors or {}).items():
            self.set_f32(name, arr)
        for name, (blocks, ne0, ne1) in (q8_blocks or {}).items():
            self.set_q8_0(name, blocks, ne0, ne1)

    def set_f32(self, name: str, arr: np.ndarray):
        arr, p = _c(arr, np.float32)
        ne0 = arr.shape[-1]
        ne1 = arr.shape[0] if arr.ndim == 2 else 1
        rc = _lib_handle().orc_model_set_f32(self.ptr, name.encode(), p, ne0, ne1)
        if rc != 0:
            raise KeyError(f"oracle: cannot set {name} ({rc})")

    def set_q8_0(self, name: str, blocks: np.ndarray, ne0: int, ne1: int):
        blocks, p = _c(blocks, np.uint8)
        rc = _lib_handle().orc_model_set_q8_0(self.ptr, name.encode(), p, ne0, ne1)
        if rc != 0:
            raise KeyError(f"oracle: cannot set {name} ({rc})")

    def get_q8(self, name: str, ne0: int, ne1: int):
        nb = (ne0 + 31) // 32
        q = np.zeros((ne1, nb * 32), np.int8)
        d = np.zeros((ne1, nb), np.uint16)
        if _lib_handle().orc_model_get_q8(self.ptr, name.encode(), q.ctypes.data, d.ctypes.data):
            raise KeyError(name)
        return q, d

    def check(self) -> bool:
        return _lib_handle().orc_model_check(self.ptr) == 0

    def kv(self, n_ctx: int) -> "KV":
        return KV(self, n_ctx)

    def prefill(self, kv: "KV", ids, pos, n_out: int = 1, hidden: bool = False):
        """Returns (rc, logits [n_out][V], hidden [L+1][nt][H] or None)."""
        ids, pi = _c(ids, np.int32)
        pos, pp = _c(pos, np.int32)
        nt = ids.size
        logits = np.zeros((max(n_out, 0), self.cfg.n_vocab), np.float32)
        hid = np.zeros((self.cfg.n_layer + 1, nt, self.cfg.n_embd), np.float32) if hidden else None
        rc = _lib_handle().orc_prefill(self.ptr, kv.ptr, pi, pp, nt, n_out,
                                       logits.ctypes.data if logits.size else None,
                                       hid.ctypes.data if hidden else None)
        return rc, logits, hid

    def __del__(self):
        if getattr(self, "ptr", None):
            _lib_handle().orc_model_free(self.ptr)
            self.ptr = None


class KV:
    def __init__(self, model: Model, n_ctx: int):
        self.model = model
        self.ptr = _lib_handle().orc_kv_create(model.ptr, n_ctx)
        if not self.ptr:
            raise ValueError("oracle: bad n_ctx")
        self.n_ctx = _lib_handle().orc_kv_ctx(self.ptr)
        self.width = model.cfg.n_head_kv * model.cfg.head_dim

    def read(self, layer: int, which: int, row0: int = 0, nrows: int | None = None) -> np.ndarray:
        nrows = self.n_ctx - row0 if nrows is None else nrows
        out = np.zeros((nrows, self.width), np.float32)
        if _lib_handle().orc_kv_read(self.ptr, layer, which, row0, nrows, out.ctypes.data, self.width):
            raise IndexError("oracle kv read")
        return out

    def write(self, layer: int, which: int, row0: int, data: np.ndarray):
        data, p = _c(data, np.float32)
        if _lib_handle().orc_kv_write(self.ptr, layer, which, row0, data.shape[0], p, self.width):
            raise IndexError("oracle kv write")

    def __del__(self):
        if getattr(self, "ptr", None):
            _lib_handle().orc_kv_free(self.ptr)
            self.ptr = None
